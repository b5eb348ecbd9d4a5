"""A cascade step as fixed launches that a CUDA graph captures once: the device-side
planner (cascade_plan_device) and the attention call that reads its prefix length from
device memory (cascade_attn_device_plan).

The planner must give cascade_plan's results exactly (random tables, every mode, the
generated batches); the captured step, replayed for batches whose shared prefix
changes between replays (all of it, half, none: the standard path), must match the
oracle on every row."""

import ctypes

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

MODES = (csp.MODE_AUTO, csp.MODE_FORCE_CASCADE, csp.MODE_FORCE_FLAT, csp.MODE_PAGE_THRESHOLDS)


def _plan_device(bt, seq, nc, bs, mode):
    lib = csp.load()
    d_bt = torch.from_numpy(np.ascontiguousarray(bt, np.int32)).cuda()
    d_sl = torch.from_numpy(np.ascontiguousarray(seq, np.int32)).cuda()
    d_nc = torch.from_numpy(np.ascontiguousarray(nc, np.int32)).cuda()
    plan = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    st = lib.cascade_plan_device(d_bt.data_ptr(), bt.shape[1], len(seq), d_sl.data_ptr(),
                                 d_nc.data_ptr(), bs, mode, plan.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == csp.CSP_OK
    torch.cuda.synchronize()
    return [int(x) for x in plan.cpu()]


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_device_planner_matches_host_planner(bs):
    rng = np.random.default_rng(700 + bs)
    for it in range(120):
        n = int(rng.integers(1, 40))
        seq = rng.integers(1, 40 * bs, size=n).astype(np.int32)
        width = int(-(-seq.max() // bs)) + 3
        table = rng.integers(0, 3, size=(n, width)).astype(np.int32)
        common = min(int(rng.integers(0, 40)), width)
        table[:, :common] = rng.integers(0, 1000, size=common)[None, :]
        nc = np.array([int(rng.integers(0, s + 1)) for s in seq], np.int32)
        mode = MODES[it % 4]
        cpl, use = csp.cascade_plan(table, seq, nc, block_size=bs, mode=mode)
        got = _plan_device(table, seq, nc, bs, mode)
        assert got == [cpl if use else 0, int(use), cpl, csp.CSP_OK], (it, got, cpl, use)


def test_device_planner_on_generated_batches_and_bad_lengths():
    for name in ("tiny", "decode", "chunked", "chunked_cap"):
        b = workloads.by_name(name)
        for mode in MODES:
            cpl, use = csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                                        block_size=b.block_size, mode=mode)
            got = _plan_device(b.block_table, b.seq_lens, b.num_computed_tokens, 16, mode)
            assert got == [cpl if use else 0, int(use), cpl, csp.CSP_OK], (name, mode)
    b = workloads.tiny_decode()
    bad = b.num_computed_tokens.copy()
    bad[3] = b.seq_lens[3] + 1                     # more computed tokens than the request has
    assert _plan_device(b.block_table, b.seq_lens, bad, 16, csp.MODE_AUTO) == \
        [0, 0, 0, csp.CSP_ERR_INVALID_ARG]
    assert _plan_device(np.zeros((0, 4), np.int32), np.zeros(0, np.int32),
                        np.zeros(0, np.int32), 16, csp.MODE_AUTO) == [0, 0, 0, 0]


def _variant(b, how):
    """The same batch with a shorter shared prefix: row 0 reads other blocks (from row
    1's private ones) from a column on, so the run every row shares ends there."""
    bt = b.block_table.copy()
    if how == "half":
        col = 32                                   # 512 of the 1024 shared tokens
    elif how == "none":
        col = 0
    else:
        return bt
    own1 = bt[1, -(-int(b.seq_lens[1]) // 16) - 1]   # a block only row 1 uses
    bt[0, col] = own1
    return bt


def test_captured_step_replays_for_changing_prefixes():
    lib = csp.load()
    b = workloads.decode_batch(seed=7001, n=16, p=1024, s=64)
    dev = H.to_device(b)
    stream = torch.cuda.Stream()
    bound = 1024
    need = csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, bound,
                              b.num_q_heads, b.num_kv_heads, b.head_dim)
    ws = csp.alloc_workspace(need, torch.device("cuda"))
    nc = torch.from_numpy(b.num_computed_tokens).cuda()
    plan = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.empty_like(dev["q"])
    lse = torch.empty((b.total_q, b.num_q_heads), dtype=torch.float32, device="cuda")

    def step(s):
        st = lib.cascade_plan_device(dev["bt"].data_ptr(), b.block_table.shape[1], b.num_reqs,
                                     dev["sl"].data_ptr(), nc.data_ptr(), 16, csp.MODE_AUTO,
                                     plan.data_ptr(), s.cuda_stream)
        assert st == csp.CSP_OK
        st = lib.cascade_attn_device_plan(
            dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), b.num_blocks,
            dev["bt"].data_ptr(), b.block_table.shape[1], dev["cu"].data_ptr(),
            dev["sl"].data_ptr(), b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k,
            plan.data_ptr(), bound, 16, b.num_q_heads, b.num_kv_heads, b.head_dim, b.scale,
            out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), s.cuda_stream)
        assert st == csp.CSP_OK

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step(stream)                                   # warm (sets the kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(stream)
    expect_cpl = {"all": 1024, "half": 512, "none": 0}
    for how in ("all", "half", "none", "all"):
        bt = _variant(b, how)
        dev["bt"].copy_(torch.from_numpy(bt))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        cpl, use = csp.cascade_plan(bt, b.seq_lens, b.num_computed_tokens, block_size=16)
        assert int(plan[2].item()) == cpl == expect_cpl[how]
        assert int(plan[0].item()) == (cpl if use else 0)
        import oracle
        ref_o, ref_l = oracle.attention(b.q, b.k_cache, b.v_cache, bt, b.cu_seqlens_q,
                                        b.seq_lens, b.scale)
        H.compare(out, lse, ref_o, ref_l, what=f"captured step, prefix {how}")
    assert csp.workspace_status(ws) == csp.CSP_OK


def test_device_plan_attention_refuses_what_it_cannot_take():
    lib = csp.load()
    wide = workloads.build_batch("wide", [300, 310], [16, 16], 288, num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, gen=torch.Generator().manual_seed(3))
    dev = H.to_device(wide)
    plan = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = csp.alloc_workspace(1 << 24, torch.device("cuda"))
    out = torch.zeros_like(dev["q"])
    st = lib.cascade_attn_device_plan(
        dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), wide.num_blocks,
        dev["bt"].data_ptr(), wide.block_table.shape[1], dev["cu"].data_ptr(),
        dev["sl"].data_ptr(), wide.num_reqs, wide.total_q, wide.max_seqlen_q,
        wide.max_seqlen_k, plan.data_ptr(), 288, 16, 32, 8, 128, wide.scale, out.data_ptr(),
        None, ws.data_ptr(), ws.numel(), None)
    assert st == csp.CSP_ERR_UNSUPPORTED        # 64 packed rows per request and KV head
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
