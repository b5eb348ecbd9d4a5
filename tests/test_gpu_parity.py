"""GPU parity: every path through the C ABI against the CPU oracle.

Small batches are checked on every output row; the full-size batches in the
benchmark's launch configuration on sampled rows.  Inputs come from the seeded
generator, with NaN-poisoned unused blocks and +-1000 in the tail slots, so a
read outside a request's pages shows up as a non-finite or wrong output.
"""

import math

import numpy as np
import pytest
import torch

from oracle import planner
from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def small(seed, n, seq, ql, shared, hq, hkv, d, scale=None):
    g = torch.Generator().manual_seed(seed)
    return workloads.build_batch(f"small{seed}", seq, ql, shared, num_q_heads=hq,
                                 num_kv_heads=hkv, head_dim=d, gen=g, scale=scale)


# (seed, seq_lens, q_lens, shared tokens, Hq, Hkv, D)
SMALL_CASES = [
    (1, [288] * 8, [1] * 8, 256, 8, 2, 64),                       # tiny decode shape
    (2, [300, 290, 333, 280, 301], [1, 1, 1, 1, 1], 272, 16, 2, 128),   # ragged prefix tile
    (3, [530, 600, 777], [5, 17, 60], 512, 32, 8, 128),           # chunked rows, group 4
    (4, [150, 170, 190, 210], [1, 1, 1, 1], 144, 8, 8, 128),      # group 1
    (5, [400] * 6, [3] * 6, 384, 32, 2, 128),                     # group 16, 3 queries
    (6, [260, 390], [40, 2], 256, 16, 2, 64),                     # group 8, D 64, prefill rows
    (7, [1000] * 3, [1] * 3, 992, 8, 4, 128),                     # long prefix, short suffix
    (8, [700, 420, 300], [100, 70, 1], 256, 16, 4, 128),          # two 256-row tiles
    (9, [300, 200], [40, 33], 128, 4, 4, 64),                     # group 1, prefill rows
    (10, [4200, 4300], [40, 50], 4096, 16, 4, 128),               # prefill rows, many prefix ranges
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=[f"case{c[0]}" for c in SMALL_CASES])
def test_small_batches_all_rows(case):
    seed, seq, ql, shared, hq, hkv, d = case
    b = small(seed, len(seq), seq, ql, shared, hq, hkv, d)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse = H.run_paged(b, dev)
    H.compare(out, lse, ref_o, ref_l, what="paged")
    cpl, _ = H.plan(b)
    assert cpl > 0
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, what="cascade")
    # cascade with a shorter prefix (still valid: any multiple of 16 <= cpl)
    out, lse = H.run_cascade(b, dev, 16)
    H.compare(out, lse, ref_o, ref_l, what="cascade cpl=16")
    # cpl = 0 is the standard path
    out, lse = H.run_cascade(b, dev, 0)
    H.compare(out, lse, ref_o, ref_l, what="cascade cpl=0")


@pytest.mark.parametrize("name", ["tiny", "decode", "chunked", "chunked_cap"])
def test_named_batches_all_rows(name):
    b = workloads.by_name(name)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, use = H.plan(b)
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, what=f"{name} cascade")
    out2, lse2 = H.run_paged(b, dev)
    H.compare(out2, lse2, ref_o, ref_l, what=f"{name} paged")
    # cascade vs flat: the pages state the two are the same result
    diff = (out.float() - out2.float()).abs().max().item()
    assert diff <= 2 * H.OUT_TOL


def test_long_prefix_sampled_rows():
    b = workloads.long_prefix()
    dev = H.to_device(b)
    rows = H.sample_rows(b, 1500, seed=4)
    ref_o, ref_l = H.oracle_ref(b, rows)
    cpl, use = H.plan(b)
    assert cpl == 16384 and use
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, rows, what="long cascade")
    out, lse = H.run_paged(b, dev)
    H.compare(out, lse, ref_o, ref_l, rows, what="long paged")


@pytest.mark.parametrize("n", [1, 2, 7, 8, 50, 100, 256])
def test_batch_size_sweep(n):
    """Results must not depend on the batch size (cascade + batch 50 vs 100 anecdote)."""
    b = workloads.decode_batch(seed=2000 + n, n=n, p=1024, s=48)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 600, seed=n)
    ref_o, ref_l = H.oracle_ref(b, rows)
    cpl, _ = H.plan(b)
    # one request shares its whole used run with itself, capped to its computed tokens
    assert cpl == (1024 if n > 1 else ((1024 + 48 - 1) // 16) * 16)
    assert (cpl, _) == planner.plan(b.block_table, b.seq_lens, b.num_computed_tokens, 16)
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, rows, what=f"N={n} cascade")
    out, lse = H.run_paged(b, dev)
    H.compare(out, lse, ref_o, ref_l, rows, what=f"N={n} paged")


GRID = [(n, p) for n in workloads.SWEEP_N for p in workloads.SWEEP_P]


@pytest.mark.parametrize("n,p", GRID, ids=[f"N{n}_P{p}" for n, p in GRID])
def test_sweep_grid(n, p):
    """Every point of the heuristic-sweep grid (S = 128), cascade and flat, against the
    oracle on sampled rows (the first and last row always among them)."""
    b = workloads.sweep_point(n, p)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 200, seed=n * 100003 + p)
    ref_o, ref_l = H.oracle_ref(b, rows)
    cpl, _ = H.plan(b)
    assert cpl == (p if n > 1 else ((p + 128 - 1) // 16) * 16)
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, rows, what=f"sweep N={n} P={p} cascade")
    out, lse = H.run_paged(b, dev)
    H.compare(out, lse, ref_o, ref_l, rows, what=f"sweep N={n} P={p} flat")


def test_request_without_queries():
    # request 1 contributes KV but no query rows this step
    b = small(21, 3, [300, 310, 305], [2, 0, 3], 288, 8, 2, 128)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse = H.run_cascade(b, dev, H.plan(b)[0])
    H.compare(out, lse, ref_o, ref_l, what="empty request")


def test_merge_states_against_oracle():
    import oracle
    rng = np.random.default_rng(7)
    t, h, d = 37, 6, 128
    o1 = rng.standard_normal((t, h, d))
    o2 = rng.standard_normal((t, h, d))
    l1 = rng.standard_normal((t, h)) * 3
    l2 = rng.standard_normal((t, h)) * 3
    l1[0, 0] = -np.inf            # one empty side
    l1[1, 1] = l2[1, 1] = -np.inf  # both empty
    for dtype in (torch.float32, torch.bfloat16):
        to = lambda x: torch.from_numpy(x).to(dtype).cuda()
        p1, p2 = to(o1), to(o2)
        ref_o, ref_l = oracle.merge_states(p1.double().cpu().numpy(), l1,
                                           p2.double().cpu().numpy(), l2)
        out, lse = csp.merge_states(p1, torch.from_numpy(l1).float().cuda(), p2,
                                    torch.from_numpy(l2).float().cuda())
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.abs(got - ref_o).max() <= 1e-2
        gl = lse.cpu().numpy()
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(gl), fin)
        assert np.all(np.abs(gl[fin] - ref_l[fin]) <= 1e-5 * np.maximum(1, np.abs(ref_l[fin])))


def test_argument_errors_launch_nothing():
    b = workloads.tiny_decode()
    dev = H.to_device(b)
    cpl = 256
    with pytest.raises(csp.CspError) as e:
        H.run_cascade(b, dev, 250)                 # not a multiple of the block size
    assert e.value.status == csp.CSP_ERR_INVALID_ARG
    need = csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
                              b.num_q_heads, b.num_kv_heads, b.head_dim)
    small_ws = torch.zeros(max(need - 512, 256), dtype=torch.uint8, device="cuda")
    lib = csp.load()
    out = torch.empty_like(dev["q"])
    st = lib.cascade_attn(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                          b.num_blocks, dev["bt"].data_ptr(), b.block_table.shape[1],
                          dev["cu"].data_ptr(), dev["sl"].data_ptr(), b.num_reqs, b.total_q,
                          b.max_seqlen_q, b.max_seqlen_k, cpl, 16, b.num_q_heads,
                          b.num_kv_heads, b.head_dim, b.scale, out.data_ptr(), None,
                          small_ws.data_ptr(), small_ws.numel(), None)
    assert st == csp.CSP_ERR_WORKSPACE
    assert lib.csp_workspace_size(8, 8, 1, 288, 0, 8, 2, 96, None) == csp.CSP_ERR_INVALID_ARG
    import ctypes
    sz = ctypes.c_size_t(0)
    assert lib.csp_workspace_size(8, 8, 1, 288, 0, 8, 2, 96, ctypes.byref(sz)) == \
        csp.CSP_ERR_UNSUPPORTED
    assert lib.csp_workspace_size(8, 8, 1, 288, 0, 12, 4, 128, ctypes.byref(sz)) == \
        csp.CSP_ERR_UNSUPPORTED            # group 3


def test_status_word_stays_clear():
    b = workloads.decode_batch(seed=77, n=16, p=512, s=64)
    dev = H.to_device(b)
    cpl, _ = H.plan(b)
    need = csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
                              b.num_q_heads, b.num_kv_heads, b.head_dim)
    ws = csp.alloc_workspace(need, "cuda")
    for _ in range(3):
        H.run_cascade(b, dev, cpl, workspace=ws)
    assert csp.workspace_status(ws) == 0


def test_validated_call_with_a_bad_block_id_launches_nothing():
    b = workloads.tiny_decode()
    dev = H.to_device(b)
    cpl, _ = H.plan(b)
    bad = b.block_table.copy()
    bad[5, (int(b.seq_lens[5]) - 1) // 16] = b.num_blocks + 7   # past the cache
    out = torch.zeros_like(dev["q"])
    lse = torch.zeros((b.total_q, b.num_q_heads), device="cuda")
    for fn in (lambda **kw: H.run_cascade(b, dev, cpl, **kw), lambda **kw: H.run_paged(b, dev, **kw)):
        with pytest.raises(csp.CspError) as e:
            fn(out=out, lse=lse, validate=(bad, b.seq_lens, b.cu_seqlens_q))
        assert e.value.status == csp.CSP_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert out.abs().max().item() == 0.0 and lse.abs().max().item() == 0.0
    # the good tables pass the same check and the call runs
    ref_o, ref_l = H.oracle_ref(b)
    o2, l2 = H.run_cascade(b, dev, cpl, validate=(b.block_table, b.seq_lens, b.cu_seqlens_q))
    H.compare(o2, l2, ref_o, ref_l, what="validated cascade")
