"""C-ABI checks that need no GPU: the library builds and loads, it exports every
function include/csp.h declares, and the host-side planner matches the planner
oracle exactly (it runs no device code)."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import planner
from shared_prefix_paged_gb300 import csp, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "csp.h"), encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"CSP_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_symbols() == sorted(csp.EXPORTS)


def test_library_loads_and_exports_every_declared_symbol():
    lib = csp.load()
    for name in _declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value
    assert lib.csp_version() >> 16 == 1
    assert lib.csp_status_string(csp.CSP_ERR_WORKSPACE) == b"CSP_ERR_WORKSPACE"


def test_planner_worked_example():
    # "vLLM Cascade Attention：用法、场景与原理解析" §四, block_size 1
    bt = np.array([[0, 1, 2, 3, 4, 5], [0, 1, 2, 3, 4, 6]], np.int32)
    cpl, use = csp.cascade_plan(bt, [6, 6], [3, 4], block_size=1,
                                mode=csp.MODE_PAGE_THRESHOLDS)
    assert (cpl, use) == (3, False)


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_planner_matches_oracle_on_random_tables(bs):
    rng = np.random.default_rng(100 + bs)
    for _ in range(300):
        n = int(rng.integers(1, 12))
        common = int(rng.integers(0, 40))
        seq = rng.integers(1, 40 * bs, size=n)
        width = int(-(-seq.max() // bs)) + 3
        table = rng.integers(0, 3, size=(n, width)).astype(np.int32)
        common = min(common, width)
        table[:, :common] = rng.integers(0, 1000, size=common)[None, :]
        nc = np.array([int(rng.integers(0, s + 1)) for s in seq], np.int32)
        want = planner.plan(table, seq, nc, bs)
        got = csp.cascade_plan(table, seq, nc, block_size=bs, mode=csp.MODE_PAGE_THRESHOLDS)
        assert got == want, (table, seq, nc)


@pytest.mark.parametrize("name", ["tiny", "decode", "chunked", "chunked_cap"])
def test_planner_matches_oracle_on_generated_batches(name):
    b = workloads.by_name(name)
    want = planner.plan(b.block_table, b.seq_lens, b.num_computed_tokens, b.block_size)
    got = csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                           block_size=b.block_size, mode=csp.MODE_PAGE_THRESHOLDS)
    assert got == want


def test_planner_modes_and_errors():
    b = workloads.decode_batch(n=8, p=512, s=32)
    args = (b.block_table, b.seq_lens, b.num_computed_tokens)
    assert csp.cascade_plan(*args, mode=csp.MODE_FORCE_FLAT) == (512, False)
    assert csp.cascade_plan(*args, mode=csp.MODE_FORCE_CASCADE) == (512, True)
    # the GB300 rule leaves a batch whose standard path streams under 8192 KV tokens
    # (8 x 544 here) to that path: both calls are latency-bound there
    assert csp.cascade_plan(*args, mode=csp.MODE_AUTO) == (512, False)
    big = workloads.decode_batch(n=16, p=512, s=32)    # 16 x 544 = 8704 tokens, 3.5x fewer
    bargs = (big.block_table, big.seq_lens, big.num_computed_tokens)
    assert csp.cascade_plan(*bargs, mode=csp.MODE_AUTO) == (512, True)
    # the GB300 rule keeps cascade for a small batch over a long prefix (the pages'
    # thresholds refuse N < 8) and refuses it where it would save too few bytes
    small = workloads.decode_batch(n=4, p=4096, s=32)
    sargs = (small.block_table, small.seq_lens, small.num_computed_tokens)
    assert csp.cascade_plan(*sargs, mode=csp.MODE_PAGE_THRESHOLDS) == (4096, False)
    assert csp.cascade_plan(*sargs, mode=csp.MODE_AUTO) == (4096, True)
    short = workloads.decode_batch(n=16, p=64, s=128)   # 16*192 vs 64+16*128 tokens: 1.46x
    rargs = (short.block_table, short.seq_lens, short.num_computed_tokens)
    assert csp.cascade_plan(*rargs, mode=csp.MODE_AUTO) == (64, False)
    assert csp.cascade_plan(np.zeros((0, 4), np.int32), [], []) == (0, False)
    with pytest.raises(csp.CspError) as e:
        csp.cascade_plan(b.block_table, b.seq_lens, b.seq_lens + 1)   # computed > seq_len
    assert e.value.status == csp.CSP_ERR_INVALID_ARG
    with pytest.raises(csp.CspError):
        csp.cascade_plan(b.block_table[:, :3], b.seq_lens, b.num_computed_tokens)  # row too short
    with pytest.raises(csp.CspError):
        csp.cascade_plan(*args, mode=9)


def test_validate_batch_accepts_generated_batches():
    for name in ("tiny", "decode", "chunked", "chunked_cap"):
        b = workloads.by_name(name)
        cpl, _ = csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                                  block_size=b.block_size)
        assert csp.validate_batch(b.block_table, b.seq_lens, b.cu_seqlens_q,
                                  block_size=b.block_size, num_blocks=b.num_blocks,
                                  common_prefix_len=cpl) == (csp.CSP_OK, -1)


def test_validate_batch_rejects_bad_tables():
    b = workloads.tiny_decode()
    bt = b.block_table.copy()
    w = bt.shape[1]
    ok = dict(block_size=16, num_blocks=b.num_blocks)
    # an id past the cache in a used entry: rejected, its flat index reported
    used = (int(b.seq_lens[3]) + 15) // 16
    bt[3, used - 1] = b.num_blocks
    assert csp.validate_batch(bt, b.seq_lens, b.cu_seqlens_q, **ok) == \
        (csp.CSP_ERR_INVALID_ARG, 3 * w + used - 1)
    bt[3, used - 1] = -1
    assert csp.validate_batch(bt, b.seq_lens, **ok)[0] == csp.CSP_ERR_INVALID_ARG
    # the same id past the row's used entries is never read: accepted
    bt = b.block_table.copy()
    if used < w:
        bt[3, used] = 10 ** 6
        assert csp.validate_batch(bt, b.seq_lens, **ok)[0] == csp.CSP_OK
    # lengths and queries
    sl = b.seq_lens.copy()
    sl[0] = -1
    assert csp.validate_batch(b.block_table, sl, **ok) == (csp.CSP_ERR_INVALID_ARG, -1)
    sl = b.seq_lens.copy()
    sl[0] = 16 * w + 1                                   # more pages than the row holds
    assert csp.validate_batch(b.block_table, sl, **ok)[0] == csp.CSP_ERR_INVALID_ARG
    cu = b.cu_seqlens_q.copy()
    cu[2] = cu[1] - 1                                    # negative query count
    assert csp.validate_batch(b.block_table, b.seq_lens, cu, **ok)[0] == \
        csp.CSP_ERR_INVALID_ARG
    cu = b.cu_seqlens_q.copy()
    cu[0] = 1
    assert csp.validate_batch(b.block_table, b.seq_lens, cu, **ok)[0] == \
        csp.CSP_ERR_INVALID_ARG
    # the prefix length: a multiple of the block size, at most the shortest request
    assert csp.validate_batch(b.block_table, b.seq_lens, common_prefix_len=250,
                              **ok)[0] == csp.CSP_ERR_INVALID_ARG
    assert csp.validate_batch(b.block_table, b.seq_lens,
                              common_prefix_len=16 * ((int(b.seq_lens.min()) + 16) // 16),
                              **ok)[0] == csp.CSP_ERR_INVALID_ARG
    assert csp.validate_batch(b.block_table, b.seq_lens, common_prefix_len=256,
                              **ok) == (csp.CSP_OK, -1)
    assert csp.validate_batch(np.zeros((0, 4), np.int32), [], **ok) == (csp.CSP_OK, -1)
    assert csp.validate_batch(b.block_table, b.seq_lens, block_size=16,
                              num_blocks=0)[0] == csp.CSP_ERR_INVALID_ARG


def test_apply_sinks_argument_errors_launch_nothing():
    lib = csp.load()
    # head_dim not a multiple of 8, or with head_dim / 8 not dividing 32; missing lse
    assert lib.csp_apply_sinks(None, None, None, 4, 8, 12, None) == csp.CSP_ERR_INVALID_ARG
    assert lib.csp_apply_sinks(None, None, None, 4, 8, 24, None) == csp.CSP_ERR_INVALID_ARG
    assert lib.csp_apply_sinks(None, None, None, 4, 0, 64, None) == csp.CSP_ERR_INVALID_ARG
    assert lib.csp_apply_sinks(None, None, None, 4, 8, 64, None) == csp.CSP_ERR_INVALID_ARG
    assert lib.csp_apply_sinks(None, None, None, 0, 8, 64, None) == csp.CSP_OK


def test_fp8kv_argument_errors_launch_nothing():
    lib = csp.load()
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    # shapes: group 3 is unsupported, head_dim 96 too
    out = ctypes.c_size_t(0)
    assert lib.csp_workspace_size_fp8kv(4, 4, 1, 64, 0, 24, 8, 128, ctypes.byref(out)) == \
        csp.CSP_ERR_UNSUPPORTED
    assert lib.csp_workspace_size_fp8kv(4, 4, 1, 64, 0, 8, 2, 96, ctypes.byref(out)) == \
        csp.CSP_ERR_UNSUPPORTED
    assert lib.csp_workspace_size_fp8kv(4, 4, 1, 64, 8, 8, 2, 64, ctypes.byref(out)) == \
        csp.CSP_ERR_INVALID_ARG                       # prefix not a multiple of 16
    # scales must be finite and positive: refused before any device work
    args = [p, p, p, 8, p, 4, p, p, 1, 1, 1, 16, 16, 16, 8, 2, 64, 0.125]
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))):
        assert lib.cascade_attn_fp8kv(*args, ks, vs, p, None, p, 4096, None) == \
            csp.CSP_ERR_INVALID_ARG
    args_flat = args[:12] + args[13:]
    assert lib.paged_attn_fp8kv(*args_flat, 0.0, 1.0, p, None, p, 4096, None) == \
        csp.CSP_ERR_INVALID_ARG


def test_step_scratch_size_checks_the_batch():
    b = workloads.tiny_decode()
    lib = csp.load()
    out = ctypes.c_size_t(0)
    cu = np.ascontiguousarray(b.cu_seqlens_q, np.int32)
    sl = np.ascontiguousarray(b.seq_lens, np.int32)
    w = b.block_table.shape[1]
    good = lib.csp_step_scratch_size(b.num_reqs, b.total_q, cu.ctypes.data, sl.ctypes.data, w,
                                     0, 8, 2, 64, ctypes.byref(out))
    # a valid batch passes the host checks; without a GPU the device query then fails
    assert good in (csp.CSP_OK, csp.CSP_ERR_CUDA)
    bad = cu.copy()
    bad[-1] += 1                                    # total_q disagrees with cu_seqlens_q
    assert lib.csp_step_scratch_size(b.num_reqs, b.total_q, bad.ctypes.data, sl.ctypes.data, w,
                                     0, 8, 2, 64, ctypes.byref(out)) == csp.CSP_ERR_INVALID_ARG
    short = sl.copy()
    short[0] = 0                                    # fewer keys than queries
    assert lib.csp_step_scratch_size(b.num_reqs, b.total_q, cu.ctypes.data, short.ctypes.data,
                                     w, 0, 8, 2, 64, ctypes.byref(out)) == \
        csp.CSP_ERR_INVALID_ARG
