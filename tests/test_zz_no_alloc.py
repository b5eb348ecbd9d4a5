"""cascade_attn_noalloc: the entry point for callers that cannot allocate device memory
(an engine with its own fixed memory pool, a plugin whose host framework owns every
allocation, a latency-critical loop where an allocation could synchronise the GPU).
It runs cascade attention with the library's own fixed device array as workspace.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It also passes on its own in a fresh
process (the first call on the device sets the array's address up).
"""

import ctypes

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 16 << 20


def _noalloc_fn():
    lib = csp.load()
    fn = lib.cascade_attn_noalloc
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [p, p, p, i32, p, i64, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                   ctypes.c_float, p, p, p]
    fn.restype = ctypes.c_int
    return fn


def _status():
    lib = csp.load()
    fn = lib.csp_noalloc_status
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    fn.restype = ctypes.c_int
    st = ctypes.c_int32(-999)
    assert fn(torch.cuda.current_stream().cuda_stream, ctypes.byref(st)) == csp.CSP_OK
    return st.value


def _call(fn, b, d, cpl, out, lse):
    stream = torch.cuda.current_stream().cuda_stream
    return fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), b.num_blocks,
              d["bt"].data_ptr(), b.block_table.shape[1], d["cu"].data_ptr(),
              d["sl"].data_ptr(), b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
              b.block_size, b.num_q_heads, b.num_kv_heads, b.head_dim, b.scale,
              out.data_ptr(), lse.data_ptr(), stream)


def _check_against_cascade_attn(fn, b):
    d = H.to_device(b)
    cpl, _ = H.plan(b)
    assert cpl > 0
    ref_out, ref_lse = H.run_cascade(b, d, cpl)      # the existing entry point
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy().astype(np.float64)
    for _ in range(2):                                # two calls in a row share the array
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full((b.total_q, b.num_q_heads), float("nan"), device="cuda")
        assert _call(fn, b, d, cpl, out, lse) == csp.CSP_OK
        assert _status() == 0                        # no bounded wait gave up
        H.compare(out, lse, ref_out, ref_lse, what="noalloc vs cascade_attn")


def test_noalloc_matches_cascade_attn_on_consecutive_calls():
    fn = _noalloc_fn()
    _check_against_cascade_attn(fn, workloads.decode_batch())          # N=64 P=4096 S=128
    _check_against_cascade_attn(fn, workloads.tiny_decode())           # another shape after


def test_noalloc_rejects_a_batch_beyond_its_array():
    fn = _noalloc_fn()
    # 64 requests x 64 new tokens x 32 heads: two partial slots of 131,072 rows
    g = torch.Generator().manual_seed(77)
    b = workloads.build_batch("wide", [320] * 64, [64] * 64, 256, num_q_heads=32,
                              num_kv_heads=8, head_dim=128, gen=g)
    cpl, _ = H.plan(b)
    need = csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
                              b.num_q_heads, b.num_kv_heads, b.head_dim)
    assert need > SCRATCH_LIMIT
    d = H.to_device(b)
    out = torch.zeros_like(d["q"])
    lse = torch.zeros((b.total_q, b.num_q_heads), device="cuda")
    assert _call(fn, b, d, cpl, out, lse) == csp.CSP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0            # nothing was launched
