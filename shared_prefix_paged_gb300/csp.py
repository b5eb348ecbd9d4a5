"""ctypes binding of libcsp_gb300.so (include/csp.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels (or, for ``cascade_plan``, its host C code).  PyTorch supplies device
memory and the current stream.  If the library cannot be loaded the first call
raises; there is no fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

from . import build as _build

CSP_OK = 0
CSP_ERR_INVALID_ARG = -1
CSP_ERR_UNSUPPORTED = -2
CSP_ERR_WORKSPACE = -3
CSP_ERR_CUDA = -4
CSP_ERR_TIMEOUT = -6

MODE_AUTO, MODE_FORCE_CASCADE, MODE_FORCE_FLAT, MODE_PAGE_THRESHOLDS = 0, 1, 2, 3
SCHEDULE_TWO_KERNELS, SCHEDULE_SINGLE, SCHEDULE_FUSED = 0, 1, 2
DTYPE_BF16, DTYPE_F32 = 0, 1

# every symbol include/csp.h declares
EXPORTS = ("cascade_plan", "csp_workspace_size", "cascade_attn", "cascade_attn_timed",
           "cascade_attn_scheduled", "paged_attn", "merge_states", "csp_workspace_status",
           "csp_status_string", "csp_last_cuda_error", "csp_version", "cascade_attn_noalloc",
           "csp_noalloc_status", "csp_cascade_schedule", "csp_validate_batch",
           "csp_apply_sinks", "cascade_plan_device", "cascade_attn_device_plan",
           "cascade_plan_levels", "csp_workspace_size_levels", "cascade_attn_levels",
           "csp_workspace_size_fp8kv", "cascade_attn_fp8kv", "paged_attn_fp8kv",
           "csp_step_scratch_size", "cascade_step_host")

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class CspError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = _lib
        name = lib.csp_status_string(status).decode() if lib else str(status)
        extra = ""
        if status == CSP_ERR_CUDA and lib:
            extra = f" (cudaError {lib.csp_last_cuda_error()})"
        super().__init__(f"{what} failed: {name}{extra}")
        self.status = status


def library_path() -> str:
    return _build.lib_path()


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Open the library (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing and (not os.path.exists(path) or _build.is_stale()):
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library missing: {path} (run the build first)")
        lib = ctypes.CDLL(path)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.cascade_plan.argtypes = [p, i64, i32, p, p, i32, i32, i32, i32, i32, i32, p, p]
        lib.csp_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, p]
        lib.csp_cascade_schedule.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, p, p]
        attn = [p, p, p, i32, p, i64, p, p, i32, i32, i32, i32]
        tail = [i32, i32, i32, i32, ctypes.c_float, p, p, p, sz, p]
        lib.cascade_attn.argtypes = attn + [i32] + tail
        lib.cascade_attn_timed.argtypes = attn + [i32] + tail + [p]
        lib.cascade_attn_scheduled.argtypes = attn + [i32] + tail + [i32, i32]
        lib.paged_attn.argtypes = attn + tail
        lib.merge_states.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, p]
        lib.csp_workspace_status.argtypes = [p, p, p]
        lib.csp_validate_batch.argtypes = [p, i64, i32, p, p, i32, i32, i32, p]
        lib.csp_apply_sinks.argtypes = [p, p, p, i32, i32, i32, p]
        lib.cascade_plan_device.argtypes = [p, i64, i32, p, p, i32, i32, p, p]
        lib.cascade_attn_device_plan.argtypes = attn + [p, i32] + tail
        lib.cascade_plan_levels.argtypes = [p, i64, i32, p, p, i32, i32, i32, p, p, p]
        lib.csp_workspace_size_levels.argtypes = [i32, i32, i32, i32, p, i32, i32, i32, i32,
                                                  i32, p]
        lib.cascade_attn_levels.argtypes = attn + [p, i32, p, i32] + tail
        f32 = ctypes.c_float
        tail8 = [i32, i32, i32, i32, f32, f32, f32, p, p, p, sz, p]
        lib.csp_workspace_size_fp8kv.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, p]
        lib.cascade_attn_fp8kv.argtypes = attn + [i32] + tail8
        lib.paged_attn_fp8kv.argtypes = attn + tail8
        lib.csp_step_scratch_size.argtypes = [i32, i32, p, p, i64, i32, i32, i32, i32, p]
        lib.cascade_step_host.argtypes = [p, p, i64, p, p, p, i32, i32, p, p, i32, i32, i32,
                                          i32, i32, f32, i32, p, p, p, sz, p, p]
        lib.csp_status_string.argtypes = [ctypes.c_int]
        lib.csp_status_string.restype = ctypes.c_char_p
        for name in ("cascade_plan", "csp_workspace_size", "cascade_attn", "cascade_attn_timed",
                     "cascade_attn_scheduled", "paged_attn",
                     "merge_states", "csp_workspace_status", "csp_last_cuda_error",
                     "csp_version", "csp_cascade_schedule", "csp_validate_batch",
                     "csp_apply_sinks", "cascade_plan_device", "cascade_attn_device_plan",
                     "cascade_plan_levels", "csp_workspace_size_levels",
                     "cascade_attn_levels", "csp_workspace_size_fp8kv", "cascade_attn_fp8kv",
                     "paged_attn_fp8kv", "csp_step_scratch_size", "cascade_step_host"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != CSP_OK:
        raise CspError(status, what)


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def cascade_plan(block_table, seq_lens, num_computed_tokens, *, block_size=16, num_q_heads=32,
                 num_kv_heads=8, head_dim=128, num_sms=0, mode=MODE_AUTO):
    """(common_prefix_len, use_cascade) for host arrays (numpy or CPU tensors)."""
    lib = load()
    bt = _host_i32(block_table)
    sl = _host_i32(seq_lens)
    nc = _host_i32(num_computed_tokens)
    n = int(sl.shape[0])
    stride = int(bt.shape[1]) if bt.ndim == 2 else 0
    cpl = ctypes.c_int32(0)
    use = ctypes.c_int32(0)
    _check(lib.cascade_plan(bt.ctypes.data if bt.size else None, stride, n,
                            sl.ctypes.data if n else None, nc.ctypes.data if n else None,
                            block_size, num_q_heads, num_kv_heads, head_dim, num_sms, mode,
                            ctypes.byref(cpl), ctypes.byref(use)), "cascade_plan")
    return int(cpl.value), bool(use.value)


def validate_batch(block_table, seq_lens, cu_seqlens_q=None, *, block_size=16, num_blocks,
                   common_prefix_len=0):
    """csp_validate_batch on host arrays: (status, flat index of the first out-of-range
    block id or -1).  Raises nothing; CSP_OK means the batch may be launched."""
    lib = load()
    bt = _host_i32(block_table)
    sl = _host_i32(seq_lens)
    cu = None if cu_seqlens_q is None else _host_i32(cu_seqlens_q)
    n = int(sl.shape[0])
    stride = int(bt.shape[1]) if bt.ndim == 2 else 0
    bad = ctypes.c_int64(0)
    st = lib.csp_validate_batch(bt.ctypes.data if bt.size else None, stride, n,
                                sl.ctypes.data if n else None,
                                None if cu is None else cu.ctypes.data, int(block_size),
                                int(num_blocks), int(common_prefix_len), ctypes.byref(bad))
    return int(st), int(bad.value)


class Planner:
    """cascade_plan over fixed host arrays (numpy int32, kept alive here), with its
    arguments marshalled once: each call passes the arrays' current contents, so a
    caller that rewrites them in place between steps re-plans without re-marshalling."""

    def __init__(self, block_table, seq_lens, num_computed_tokens, *, block_size=16,
                 num_q_heads=32, num_kv_heads=8, head_dim=128, num_sms=0, mode=MODE_AUTO):
        self._lib = load()
        self.block_table = _host_i32(block_table)
        self.seq_lens = _host_i32(seq_lens)
        self.num_computed_tokens = _host_i32(num_computed_tokens)
        self._cpl = ctypes.c_int32(0)
        self._use = ctypes.c_int32(0)
        n = int(self.seq_lens.shape[0])
        bt = self.block_table
        self._args = (bt.ctypes.data if bt.size else None,
                      int(bt.shape[1]) if bt.ndim == 2 else 0, n,
                      self.seq_lens.ctypes.data if n else None,
                      self.num_computed_tokens.ctypes.data if n else None, block_size,
                      num_q_heads, num_kv_heads, head_dim, num_sms, mode,
                      ctypes.byref(self._cpl), ctypes.byref(self._use))

    def __call__(self):
        """(common_prefix_len, use_cascade) for the arrays' current contents."""
        _check(self._lib.cascade_plan(*self._args), "cascade_plan")
        return self._cpl.value, self._use.value != 0


class PreparedCall:
    """One attention call (cascade_attn or paged_attn) on fixed device tensors, its
    arguments marshalled once.  Calling it launches on `stream` with the step's prefix
    length: the tensors' current contents are the step's inputs and outputs."""

    def __init__(self, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *,
                 max_seqlen_q, max_seqlen_k, softmax_scale, out, lse, workspace, stream=None):
        self._lib = load()
        total_q, hq, d = q.shape
        num_blocks, bs, hkv, _ = k_cache.shape
        n = int(seqused_k.shape[0])
        self._keep = (q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, out, lse,
                      workspace)
        self._head = [_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
                      int(block_table.stride(0)), _ptr(cu_seqlens_q), _ptr(seqused_k), n,
                      total_q, int(max_seqlen_q), int(max_seqlen_k)]
        self._tail = [bs, hq, hkv, d, ctypes.c_float(float(softmax_scale)), _ptr(out),
                      _ptr(lse), _ptr(workspace), workspace.numel(),
                      _stream_ptr(stream, q.device)]
        self._cascade = self._lib.cascade_attn
        self._paged = self._lib.paged_attn

    def __call__(self, common_prefix_len: int, use_cascade: bool = True) -> None:
        if use_cascade:
            st = self._cascade(*self._head, int(common_prefix_len), *self._tail)
            _check(st, "cascade_attn")
        else:
            _check(self._paged(*self._head, *self._tail), "paged_attn")


def workspace_size(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len,
                   num_q_heads, num_kv_heads, head_dim) -> int:
    lib = load()
    out = ctypes.c_size_t(0)
    _check(lib.csp_workspace_size(num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                                  common_prefix_len, num_q_heads, num_kv_heads, head_dim,
                                  ctypes.byref(out)), "csp_workspace_size")
    return int(out.value)


def cascade_schedule(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len,
                     num_q_heads, num_kv_heads, head_dim):
    """(schedule, prefix key ranges) that cascade_attn uses for this batch shape on the
    current device: SCHEDULE_TWO_KERNELS, SCHEDULE_SINGLE or SCHEDULE_FUSED."""
    lib = load()
    sched = ctypes.c_int32(0)
    splits = ctypes.c_int32(0)
    _check(lib.csp_cascade_schedule(num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                                    common_prefix_len, num_q_heads, num_kv_heads, head_dim,
                                    ctypes.byref(sched), ctypes.byref(splits)),
           "csp_cascade_schedule")
    return int(sched.value), int(splits.value)


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def alloc_workspace(nbytes: int, device):
    """Zero-filled, 256-byte-aligned device workspace (torch allocations are)."""
    import torch
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def _attn(fn_name, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *, max_seqlen_q,
          max_seqlen_k, softmax_scale, common_prefix_len=None, out=None, lse=None,
          workspace=None, stream=None, phase_events=None, schedule=None, prefix_ranges=0,
          validate=None, sinks=None):
    import torch
    lib = load()
    total_q, hq, d = q.shape
    num_blocks, bs, hkv, _ = k_cache.shape
    n = int(seqused_k.shape[0])
    cpl = 0 if common_prefix_len is None else int(common_prefix_len)
    if validate is not None:
        # opt-in: host copies (block_table, seq_lens, cu_seqlens_q) checked by the
        # library before anything is launched
        st, bad = validate_batch(*validate, block_size=bs, num_blocks=num_blocks,
                                 common_prefix_len=cpl)
        _check(st, f"csp_validate_batch (first bad block-table index {bad})")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:  # a caller's workspace is checked by the library itself
        workspace = alloc_workspace(
            workspace_size(n, total_q, max_seqlen_q, max_seqlen_k, cpl, hq, hkv, d), q.device)
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
            int(block_table.stride(0)), _ptr(cu_seqlens_q), _ptr(seqused_k), n, total_q,
            int(max_seqlen_q), int(max_seqlen_k)]
    if fn_name == "cascade_attn":
        args.append(cpl)
    args += [bs, hq, hkv, d, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
             workspace.numel(), _stream_ptr(stream, q.device)]
    if schedule is not None:
        if phase_events is not None:
            raise ValueError("schedule and phase_events do not combine")
        fn_name = "cascade_attn_scheduled"
        args += [int(schedule), int(prefix_ranges)]
    if phase_events is not None:
        fn_name = "cascade_attn_timed"
        if len(phase_events) != 4 or any(ev.cuda_event == 0 for ev in phase_events):
            raise ValueError("phase_events: four created CUDA events (record each once first)")
        handles = (ctypes.c_void_p * 4)(*[ev.cuda_event for ev in phase_events])
        args.append(ctypes.cast(handles, ctypes.c_void_p))
    _check(getattr(lib, fn_name)(*args), fn_name)
    if sinks is not None:
        apply_sinks(out, lse, sinks, stream=stream)
    return out, lse


def cascade_attn(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *, max_seqlen_q,
                 max_seqlen_k, common_prefix_len, softmax_scale, out=None, lse=None,
                 workspace=None, stream=None, phase_events=None, schedule=None,
                 prefix_ranges=0, validate=None, sinks=None):
    """Cascade attention (prefix phase + suffix phase + LSE merge) on device tensors.

    sinks: optional fp32 device tensor [Hq] of per-head sink logits (natural log),
    applied to the result by csp_apply_sinks.
    validate: optional host copies (block_table, seq_lens, cu_seqlens_q) that the
    library checks (csp_validate_batch) before launching; a bad batch raises
    CspError(CSP_ERR_INVALID_ARG) and nothing runs on the device.
    workspace: a uint8 device tensor of at least workspace_size(...) bytes (allocated
    here when None); one that is too small raises (CSP_ERR_WORKSPACE).
    phase_events: optional four torch.cuda.Event(enable_timing=True); when given, the
    call goes through cascade_attn_timed and records them between the kernels.
    schedule: SCHEDULE_TWO_KERNELS, SCHEDULE_SINGLE or SCHEDULE_FUSED to override the
    cost model (cascade_attn_scheduled), with prefix_ranges > 0 fixing the single
    kernel's number of prefix key ranges.
    """
    return _attn("cascade_attn", q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                 max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                 softmax_scale=softmax_scale, common_prefix_len=common_prefix_len, out=out,
                 lse=lse, workspace=workspace, stream=stream, phase_events=phase_events,
                 schedule=schedule, prefix_ranges=prefix_ranges, validate=validate,
                 sinks=sinks)


def paged_attn(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *, max_seqlen_q,
               max_seqlen_k, softmax_scale, out=None, lse=None, workspace=None, stream=None,
               validate=None, sinks=None):
    """Standard (flat) paged attention on device tensors (validate, sinks: as for
    cascade_attn)."""
    return _attn("paged_attn", q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                 max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                 softmax_scale=softmax_scale, out=out, lse=lse, workspace=workspace,
                 stream=stream, validate=validate, sinks=sinks)


SEG_INTS = 7  # level, r_lo, r_hi, k_lo, k_hi, tok_lo, tok_hi


def cascade_plan_levels(block_table, seq_lens, num_computed_tokens, *, block_size=16,
                        max_levels=3, max_segments=256):
    """(segments int32 [S, 7], suffix_start int32 [num_reqs]) of the multi-level planner
    for host arrays; segments rows are (level, r_lo, r_hi, k_lo, k_hi, tok_lo, tok_hi)."""
    lib = load()
    bt = _host_i32(block_table)
    sl = _host_i32(seq_lens)
    nc = _host_i32(num_computed_tokens)
    n = int(sl.shape[0])
    stride = int(bt.shape[1]) if bt.ndim == 2 else 0
    segs = np.zeros((max(max_segments, 1), SEG_INTS), np.int32)
    start = np.zeros(max(n, 1), np.int32)
    count = ctypes.c_int32(0)
    _check(lib.cascade_plan_levels(bt.ctypes.data if bt.size else None, stride, n,
                                   sl.ctypes.data if n else None,
                                   nc.ctypes.data if n else None, block_size, max_levels,
                                   max_segments, segs.ctypes.data, ctypes.byref(count),
                                   start.ctypes.data), "cascade_plan_levels")
    return segs[:count.value].copy(), start[:n].copy()


def workspace_size_levels(num_reqs, total_q, max_seqlen_q, max_seqlen_k, segments,
                          max_suffix_len, num_q_heads, num_kv_heads, head_dim) -> int:
    lib = load()
    seg = _host_i32(segments).reshape(-1, SEG_INTS)
    out = ctypes.c_size_t(0)
    _check(lib.csp_workspace_size_levels(num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                                         seg.ctypes.data if seg.size else None, seg.shape[0],
                                         max_suffix_len, num_q_heads, num_kv_heads, head_dim,
                                         ctypes.byref(out)), "csp_workspace_size_levels")
    return int(out.value)


def cascade_attn_levels(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *,
                        max_seqlen_q, max_seqlen_k, segments, suffix_start, max_suffix_len,
                        softmax_scale, out=None, lse=None, workspace=None, stream=None):
    """Multi-level cascade attention on device tensors: segments as cascade_plan_levels
    returns them (host), suffix_start an int32 device tensor [num_reqs], max_suffix_len
    the longest suffix in keys (seqused_k - suffix_start, maximum over requests)."""
    import torch
    lib = load()
    total_q, hq, d = q.shape
    num_blocks, bs, hkv, _ = k_cache.shape
    n = int(seqused_k.shape[0])
    seg = _host_i32(segments).reshape(-1, SEG_INTS)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(
            workspace_size_levels(n, total_q, max_seqlen_q, max_seqlen_k, seg,
                                  max_suffix_len, hq, hkv, d), q.device)
    _check(lib.cascade_attn_levels(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
        int(block_table.stride(0)), _ptr(cu_seqlens_q), _ptr(seqused_k), n, total_q,
        int(max_seqlen_q), int(max_seqlen_k), seg.ctypes.data if seg.size else None,
        seg.shape[0], _ptr(suffix_start), int(max_suffix_len), bs, hq, hkv, d,
        float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream_ptr(stream, q.device)), "cascade_attn_levels")
    return out, lse


def workspace_size_fp8kv(num_reqs, total_q, max_seqlen_q, max_seqlen_k, common_prefix_len,
                         num_q_heads, num_kv_heads, head_dim) -> int:
    lib = load()
    out = ctypes.c_size_t(0)
    _check(lib.csp_workspace_size_fp8kv(num_reqs, total_q, max_seqlen_q, max_seqlen_k,
                                        common_prefix_len, num_q_heads, num_kv_heads, head_dim,
                                        ctypes.byref(out)), "csp_workspace_size_fp8kv")
    return int(out.value)


def attn_fp8kv(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, *, max_seqlen_q,
               max_seqlen_k, softmax_scale, k_scale, v_scale, common_prefix_len=0, out=None,
               lse=None, workspace=None, stream=None):
    """Attention over an FP8 (E4M3) KV cache: k_cache / v_cache uint8 device tensors
    [num_blocks, 16, Hkv, D] of E4M3 bytes, values decode(byte) * k_scale (v_scale).
    common_prefix_len > 0: cascade_attn_fp8kv; 0: paged_attn_fp8kv (the standard path)."""
    import torch
    lib = load()
    total_q, hq, d = q.shape
    num_blocks, bs, hkv, _ = k_cache.shape
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise ValueError("k_cache and v_cache: uint8 tensors of E4M3 bytes")
    n = int(seqused_k.shape[0])
    cpl = int(common_prefix_len)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size_fp8kv(n, total_q, max_seqlen_q, max_seqlen_k,
                                                         cpl, hq, hkv, d), q.device)
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
            int(block_table.stride(0)), _ptr(cu_seqlens_q), _ptr(seqused_k), n, total_q,
            int(max_seqlen_q), int(max_seqlen_k)]
    if cpl > 0:
        args.append(cpl)
    args += [bs, hq, hkv, d, float(softmax_scale), float(k_scale), float(v_scale), _ptr(out),
             _ptr(lse), _ptr(workspace), workspace.numel(), _stream_ptr(stream, q.device)]
    name = "cascade_attn_fp8kv" if cpl > 0 else "paged_attn_fp8kv"
    _check(getattr(lib, name)(*args), name)
    return out, lse


class HostStep:
    """cascade_step_host on fixed host arrays (numpy, ideally in pinned memory) and device
    caches: arguments marshalled once; each call copies the step's inputs in, plans,
    runs the attention call, copies out / lse back into the given host arrays and
    waits.  Returns the prefix length used (0: the standard path)."""

    def __init__(self, q, block_table, cu_seqlens_q, seq_lens, num_computed_tokens, k_cache,
                 v_cache, *, softmax_scale, out, lse, scratch, mode=MODE_AUTO, stream=None):
        lib = load()
        self._keep = (q, block_table, cu_seqlens_q, seq_lens, num_computed_tokens, out, lse)
        num_blocks, bs, hkv, d = k_cache.shape
        total_q, hq, _ = q.shape
        n = int(seq_lens.shape[0])
        self._cpl = ctypes.c_int32(0)
        ptr = lambda a: ctypes.c_void_p(a.ctypes.data if hasattr(a, "ctypes") else a.data_ptr())
        self._fn = lib.cascade_step_host
        self._args = (ptr(q), ptr(block_table), int(block_table.shape[1]), ptr(cu_seqlens_q),
                      ptr(seq_lens), ptr(num_computed_tokens), n, total_q, _ptr(k_cache),
                      _ptr(v_cache), num_blocks, bs, hq, hkv, d, float(softmax_scale), mode,
                      ptr(out), ptr(lse), _ptr(scratch), scratch.numel(),
                      _stream_ptr(stream, k_cache.device), ctypes.byref(self._cpl))

    def __call__(self) -> int:
        _check(self._fn(*self._args), "cascade_step_host")
        return int(self._cpl.value)


def step_scratch_size(cu_seqlens_q, seq_lens, bt_row_stride, common_prefix_len, num_q_heads,
                      num_kv_heads, head_dim) -> int:
    lib = load()
    cu = _host_i32(cu_seqlens_q)
    sl = _host_i32(seq_lens)
    n = int(sl.shape[0])
    out = ctypes.c_size_t(0)
    _check(lib.csp_step_scratch_size(n, int(cu[-1]) if n else 0, cu.ctypes.data,
                                     sl.ctypes.data if n else None, int(bt_row_stride),
                                     int(common_prefix_len), num_q_heads, num_kv_heads,
                                     head_dim, ctypes.byref(out)), "csp_step_scratch_size")
    return int(out.value)


def apply_sinks(out, lse, sinks, *, stream=None):
    """csp_apply_sinks: per-head sink logits (fp32 device tensor [Hq], natural log)
    folded into a finished result (out bf16 [T, Hq, D] and lse fp32 [T, Hq], in place)."""
    import torch
    lib = load()
    t, hq, d = out.shape
    if sinks.dtype != torch.float32 or sinks.numel() != hq or not sinks.is_cuda:
        raise ValueError("sinks: an fp32 device tensor with one logit per query head")
    _check(lib.csp_apply_sinks(_ptr(out), _ptr(lse), _ptr(sinks.contiguous()), t, hq, d,
                               _stream_ptr(stream, out.device)), "csp_apply_sinks")
    return out, lse


def merge_states(prefix_out, prefix_lse, suffix_out, suffix_lse, *, out=None, out_lse=None,
                 stream=None):
    """LSE merge of two partials ([T, H, D] bf16 or fp32, LSE fp32 [T, H], natural log)."""
    import torch
    lib = load()
    t, h, d = prefix_out.shape
    if out is None:
        out = torch.empty((t, h, d), dtype=torch.bfloat16, device=prefix_out.device)
    if out_lse is None:
        out_lse = torch.empty((t, h), dtype=torch.float32, device=prefix_out.device)
    dt = DTYPE_F32 if prefix_out.dtype == torch.float32 else DTYPE_BF16
    assert suffix_out.dtype == prefix_out.dtype
    _check(lib.merge_states(_ptr(out), _ptr(out_lse), _ptr(prefix_out), _ptr(prefix_lse),
                            _ptr(suffix_out), _ptr(suffix_lse), t, h, d, dt,
                            _stream_ptr(stream, prefix_out.device)), "merge_states")
    return out, out_lse


def workspace_status(workspace, stream=None) -> int:
    lib = load()
    st = ctypes.c_int32(0)
    _check(lib.csp_workspace_status(_ptr(workspace), _stream_ptr(stream, workspace.device),
                                    ctypes.byref(st)), "csp_workspace_status")
    return int(st.value)


def version() -> int:
    return load().csp_version()
