"""The oracle: a plain, slow CPU statement of what cascade attention computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import anything in this package.  The CUDA
library and its Python binding never import it, and it imports nothing from
them.

* ``attention_oracle.c`` — standard, prefix-phase and suffix-phase attention over
  a paged KV cache, and the LSE merge, all in IEEE double (built with gcc, loaded
  with ctypes; see its header for the definitions and the passages they follow).
* ``planner.py`` — the common-prefix planner and the pages' thresholds.

Pins (in ``tests/``, run with ``-m "not gpu"``): dense attention through numpy /
scipy library routines on tiny inputs, closed forms (one key, zero query, equal
keys), the LSE-merge identity, page-layout invariance, the worked planner example
of §四 of "vLLM Cascade Attention：用法、场景与原理解析", a brute-force planner on
random tables, and planted-fault builds that each pin must catch.  The use-cascade
cost model beyond the pages' thresholds is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import planner  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

FULL, PREFIX, SUFFIX = 0, 1, 2


def _lib_path(mutant: int) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle with gcc (portable C, no machine-specific flags)."""
    path = _lib_path(mutant)
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{path}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        p = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_attention.argtypes = [p, p, p, i32, i32, p, i64, p, p, i32, i32, i32, i32, f64,
                                         i32, i32, p, p, i32]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [p, p, p, i32, i32, p, i64, p, p, i32, i32, i32, i32,
                                              f64, i32, i32, p, p, i64, p, p, i32]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_sinks.argtypes = [p, p, p, i32, i32, p, i64, p, p, i32, i32, i32,
                                               i32, f64, p, p, p, i64, p, p, i32]
        lib.oracle_attention_sinks.restype = ctypes.c_int
        lib.oracle_attention_fp8kv.argtypes = [p, p, p, i32, i32, p, i64, p, p, i32, i32, i32,
                                               i32, f64, f64, f64, i32, i32, p, p, i64, p, p,
                                               i32]
        lib.oracle_attention_fp8kv.restype = ctypes.c_int
        lib.oracle_e4m3_decode.argtypes = [p]
        lib.oracle_e4m3_decode.restype = None
        lib.oracle_merge_states.argtypes = [p, p, p, p, i64, i32, p, p]
        lib.oracle_merge_states.restype = None
        lib.oracle_mutant_id.restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def _bits(t) -> np.ndarray:
    """bf16 tensor (torch, CPU) or uint16 array -> contiguous uint16 bit array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = np.asarray(a.cpu().numpy() if hasattr(a, "cpu") else a)
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale, *,
              mode=FULL, cpl=0, rows=None, n_threads=None, mutant=0, sinks=None):
    """Oracle attention.

    q: bf16 [total_q, Hq, D]; k_cache / v_cache: bf16 [num_blocks, bs, Hkv, D];
    block_table int32 [N, W]; cu_seqlens_q int32 [N+1]; seq_lens int32 [N].
    rows: None for every (token, head) row, or an int array [n, 2] of
    (token, head) pairs.  sinks: None, or one logit per query head (float [Hq],
    natural log, -inf for none) for the standard path with attention sinks.
    Returns (out float64 [n_rows, D] or [total_q, Hq, D], lse float64 [n_rows] or
    [total_q, Hq]).
    """
    lib = _load(mutant)
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    total_q, Hq, D = qb.shape
    num_blocks, bs, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    bt = _i32(block_table)
    cu = _i32(cu_seqlens_q)
    sl = _i32(seq_lens)
    N = sl.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == N and cu.shape[0] == N + 1
    assert int(cu[-1]) == total_q
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    if sinks is not None:
        assert mode == FULL, "sinks belong to the standard path"
        sk = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64).reshape(-1))
        assert sk.shape[0] == Hq
        if rows is None:
            out = np.empty((total_q, Hq, D), np.float64)
            lse = np.empty((total_q, Hq), np.float64)
            st = lib.oracle_attention_sinks(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, bs,
                                            _ptr(bt), bt.shape[1], _ptr(cu), _ptr(sl), N, Hq,
                                            Hkv, D, float(scale), _ptr(sk), None, None, 0,
                                            _ptr(out), _ptr(lse), int(n_threads))
        else:
            rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
            rt = np.ascontiguousarray(rows[:, 0])
            rh = np.ascontiguousarray(rows[:, 1])
            n = rows.shape[0]
            out = np.empty((n, D), np.float64)
            lse = np.empty((n,), np.float64)
            st = lib.oracle_attention_sinks(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, bs,
                                            _ptr(bt), bt.shape[1], _ptr(cu), _ptr(sl), N, Hq,
                                            Hkv, D, float(scale), _ptr(sk), _ptr(rt), _ptr(rh),
                                            n, _ptr(out), _ptr(lse), int(n_threads))
    elif rows is None:
        out = np.empty((total_q, Hq, D), np.float64)
        lse = np.empty((total_q, Hq), np.float64)
        st = lib.oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, bs, _ptr(bt),
                                  bt.shape[1], _ptr(cu), _ptr(sl), N, Hq, Hkv, D, float(scale),
                                  mode, int(cpl), _ptr(out), _ptr(lse), int(n_threads))
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        rt = np.ascontiguousarray(rows[:, 0])
        rh = np.ascontiguousarray(rows[:, 1])
        n = rows.shape[0]
        out = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
        st = lib.oracle_attention_rows(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, bs, _ptr(bt),
                                       bt.shape[1], _ptr(cu), _ptr(sl), N, Hq, Hkv, D,
                                       float(scale), mode, int(cpl), _ptr(rt), _ptr(rh), n,
                                       _ptr(out), _ptr(lse), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attention failed with status {st} (bad block id or shape)")
    return out, lse


def _bytes(t) -> np.ndarray:
    """uint8 tensor (torch, CPU) or array -> contiguous uint8 array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint8
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.uint8, t.dtype
    return t.detach().cpu().contiguous().numpy()


def e4m3_values(*, mutant=0) -> np.ndarray:
    """float64 [256]: the value of every E4M3 byte, from the format's definition."""
    out = np.empty(256, np.float64)
    _load(mutant).oracle_e4m3_decode(_ptr(out))
    return out


def attention_fp8kv(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale, k_scale,
                    v_scale, *, mode=FULL, cpl=0, rows=None, n_threads=None, mutant=0):
    """Oracle attention over an FP8 (E4M3) KV cache with per-tensor scales.

    k_cache / v_cache: uint8 [num_blocks, bs, Hkv, D] of E4M3 bytes; an element's value
    is decode(byte) * k_scale (or * v_scale).  Other arguments and the result: as for
    attention()."""
    lib = _load(mutant)
    qb, kb, vb = _bits(q), _bytes(k_cache), _bytes(v_cache)
    total_q, Hq, D = qb.shape
    num_blocks, bs, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    bt, cu, sl = _i32(block_table), _i32(cu_seqlens_q), _i32(seq_lens)
    N = sl.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == N and cu.shape[0] == N + 1
    assert int(cu[-1]) == total_q
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    if rows is None:
        out = np.empty((total_q, Hq, D), np.float64)
        lse = np.empty((total_q, Hq), np.float64)
        rt = rh = None
        n = total_q * Hq
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        rt = np.ascontiguousarray(rows[:, 0])
        rh = np.ascontiguousarray(rows[:, 1])
        n = rows.shape[0]
        out = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
    st = lib.oracle_attention_fp8kv(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, bs, _ptr(bt),
                                    bt.shape[1], _ptr(cu), _ptr(sl), N, Hq, Hkv, D, float(scale),
                                    float(k_scale), float(v_scale), mode, int(cpl),
                                    _ptr(rt) if rt is not None else None,
                                    _ptr(rh) if rh is not None else None, n, _ptr(out),
                                    _ptr(lse), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attention_fp8kv failed with status {st}")
    return out, lse


def merge_states(o1, l1, o2, l2, *, mutant=0):
    """LSE merge of two partials; o: float64 [..., D], l: float64 [...]."""
    lib = _load(mutant)
    o1 = np.ascontiguousarray(o1, np.float64)
    o2 = np.ascontiguousarray(o2, np.float64)
    l1 = np.ascontiguousarray(l1, np.float64)
    l2 = np.ascontiguousarray(l2, np.float64)
    D = o1.shape[-1]
    n = l1.size
    assert o1.size == n * D and o2.shape == o1.shape and l2.shape == l1.shape
    out = np.empty_like(o1)
    lse = np.empty_like(l1)
    lib.oracle_merge_states(_ptr(o1), _ptr(l1), _ptr(o2), _ptr(l2), n, D, _ptr(out), _ptr(lse))
    return out, lse
