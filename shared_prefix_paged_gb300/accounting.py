"""Algorithmic byte and flop counts used for the roofline figures.

"vLLM Cascade Attention：用法、场景与原理解析" §五 counts KV traffic in tokens: the
standard path loads N x (P + S) tokens (every request reads its whole KV), cascade
loads P + N x S (the shared prefix once, then each suffix).  These helpers turn
such counts into bytes for a concrete batch: one KV token is K and V for every
KV head, 2 x Hkv x D bf16 values.
"""

from __future__ import annotations

import numpy as np


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return 2 * num_kv_heads * head_dim * elem_bytes


def flat_kv_tokens(seq_lens) -> int:
    """Standard path: every request reads all of its KV."""
    return int(np.asarray(seq_lens, dtype=np.int64).sum())


def cascade_kv_tokens(seq_lens, common_prefix_len: int) -> int:
    """Cascade: the shared prefix once, then each request's KV after it."""
    s = np.asarray(seq_lens, dtype=np.int64)
    if s.size == 0:
        return 0
    return int(common_prefix_len) + int((s - common_prefix_len).sum())


def prefix_flops(total_q: int, num_q_heads: int, head_dim: int, common_prefix_len: int) -> int:
    """QK^T and PV of the prefix phase: 2 matmuls x 2 flops per multiply-add."""
    return 4 * total_q * num_q_heads * common_prefix_len * head_dim


def cascade_min_bytes(batch, common_prefix_len: int) -> int:
    """Minimal HBM bytes of one cascade call: KV once, q read, out (bf16) + lse written."""
    kv = cascade_kv_tokens(batch.seq_lens, common_prefix_len) * kv_bytes_per_token(
        batch.num_kv_heads, batch.head_dim)
    rows = batch.total_q * batch.num_q_heads
    return kv + rows * batch.head_dim * 2 * 2 + rows * 4


def flat_min_bytes(batch) -> int:
    """Algorithmic bytes of the standard path: each request's whole KV, q, out and lse."""
    kv = flat_kv_tokens(batch.seq_lens) * kv_bytes_per_token(batch.num_kv_heads, batch.head_dim)
    rows = batch.total_q * batch.num_q_heads
    return kv + rows * batch.head_dim * 2 * 2 + rows * 4


def levels_kv_tokens(seq_lens, segments, suffix_start) -> int:
    """Multi-level cascade (§七, num_levels): each segment's shared keys once, then each
    request's KV after its deepest segment.  segments: rows (level, r_lo, r_hi, k_lo,
    k_hi, ...)."""
    s = np.asarray(seq_lens, dtype=np.int64)
    st = np.asarray(suffix_start, dtype=np.int64)
    shared = sum(int(g[4]) - int(g[3]) for g in segments)
    return shared + int((s - st).sum())


def levels_min_bytes(batch, segments, suffix_start) -> int:
    """Minimal HBM bytes of one multi-level call: KV once, q read, out + lse written."""
    kv = levels_kv_tokens(batch.seq_lens, segments, suffix_start) * kv_bytes_per_token(
        batch.num_kv_heads, batch.head_dim)
    rows = batch.total_q * batch.num_q_heads
    return kv + rows * batch.head_dim * 2 * 2 + rows * 4
