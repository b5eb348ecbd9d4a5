"""Seeded synthetic batches for cascade attention over a paged KV cache.

This module only draws inputs: lengths, a shuffled physical block pool, block
tables, and bf16 Q/K/V.  It holds none of the method's arithmetic (no planner,
no attention, no merge), so both the CUDA path and the CPU oracle can take their
inputs from it.

Shapes follow the workloads on "vLLM Cascade Attention：用法、场景与原理解析"
(§五: N=64 requests, shared prefix P=4096, suffix S=128, decode) plus four more
batch shapes of the same kind (tiny decode, chunked prefill, long prefix, and an
N x P sweep).  No public dataset is involved: values are N(0, 1) draws.

Recipe (one torch CPU generator per batch, draws always in this order):
  1. lengths (config specific);
  2. ``randperm`` of the physical block pool, whose size is
     ceil(1.25 * blocks needed) + 1; the shared prefix takes the first ids of the
     permutation, then each request's private blocks in request order; the rest
     stay unused;
  3. q, then K, then V: ``randn`` in fp32, rounded to bf16 (K times ``k_scale``
     first, exact for powers of two).
Then poisoning, so that a read of anything outside the batch shows up:
  * unused blocks hold NaN in K and V, and every block-table entry past a
    request's last used block points at one of them;
  * slots past seq_len in a request's last (private) block hold +-1000.

A request's KV holds its already-computed tokens followed by this step's query
tokens (seq_len = num_computed_tokens + q_len), as in the R1/R2 example of §四.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16
SWEEP_N = (4, 8, 16, 32, 64, 128, 256)
SWEEP_P = (128, 256, 1024, 4096, 16384)


@dataclasses.dataclass
class Batch:
    """One batch of inputs, all on the CPU.  Tensors are contiguous."""
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    seq_lens: np.ndarray            # int32 [N], KV length incl. this step's queries
    num_computed_tokens: np.ndarray  # int32 [N]
    q_lens: np.ndarray              # int32 [N]
    cu_seqlens_q: np.ndarray        # int32 [N + 1]
    block_table: np.ndarray         # int32 [N, W]
    num_blocks: int
    shared_blocks: int              # leading blocks the generator made physically shared
    q: torch.Tensor                 # bf16 [total_q, Hq, D]
    k_cache: torch.Tensor           # bf16 [num_blocks, bs, Hkv, D]
    v_cache: torch.Tensor           # bf16 [num_blocks, bs, Hkv, D]

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if self.num_reqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens.max()) if self.num_reqs else 0


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def build_batch(name: str, seq_lens, q_lens, shared_tokens: int, *, num_q_heads: int,
                num_kv_heads: int, head_dim: int, gen: torch.Generator,
                block_size: int = BLOCK_SIZE, scale: Optional[float] = None,
                k_scale: float = 1.0, pad_cols: int = 2) -> Batch:
    """Lay out one batch given its lengths (steps 2-3 of the module recipe).

    ``shared_tokens`` leading tokens live in physical blocks shared by every
    request (rounded up to whole blocks; a request uses only as many of them as
    its own length needs).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    n = int(seq_lens.shape[0])
    assert q_lens.shape == (n,)
    assert np.all(q_lens >= 0) and np.all(seq_lens >= q_lens)
    bs = block_size
    shared_blocks = _cdiv(shared_tokens, bs)
    used = [_cdiv(int(s), bs) for s in seq_lens]
    private = [u - min(u, shared_blocks) for u in used]
    needed = shared_blocks + sum(private)
    num_blocks = math.ceil(1.25 * needed) + 1
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int64)
    shared_ids = perm[:shared_blocks]
    cursor = shared_blocks
    width = max(used, default=0) + pad_cols
    unused = perm[needed:]
    assert unused.size >= 1
    pad_id = int(unused[0])
    table = np.full((n, max(width, 1)), pad_id, dtype=np.int64)
    last_private = []  # (block id, first tail slot) of partially filled private last blocks
    for r in range(n):
        k_shared = min(used[r], shared_blocks)
        table[r, :k_shared] = shared_ids[:k_shared]
        ids = perm[cursor:cursor + private[r]]
        cursor += private[r]
        table[r, k_shared:used[r]] = ids
        tail = int(seq_lens[r]) % bs
        if private[r] > 0 and tail != 0:
            last_private.append((int(ids[-1]), tail))
    return _draw(name, seq_lens, q_lens, table, num_blocks, shared_blocks, unused, last_private,
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 gen=gen, block_size=bs, scale=scale, k_scale=k_scale)


def _draw(name, seq_lens, q_lens, table, num_blocks, shared_blocks, unused, last_private, *,
          num_q_heads, num_kv_heads, head_dim, gen, block_size, scale, k_scale) -> Batch:
    """Step 3 of the module recipe and the poisoning, for a laid-out block table."""
    n = int(seq_lens.shape[0])
    bs = block_size
    total_q = int(q_lens.sum())
    hq, hkv, d = num_q_heads, num_kv_heads, head_dim
    q = torch.randn((total_q, hq, d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((num_blocks, bs, hkv, d), generator=gen, dtype=torch.float32)
    if k_scale != 1.0:
        k.mul_(k_scale)
    k = k.to(torch.bfloat16)
    v = torch.randn((num_blocks, bs, hkv, d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    if unused.size:
        idx = torch.from_numpy(unused)
        k[idx] = float("nan")
        v[idx] = float("nan")
    for blk, tail in last_private:
        sign = torch.where(torch.arange(d) % 2 == 0, 1.0, -1.0).to(torch.bfloat16)
        k[blk, tail:] = 1000.0 * sign
        v[blk, tail:] = -1000.0 * sign
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return Batch(
        name=name, block_size=bs, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
        seq_lens=seq_lens.astype(np.int32), num_computed_tokens=(seq_lens - q_lens).astype(np.int32),
        q_lens=q_lens.astype(np.int32), cu_seqlens_q=cu, block_table=table.astype(np.int32),
        num_blocks=num_blocks, shared_blocks=shared_blocks, q=q.contiguous(),
        k_cache=k.contiguous(), v_cache=v.contiguous())


def build_tree_batch(name: str, chunk_lens, paths, private_lens, q_lens, *,
                     num_q_heads: int, num_kv_heads: int, head_dim: int,
                     gen: torch.Generator, block_size: int = BLOCK_SIZE,
                     scale: Optional[float] = None, pad_cols: int = 2) -> Batch:
    """A batch whose requests share chunks of KV along a tree: request r's KV is the
    chunks ``paths[r]`` (ids into ``chunk_lens``, each a whole number of blocks, laid
    out once and shared by every request whose path holds it), then
    ``private_lens[r]`` tokens of its own; its last ``q_lens[r]`` positions are this
    step's queries.  Physical ids: the chunks' blocks take the first ids of the pool's
    permutation in chunk order, then each request's private blocks; draws and
    poisoning as for ``build_batch``."""
    bs = block_size
    chunk_lens = [int(c) for c in chunk_lens]
    assert all(c > 0 and c % bs == 0 for c in chunk_lens)
    n = len(paths)
    assert len(private_lens) == n and len(q_lens) == n
    seq_lens = np.array([sum(chunk_lens[c] for c in paths[r]) + int(private_lens[r])
                         for r in range(n)], np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    assert np.all(q_lens >= 0) and np.all(seq_lens >= q_lens)
    chunk_blocks = [c // bs for c in chunk_lens]
    private = [_cdiv(int(p), bs) for p in private_lens]
    needed = sum(chunk_blocks) + sum(private)
    num_blocks = math.ceil(1.25 * needed) + 1
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(chunk_blocks)]).astype(np.int64)
    cursor = int(starts[-1])
    used = [sum(chunk_blocks[c] for c in paths[r]) + private[r] for r in range(n)]
    width = max(used, default=0) + pad_cols
    unused = perm[needed:]
    assert unused.size >= 1
    table = np.full((n, max(width, 1)), int(unused[0]), dtype=np.int64)
    last_private = []
    for r in range(n):
        col = 0
        for c in paths[r]:
            table[r, col:col + chunk_blocks[c]] = perm[starts[c]:starts[c + 1]]
            col += chunk_blocks[c]
        ids = perm[cursor:cursor + private[r]]
        cursor += private[r]
        table[r, col:col + private[r]] = ids
        tail = int(private_lens[r]) % bs
        if private[r] > 0 and tail != 0:
            last_private.append((int(ids[-1]), tail))
    first = {p[0] for p in paths if p}
    shared_blocks = chunk_blocks[first.pop()] if len(first) == 1 and all(paths) else 0
    return _draw(name, seq_lens, q_lens, table, num_blocks, shared_blocks, unused,
                 last_private, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, gen=gen, block_size=bs, scale=scale, k_scale=1.0)


def to_fp8(b: Batch, k_scale: float = 2.0 ** -6, v_scale: float = 2.0 ** -6):
    """The batch's K and V caches as E4M3 bytes (uint8, same shape) for per-tensor scales
    k_scale, v_scale: byte = E4M3(x / scale), by torch's float8_e4m3fn rounding (an
    input draw, not the method).  Poisoned values stay unusable: NaN stays NaN and the
    +-1000 tail slots saturate to NaN.  Returns (k_bytes, v_bytes)."""
    k8 = (b.k_cache.float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (b.v_cache.float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return k8.contiguous(), v8.contiguous()


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(seed)


def tiny_decode(seed: int = 1001) -> Batch:
    """8 requests, 256-token shared prefix, 32-token suffix (incl. the query), 1 query each;
    Hq 8, Hkv 2, D 64, scale 1/8."""
    g = _gen(seed)
    n, p, s = 8, 256, 32
    return build_batch("tiny_decode_N8_P256_S32", [p + s] * n, [1] * n, p, num_q_heads=8,
                       num_kv_heads=2, head_dim=64, gen=g, scale=0.125)


def decode_batch(seed: int = 1002, n: int = 64, p: int = 4096, s: int = 128,
                 num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128) -> Batch:
    """N requests sharing a P-token prefix, each with S private tokens (the last is the
    single query token).  Default: the N=64, P=4096, S=128 decode batch."""
    g = _gen(seed)
    return build_batch(f"decode_N{n}_P{p}_S{s}", [p + s] * n, [1] * n, p,
                       num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, gen=g)


def chunked_prefill(seed: int = 1003, shared_tokens: int = 2048) -> Batch:
    """32 requests; num_computed_tokens ~ U[2048, 3072], q_len ~ U[1, 64] (inclusive);
    the first ``shared_tokens`` tokens sit in shared blocks (2048: the plain mix; 3072:
    a shared run longer than some requests' computed KV, so the min-computed cap bites)."""
    g = _gen(seed)
    n = 32
    nc = torch.randint(2048, 3073, (n,), generator=g).numpy()
    ql = torch.randint(1, 65, (n,), generator=g).numpy()
    return build_batch(f"chunked_prefill_N32_shared{shared_tokens}", nc + ql, ql, shared_tokens,
                       num_q_heads=32, num_kv_heads=8, head_dim=128, gen=g)


def long_prefix(seed: int = 1004) -> Batch:
    """256 requests, 16384-token shared prefix, suffix ~ U[64, 1024] (incl. the query),
    1 query each; Hq 64, Hkv 8, D 128; K drawn N(0,1) then scaled by 2."""
    g = _gen(seed)
    n, p = 256, 16384
    s = torch.randint(64, 1025, (n,), generator=g).numpy()
    return build_batch("long_prefix_N256_P16384", p + s, np.ones(n, np.int64), p,
                       num_q_heads=64, num_kv_heads=8, head_dim=128, gen=g, k_scale=2.0)


def sweep_point(n: int, p: int, s: int = 128) -> Batch:
    """One point of the N x P decode sweep (suffix S=128, Hq 32, Hkv 8, D 128)."""
    i_n = SWEEP_N.index(n) if n in SWEEP_N else 0
    i_p = SWEEP_P.index(p) if p in SWEEP_P else 0
    return decode_batch(seed=1000 + 100 * i_n + i_p, n=n, p=p, s=s)


def tree_decode(seed: int = 1005, head_dim: int = 128, chunked: bool = False) -> Batch:
    """A three-level decode batch: 16 requests over one 1024-token system prompt; two
    families of 8 over their own documents (512 and 768 tokens); within the first
    family two groups of 4 over 256-token sub-documents; 40 to 200 private tokens each
    (the last one the query).  Hq 32, Hkv 8.  chunked: request 5 prefills its last 300
    tokens (past its private ones, into its sub-document: the planner's cap then
    shortens its segments) and request 12 its last 64."""
    g = _gen(seed)
    chunks = [1024, 512, 768, 256, 256]
    paths = [(0, 1, 3)] * 4 + [(0, 1, 4)] * 4 + [(0, 2)] * 8
    private = torch.randint(40, 201, (16,), generator=g).tolist()
    q = [1] * 16
    if chunked:
        q[5] = 300
        q[12] = 64
    return build_tree_batch(f"tree_decode_D{head_dim}" + ("_chunked" if chunked else ""),
                            chunks, paths, private, q, num_q_heads=32, num_kv_heads=8,
                            head_dim=head_dim, gen=g)


def tree_families(seed: int = 1011, families: int = 8, per_family: int = 16,
                  system: int = 2048, doc: int = 4096, s: int = 128) -> Batch:
    """Families of decode requests over one system prompt: ``families`` groups of
    ``per_family`` requests, each group over its own ``doc``-token document after the
    ``system``-token prompt, each request with ``s`` private tokens (the last one the
    query).  Hq 32, Hkv 8, D 128.  Default: 128 requests, 2048 + 4096 + 128 tokens."""
    g = _gen(seed)
    chunks = [system] + [doc] * families
    paths = [(0, 1 + f) for f in range(families) for _ in range(per_family)]
    n = families * per_family
    return build_tree_batch(f"tree_F{families}x{per_family}_sys{system}_doc{doc}_S{s}",
                            chunks, paths, [s] * n, [1] * n, num_q_heads=32, num_kv_heads=8,
                            head_dim=128, gen=g)


def by_name(name: str) -> Batch:
    """The named batch shapes used by the tests and the benchmark."""
    table = {
        "tiny": tiny_decode,
        "decode": decode_batch,
        "chunked": chunked_prefill,
        "chunked_cap": lambda: chunked_prefill(seed=1013, shared_tokens=3072),
        "long": long_prefix,
        "tree": tree_decode,
        "tree_chunked": lambda: tree_decode(seed=1006, chunked=True),
        "families": tree_families,
    }
    return table[name]()
