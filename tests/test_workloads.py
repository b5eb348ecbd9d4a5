"""Generator and byte-accounting checks (CPU only)."""

import json
import math
import os

import numpy as np
import torch

import oracle
from oracle import planner
from shared_prefix_paged_gb300 import accounting, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_traffic_example_from_the_pages():
    with open(os.path.join(GOLDEN, "kv_traffic_example.json"), encoding="utf-8") as f:
        ex = json.load(f)
    n, p, s = ex["num_reqs"], ex["prefix_tokens"], ex["suffix_tokens"]
    seq = [p + s] * n
    flat = accounting.flat_kv_tokens(seq)
    casc = accounting.cascade_kv_tokens(seq, p)
    assert flat == ex["expected"]["standard_kv_tokens"]
    assert casc == ex["expected"]["cascade_kv_tokens"]
    assert casc - p == ex["expected"]["cascade_suffix_kv_tokens"]
    assert round(flat / casc) == ex["expected"]["reduction"]
    # the same example in bytes (8 KV heads, D 128): 50,331,648 B for cascade
    assert casc * accounting.kv_bytes_per_token(8, 128) == 50_331_648


def test_generator_is_deterministic_and_shaped():
    a = workloads.tiny_decode()
    b = workloads.tiny_decode()
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert np.array_equal(a.block_table, b.block_table)
    assert a.q.shape == (8, 8, 64) and a.k_cache.shape[1:] == (16, 2, 64)
    assert a.scale == 0.125
    assert list(a.seq_lens) == [288] * 8 and list(a.q_lens) == [1] * 8
    assert a.k_cache.is_contiguous() and a.v_cache.is_contiguous()


def test_poison_placement():
    b = workloads.chunked_prefill()
    bs = b.block_size
    used_ids = set()
    for r in range(b.num_reqs):
        u = -(-int(b.seq_lens[r]) // bs)
        used_ids.update(int(x) for x in b.block_table[r, :u])
        pad = b.block_table[r, u:]
        assert pad.size > 0
        for x in pad:       # padding points at poisoned (NaN) blocks
            assert torch.isnan(b.k_cache[int(x)].float()).all()
    for blk in used_ids:
        assert not torch.isnan(b.k_cache[blk].float()).any()
    # tails of partially filled private last blocks hold +-1000
    for r in range(b.num_reqs):
        s = int(b.seq_lens[r])
        if s % bs and (s - 1) // bs >= b.shared_blocks:
            blk = int(b.block_table[r, (s - 1) // bs])
            assert b.k_cache[blk, s % bs:].float().abs().max() == 1000.0


def test_planner_oracle_on_generated_batches():
    b = workloads.decode_batch(n=8, p=512, s=32)
    assert planner.plan(b.block_table, b.seq_lens, b.num_computed_tokens, 16) == (512, True)
    c = workloads.chunked_prefill()
    cpl, _ = planner.plan(c.block_table, c.seq_lens, c.num_computed_tokens, 16)
    assert cpl == 2048
    cap = workloads.chunked_prefill(seed=1013, shared_tokens=3072)
    cpl, _ = planner.plan(cap.block_table, cap.seq_lens, cap.num_computed_tokens, 16)
    m = int(cap.num_computed_tokens.min())
    assert m < 3072 and cpl == (m // 16) * 16


def test_oracle_never_touches_poison_on_tiny_batch():
    b = workloads.tiny_decode()
    o, l = oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, b.scale)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    # the query sees all 288 keys: lse >= log-mean-exp bound is finite and moderate
    assert np.all(l > math.log(1)) or np.all(np.isfinite(l))
