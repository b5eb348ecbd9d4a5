"""GPU parity of the FP8 (E4M3) KV cache entry points (cascade_attn_fp8kv,
paged_attn_fp8kv) against the oracle's FP8 reading: attention over decode(byte) *
scale.  The caches are the generated bf16 caches quantised with torch's
float8_e4m3fn (an input draw); both sides read the same bytes."""

import numpy as np
import pytest
import torch

import oracle
from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _oracle(b, k8, v8, ks, vs, rows=None):
    return oracle.attention_fp8kv(b.q, k8, v8, b.block_table, b.cu_seqlens_q, b.seq_lens, b.scale,
                                  ks, vs, rows=rows)


def _run(b, dev, k8, v8, ks, vs, cpl):
    return csp.attn_fp8kv(dev["q"], k8.cuda(), v8.cuda(), dev["bt"], dev["cu"], dev["sl"],
                          max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                          softmax_scale=b.scale, k_scale=ks, v_scale=vs, common_prefix_len=cpl)


SCALES = [(2.0 ** -6, 2.0 ** -6), (0.0173, 0.0291)]


def _fitted_scales(b):
    """Per-tensor scales that map the cache's largest used magnitude (the +-1000 poison
    of unused slots aside) just inside E4M3's range, as a KV cache would pick them."""
    def amax(t):
        x = t.float().abs()
        return float(x[torch.isfinite(x) & (x < 999.0)].max())
    return amax(b.k_cache) / 440.0, amax(b.v_cache) / 440.0


@pytest.mark.parametrize("scales", SCALES, ids=["pow2", "other"])
@pytest.mark.parametrize("name", ["tiny", "chunked"])
def test_fp8_small_and_chunked_all_rows(name, scales):
    b = workloads.by_name(name)
    ks, vs = scales
    k8, v8 = workloads.to_fp8(b, ks, vs)
    dev = H.to_device(b)
    ref_o, ref_l = _oracle(b, k8, v8, ks, vs)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    for c in (cpl, 0):
        out, lse = _run(b, dev, k8, v8, ks, vs, c)
        H.compare(out, lse, ref_o, ref_l, what=f"{name} fp8 cpl={c} scales={scales}")


@pytest.mark.parametrize("name", ["decode", "long"])
def test_fp8_decode_and_long_sampled(name):
    b = workloads.by_name(name)
    ks, vs = _fitted_scales(b)
    k8, v8 = workloads.to_fp8(b, ks, vs)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 300, seed=71)
    ref_o, ref_l = _oracle(b, k8, v8, ks, vs, rows)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    for c in (cpl, 0):
        out, lse = _run(b, dev, k8, v8, ks, vs, c)
        H.compare(out, lse, ref_o, ref_l, rows=rows, what=f"{name} fp8 cpl={c}")


CASES = [
    # seed, seq_lens, q_lens, shared, Hq, Hkv, D: a request without a query, ragged
    # pages and row tiles, GQA groups 1 and 8, a long prefix in several key ranges
    (81, [300, 333, 290, 401], [1, 0, 7, 2], 288, 32, 8, 128),
    (82, [1500] * 6, [33, 65, 1, 2, 129, 7], 1024, 16, 16, 64),
    (83, [5000, 5100, 5010], [1, 1, 1], 4096, 64, 8, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_fp8_ragged_batches(case):
    seed, seq, ql, shared, hq, hkv, d = case
    g = torch.Generator().manual_seed(seed)
    b = workloads.build_batch(f"fp8_{seed}", seq, ql, shared, num_q_heads=hq, num_kv_heads=hkv,
                              head_dim=d, gen=g)
    ks, vs = _fitted_scales(b)
    k8, v8 = workloads.to_fp8(b, ks, vs)
    dev = H.to_device(b)
    ref_o, ref_l = _oracle(b, k8, v8, ks, vs)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    assert cpl > 0
    for c in (cpl, 0):
        out, lse = _run(b, dev, k8, v8, ks, vs, c)
        H.compare(out, lse, ref_o, ref_l, what=f"fp8 case{seed} cpl={c}")


def test_fp8_workspace_too_small_launches_nothing():
    b = workloads.tiny_decode()
    k8, v8 = workloads.to_fp8(b)
    dev = H.to_device(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    need = csp.workspace_size_fp8kv(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
                                    b.num_q_heads, b.num_kv_heads, b.head_dim)
    small = csp.alloc_workspace(need - 256, "cuda")
    out = torch.full_like(dev["q"], 7.0)
    with pytest.raises(csp.CspError) as e:
        csp.attn_fp8kv(dev["q"], k8.cuda(), v8.cuda(), dev["bt"], dev["cu"], dev["sl"],
                       max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                       softmax_scale=b.scale, k_scale=1.0, v_scale=1.0, common_prefix_len=cpl,
                       out=out, workspace=small)
    assert e.value.status == csp.CSP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
