"""NaN in a key that a row attends to reaches that row's output and LSE on every
path, as in the oracle (the reading "NaN inputs propagate"); rows that never see the
key stay finite and equal to the oracle's."""

import numpy as np
import pytest
import torch

import oracle
from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _batch(seed, where):
    g = torch.Generator().manual_seed(seed)
    b = workloads.build_batch(f"nan{seed}", [300, 320, 350, 310], [1, 1, 2, 1], 288,
                              num_q_heads=8, num_kv_heads=2, head_dim=64, gen=g)
    # K of one used key: in the shared prefix (key 10, KV head 0) or in request 2's own
    # keys (key 295, KV head 1)
    r, key, head = (0, 10, 0) if where == "prefix" else (2, 295, 1)
    blk = int(b.block_table[r, key // 16])
    b.k_cache[blk, key % 16, head, 5] = float("nan")
    return b


def _check(out, lse, ref_o, ref_l, what):
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy().astype(np.float64)
    want_nan = np.isnan(ref_l)
    assert want_nan.any(), "the planted NaN reaches some row in the oracle"
    assert np.array_equal(np.isnan(l), want_nan), f"{what}: NaN LSE rows differ"
    assert np.array_equal(np.isnan(o).any(-1), np.isnan(ref_o).any(-1)), \
        f"{what}: NaN output rows differ"
    ok = ~want_nan
    assert np.abs(o[ok] - ref_o[ok]).max() <= H.OUT_TOL, what
    assert (np.abs(l[ok] - ref_l[ok]) <= H.LSE_REL * np.maximum(1.0, np.abs(ref_l[ok]))).all(), what


@pytest.mark.parametrize("where", ["prefix", "suffix"])
def test_nan_key_propagates_on_every_schedule(where):
    b = _batch(91, where)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    out, lse = H.run_paged(b, dev)
    _check(out, lse, ref_o, ref_l, f"{where} flat")
    for sch in (csp.SCHEDULE_TWO_KERNELS, csp.SCHEDULE_SINGLE, csp.SCHEDULE_FUSED):
        out, lse = H.run_cascade(b, dev, cpl, schedule=sch)
        _check(out, lse, ref_o, ref_l, f"{where} cascade schedule {sch}")


@pytest.mark.parametrize("where", ["prefix", "suffix"])
def test_nan_byte_propagates_with_an_fp8_cache(where):
    b = _batch(92, where)
    ks, vs = 2.0 ** -6, 2.0 ** -6
    k8, v8 = workloads.to_fp8(b, ks, vs)   # the planted NaN becomes the E4M3 NaN byte
    dev = H.to_device(b)
    ref_o, ref_l = oracle.attention_fp8kv(b.q, k8, v8, b.block_table, b.cu_seqlens_q,
                                          b.seq_lens, b.scale, ks, vs)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    for c in (cpl, 0):
        out, lse = csp.attn_fp8kv(dev["q"], k8.cuda(), v8.cuda(), dev["bt"], dev["cu"],
                                  dev["sl"], max_seqlen_q=b.max_seqlen_q,
                                  max_seqlen_k=b.max_seqlen_k, softmax_scale=b.scale,
                                  k_scale=ks, v_scale=vs, common_prefix_len=c)
        _check(out, lse, ref_o, ref_l, f"{where} fp8 cpl={c}")
