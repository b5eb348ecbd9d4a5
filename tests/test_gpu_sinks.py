"""GPU parity of attention sinks: cascade_attn and paged_attn with per-head sink logits
(applied by csp_apply_sinks) against the oracle's standard path with the same sinks.

The sinks are drawn per head from N(0, 3^2), with one head at -inf (no sink: the plain
result) and one far above every score (the sink takes almost all the weight)."""

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _sinks(hq, seed):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal(hq) * 3.0
    s[0] = -np.inf
    s[-1] = 40.0
    return s


def _oracle(b, sinks, rows=None):
    import oracle
    return oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, b.scale, rows=rows, sinks=sinks)


CASES = [
    (51, [288] * 8, [1] * 8, 256, 8, 2, 64),
    (52, [530, 600, 777], [5, 17, 60], 512, 32, 8, 128),
    (53, [300, 320, 350, 310], [4, 3, 1, 2], 288, 32, 8, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_sinks_small_batches(case):
    seed, seq, ql, shared, hq, hkv, d = case
    g = torch.Generator().manual_seed(seed)
    b = workloads.build_batch(f"sinks{seed}", seq, ql, shared, num_q_heads=hq,
                              num_kv_heads=hkv, head_dim=d, gen=g)
    dev = H.to_device(b)
    s = _sinks(hq, seed)
    ref_o, ref_l = _oracle(b, s)
    st = torch.from_numpy(s).float().cuda()
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    out, lse = H.run_cascade(b, dev, cpl, sinks=st)
    H.compare(out, lse, ref_o, ref_l, what=f"sinks{seed} cascade")
    out, lse = H.run_paged(b, dev, sinks=st)
    H.compare(out, lse, ref_o, ref_l, what=f"sinks{seed} paged")


def test_sinks_decode_batch_sampled_rows():
    b = workloads.decode_batch()
    dev = H.to_device(b)
    s = _sinks(b.num_q_heads, 54)
    rows = H.sample_rows(b, 600, seed=54)
    ref_o, ref_l = _oracle(b, s, rows)
    cpl, _ = H.plan(b)
    out, lse = H.run_cascade(b, dev, cpl, sinks=torch.from_numpy(s).float().cuda())
    H.compare(out, lse, ref_o, ref_l, rows, what="sinks decode cascade")


def test_sinks_minus_inf_is_the_plain_result():
    b = workloads.tiny_decode()
    dev = H.to_device(b)
    cpl, _ = H.plan(b)
    o1, l1 = H.run_cascade(b, dev, cpl)
    o2, l2 = H.run_cascade(b, dev, cpl,
                           sinks=torch.full((b.num_q_heads,), float("-inf"), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
