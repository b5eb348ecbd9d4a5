"""Shared helpers of the GPU parity tests: move a generated batch to the device, run
the C-ABI paths, and compare with the oracle at the stated tolerances."""

from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from shared_prefix_paged_gb300 import csp

# bf16 output: max-abs error <= 2e-2; fp32 LSE: |error| <= 1e-3 * max(1, |lse|).  The
# LSE bound is relative with a floor of 1: |lse| can sit near 0 (a row whose scores sum
# to about 1), where a purely relative bound would demand more than fp32 accumulation
# of the sum gives.
OUT_TOL = 2e-2
LSE_REL = 1e-3

# When set, every comparison appends one JSON line (case, max-abs out error, worst
# LSE error as a fraction of its bound) to this file: the margins left under the
# tolerances are then measured, not argued.
_LOG = os.environ.get("CSP_PARITY_LOG")


def to_device(b, device="cuda"):
    dev = torch.device(device)
    return dict(q=b.q.to(dev), k=b.k_cache.to(dev), v=b.v_cache.to(dev),
                bt=torch.from_numpy(b.block_table).to(dev),
                cu=torch.from_numpy(b.cu_seqlens_q).to(dev),
                sl=torch.from_numpy(b.seq_lens).to(dev))


def run_paged(b, d, **kw):
    return csp.paged_attn(d["q"], d["k"], d["v"], d["bt"], d["cu"], d["sl"],
                          max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                          softmax_scale=b.scale, **kw)


def run_cascade(b, d, cpl, **kw):
    return csp.cascade_attn(d["q"], d["k"], d["v"], d["bt"], d["cu"], d["sl"],
                            max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                            common_prefix_len=cpl, softmax_scale=b.scale, **kw)


def plan(b, mode=csp.MODE_PAGE_THRESHOLDS):
    return csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                            block_size=b.block_size, num_q_heads=b.num_q_heads,
                            num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, mode=mode)


def sample_rows(b, n, seed=0):
    """n distinct (token, head) rows, always including the first and last row."""
    total = b.total_q * b.num_q_heads
    rng = np.random.default_rng(seed)
    flat = rng.choice(total, size=min(n, total), replace=False)
    flat = np.unique(np.concatenate([flat, [0, total - 1]]))
    return np.stack([flat // b.num_q_heads, flat % b.num_q_heads], 1).astype(np.int32)


def oracle_ref(b, rows=None):
    return oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, b.scale, rows=rows)


def compare(out, lse, ref_o, ref_l, rows=None, what=""):
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[rows[:, 0], rows[:, 1]]
        l = l[rows[:, 0], rows[:, 1]]
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = float(np.abs(o - ref_o).max(initial=0.0))
    assert err <= OUT_TOL, f"{what}: out max-abs error {err:.3e}"
    lerr = np.abs(l - ref_l)
    bound = LSE_REL * np.maximum(1.0, np.abs(ref_l))
    worst = float((lerr / bound).max(initial=0.0))
    if _LOG:
        with open(_LOG, "a") as f:
            f.write(json.dumps({"case": what, "out_err": err, "lse_frac": worst,
                                "rows": int(o.shape[0])}) + "\n")
    assert worst <= 1.0, f"{what}: lse error {worst:.2f}x the bound"
    return err
