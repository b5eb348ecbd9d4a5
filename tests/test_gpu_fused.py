"""GPU parity of the fused cascade schedule (one launch: the prefix phase's CTAs and
tcgen05 suffix CTAs in one grid, each row group merged by its last contributor)
against the oracle, on prefill-shaped and decode batches."""

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

FUSED = dict(schedule=csp.SCHEDULE_FUSED)


@pytest.mark.parametrize("name", ["tiny", "chunked", "chunked_cap"])
def test_fused_small_and_chunked_all_rows(name):
    b = workloads.by_name(name)
    dev = H.to_device(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse = H.run_cascade(b, dev, cpl, **FUSED)
    H.compare(out, lse, ref_o, ref_l, what=f"{name} fused")


@pytest.mark.parametrize("name", ["decode", "long"])
def test_fused_decode_and_long_prefix_sampled(name):
    b = workloads.by_name(name)
    dev = H.to_device(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    rows = H.sample_rows(b, 400, seed=31)
    ref_o, ref_l = H.oracle_ref(b, rows)
    out, lse = H.run_cascade(b, dev, cpl, **FUSED)
    H.compare(out, lse, ref_o, ref_l, rows=rows, what=f"{name} fused")


CASES = [
    # seed, seq_lens, q_lens, shared, Hq, Hkv, D: several prefix ranges and suffix
    # splits, a request with no query, ragged row tiles, group 1 and 8
    (61, [2100, 2300, 4000, 2600], [70, 1, 300, 0], 2048, 32, 8, 128),
    (62, [1500] * 6, [33, 65, 1, 2, 129, 7], 1024, 16, 16, 64),
    (63, [700, 900, 1100], [64, 64, 64], 512, 64, 8, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_fused_ragged_batches(case):
    seed, seq, ql, shared, hq, hkv, d = case
    g = torch.Generator().manual_seed(seed)
    b = workloads.build_batch(f"fused{seed}", seq, ql, shared, num_q_heads=hq,
                              num_kv_heads=hkv, head_dim=d, gen=g)
    dev = H.to_device(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    assert cpl > 0
    ref_o, ref_l = H.oracle_ref(b)
    # the workspace left dirty by an earlier call: the counters start from zero anyway
    ws = csp.alloc_workspace(csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q,
                                                b.max_seqlen_k, cpl, hq, hkv, d), "cuda")
    for _ in range(2):
        out, lse = H.run_cascade(b, dev, cpl, workspace=ws, **FUSED)
    H.compare(out, lse, ref_o, ref_l, what=f"fused case{seed}")
    assert csp.workspace_status(ws) == 0
