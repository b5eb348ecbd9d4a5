"""GPU parity of the multi-level cascade (cascade_attn_levels): the library's level
planner, then attention through every segment, each request's suffix and the LSE
merge, against the oracle's standard path (the result the levels reach up to
rounding: "vLLM Cascade Attention：用法、场景与原理解析" §一 and §七)."""

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def run_levels(b, dev, max_levels, *, workspace=None, segs=None, start=None):
    if segs is None:
        segs, start = csp.cascade_plan_levels(b.block_table, b.seq_lens,
                                              b.num_computed_tokens,
                                              block_size=b.block_size, max_levels=max_levels)
    max_suffix = int((b.seq_lens - start).max()) if b.num_reqs else 0
    out, lse = csp.cascade_attn_levels(
        dev["q"], dev["k"], dev["v"], dev["bt"], dev["cu"], dev["sl"],
        max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k, segments=segs,
        suffix_start=torch.from_numpy(start).cuda(), max_suffix_len=max_suffix,
        softmax_scale=b.scale, workspace=workspace)
    return out, lse, segs


def _poisoned_workspace(b, segs, start):
    """A workspace whose slots hold NaN bytes: a slot no segment writes must be skipped
    by its lse, never read for its values."""
    max_suffix = int((b.seq_lens - start).max())
    n = csp.workspace_size_levels(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, segs,
                                  max_suffix, b.num_q_heads, b.num_kv_heads, b.head_dim)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0   # the status word starts clear
    return ws


@pytest.mark.parametrize("name", ["tree", "tree_chunked"])
@pytest.mark.parametrize("max_levels", [1, 2, 3])
def test_tree_batches_all_rows(name, max_levels):
    b = workloads.by_name(name)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    segs, start = csp.cascade_plan_levels(b.block_table, b.seq_lens, b.num_computed_tokens,
                                          max_levels=max_levels)
    assert int(segs[:, 0].max()) == min(max_levels, 3) - 1
    ws = _poisoned_workspace(b, segs, start)
    out, lse, _ = run_levels(b, dev, max_levels, workspace=ws, segs=segs, start=start)
    H.compare(out, lse, ref_o, ref_l, what=f"{name} levels={max_levels}")
    assert csp.workspace_status(ws) == 0


def test_tree_head_dim_64():
    b = workloads.tree_decode(seed=1007, head_dim=64)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse, segs = run_levels(b, dev, 3)
    assert int(segs[:, 0].max()) == 2
    H.compare(out, lse, ref_o, ref_l, what="tree D64")


def test_deep_segments_with_several_key_ranges():
    # level-0 and level-1 segments long enough (4096 and 2048 keys) to take 4 and 2 key
    # ranges each, and a third level of 1024 keys; 24 decode requests
    g = torch.Generator().manual_seed(1008)
    chunks = [4096, 2048, 2048, 1024, 1024]
    paths = [(0, 1, 3)] * 6 + [(0, 1, 4)] * 6 + [(0, 2)] * 12
    private = torch.randint(16, 300, (24,), generator=g).tolist()
    b = workloads.build_tree_batch("tree_long", chunks, paths, private, [1] * 24,
                                   num_q_heads=32, num_kv_heads=8, head_dim=128, gen=g)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 400, seed=1008)
    ref_o, ref_l = H.oracle_ref(b, rows)
    out, lse, segs = run_levels(b, dev, 3)
    assert [tuple(s[:5]) for s in segs.tolist()] == [
        (0, 0, 24, 0, 4096), (1, 0, 12, 4096, 6144), (2, 0, 6, 6144, 7168),
        (2, 6, 12, 6144, 7168), (1, 12, 24, 4096, 6144)]
    H.compare(out, lse, ref_o, ref_l, rows=rows, what="tree_long")


def test_two_level_batches_through_the_level_path():
    # the decode and chunked-prefill batches have one shared prefix: one level
    for name in ("decode", "chunked"):
        b = workloads.by_name(name)
        dev = H.to_device(b)
        rows = H.sample_rows(b, 300, seed=1009)
        ref_o, ref_l = H.oracle_ref(b, rows)
        out, lse, segs = run_levels(b, dev, 3)
        assert segs.shape[0] == 1
        H.compare(out, lse, ref_o, ref_l, rows=rows, what=f"{name} via levels")


def test_no_segments_is_the_standard_path():
    b = workloads.tiny_decode()
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    segs = np.zeros((0, 7), np.int32)
    start = np.zeros(b.num_reqs, np.int32)
    out, lse, _ = run_levels(b, dev, 3, segs=segs, start=start)
    H.compare(out, lse, ref_o, ref_l, what="no segments")


def test_segment_without_query_rows():
    # the second family's requests have no query this step: its segment has no rows
    g = torch.Generator().manual_seed(1010)
    chunks = [512, 256, 256]
    paths = [(0, 1)] * 4 + [(0, 2)] * 4
    b = workloads.build_tree_batch("tree_idle", chunks, paths, [40] * 8,
                                   [1, 2, 1, 3, 0, 0, 0, 0], num_q_heads=8, num_kv_heads=2,
                                   head_dim=64, gen=g)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse, segs = run_levels(b, dev, 3)
    assert any(s[5] == s[6] for s in segs.tolist())
    H.compare(out, lse, ref_o, ref_l, what="segment without rows")


@pytest.mark.parametrize("shape", [(8, 16, 2048, 4096), (4, 16, 1024, 8192), (16, 8, 4096, 2048)])
def test_family_batches_the_benchmark_times(shape):
    fam, per, system, doc = shape
    b = workloads.tree_families(families=fam, per_family=per, system=system, doc=doc)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 500, seed=1012)
    ref_o, ref_l = H.oracle_ref(b, rows)
    out, lse, segs = run_levels(b, dev, 3)
    assert segs.shape[0] == 1 + fam
    H.compare(out, lse, ref_o, ref_l, rows=rows, what=f"families {shape}")
