"""Multi-level cascade planner in the library: equal to the planner oracle (pinned in
test_oracle_levels.py) on random prefix trees and generated batches, its errors, and the
library's host checks of a segment list.  No device code runs here."""

import ctypes

import numpy as np
import pytest

from oracle import planner
from shared_prefix_paged_gb300 import csp, workloads
from tests.test_oracle_levels import BS, _hand_table, _random_tree


def _c_plan(bt, seq, nc, max_levels):
    segs, start = csp.cascade_plan_levels(bt, seq, nc, block_size=BS, max_levels=max_levels)
    return [tuple(int(x) for x in s[:5]) for s in segs], start.tolist(), segs


@pytest.mark.parametrize("max_levels", [1, 2, 3, 8])
def test_library_planner_matches_oracle(max_levels):
    rng = np.random.default_rng(720 + max_levels)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        bt, seq, nc = _random_tree(rng, n, BS)
        want = planner.plan_levels(bt, seq, nc, BS, max_levels)
        got, start, raw = _c_plan(bt, seq, nc, max_levels)
        assert (got, start) == (want[0], want[1])
        # token ranges: the segment's requests' query rows
        q = (seq - nc).astype(np.int64)
        cu = np.concatenate([[0], np.cumsum(q)])
        for s in raw:
            assert (s[5], s[6]) == (cu[s[1]], cu[s[2]])


@pytest.mark.parametrize("name", ["tree", "tree_chunked", "decode", "chunked"])
def test_library_planner_on_generated_batches(name):
    b = workloads.by_name(name)
    want = planner.plan_levels(b.block_table, b.seq_lens, b.num_computed_tokens, BS, 4)
    got, start, _ = _c_plan(b.block_table, b.seq_lens, b.num_computed_tokens, 4)
    assert (got, start) == (want[0], want[1])
    if name == "tree":
        assert max(s[0] for s in got) == 2     # three levels in the generated tree


def test_planner_errors():
    bt, seq = _hand_table()
    with pytest.raises(csp.CspError):
        csp.cascade_plan_levels(bt, seq, seq + 1)                    # computed > seq_len
    with pytest.raises(csp.CspError):
        csp.cascade_plan_levels(bt, seq, seq, max_levels=0)
    with pytest.raises(csp.CspError) as e:
        csp.cascade_plan_levels(bt, seq, seq - 1, max_levels=4, max_segments=2)
    assert e.value.status == csp.CSP_ERR_UNSUPPORTED
    segs, start = csp.cascade_plan_levels(np.zeros((0, 4), np.int32), [], [])
    assert segs.shape == (0, 7) and start.shape == (0,)


def _size_status(segs, n=6, total_q=6, max_k=128, max_suffix=64):
    lib = csp.load()
    a = np.ascontiguousarray(np.asarray(segs, np.int32).reshape(-1, 7))
    out = ctypes.c_size_t(0)
    return lib.csp_workspace_size_levels(n, total_q, 1, max_k,
                                         a.ctypes.data if a.size else None, a.shape[0],
                                         max_suffix, 8, 2, 64, ctypes.byref(out))


@pytest.mark.parametrize("segs", [
    [(0, 0, 6, 0, 32, 0, 6), (0, 3, 6, 32, 48, 3, 6)],     # two segments of one level share requests
    [(0, 0, 6, 0, 32, 0, 6), (1, 0, 3, 16, 64, 0, 3)],     # deeper keys start inside the parent's
    [(0, 0, 3, 0, 32, 0, 3), (1, 0, 6, 32, 64, 0, 6)],     # deeper segment holds more requests
    [(0, 0, 6, 0, 40, 0, 6)],                               # key end not a multiple of 16
    [(0, 0, 7, 0, 32, 0, 6)],                               # request past the batch
    [(0, 2, 2, 0, 32, 0, 0)],                               # no requests at all
    [(0, 0, 6, 0, 144, 0, 6)],                              # keys past the longest request
    [(8, 0, 6, 0, 32, 0, 6)],                               # level past the deepest allowed
    [(0, 0, 6, 0, 32, 0, 7)],                               # rows past total_q
])
def test_segment_list_checks(segs):
    assert _size_status(segs) == csp.CSP_ERR_INVALID_ARG


def test_segment_list_check_accepts_planned_segments_before_the_device_query():
    bt, seq = _hand_table()
    segs, _, raw = _c_plan(bt, seq, seq - 1, 4)
    st = _size_status(raw, n=6, total_q=6, max_k=int(seq.max()), max_suffix=32)
    # a valid list passes the host checks; without a GPU the device query then fails
    assert st in (csp.CSP_OK, csp.CSP_ERR_CUDA)
    assert _size_status(raw, n=6, total_q=6, max_k=int(seq.max()), max_suffix=-1) == \
        csp.CSP_ERR_INVALID_ARG
