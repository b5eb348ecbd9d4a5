"""Multi-level cascade planner oracle ("vLLM Cascade Attention：用法、场景与原理解析"
§七: any number of levels; §八 Step 1-2 within each segment), pinned by a hand-worked
example, by its reduction to the two-level planner, and by invariants that any correct
plan satisfies, checked by brute force on random prefix trees."""

import numpy as np
import pytest

from oracle import planner

BS = 16


def _hand_table():
    """6 requests, block size 16.  Blocks 1, 2 (keys 0-32) are shared by all; blocks
    3, 4 (keys 32-64) by requests 0-2; block 5 (keys 64-80) by requests 0-1; block 6
    (keys 32-48) by requests 3-5; every other block is a request's own."""
    rows = [[1, 2, 3, 4, 5, 10, 11],
            [1, 2, 3, 4, 5, 12, 13],
            [1, 2, 3, 4, 20, 21, 22],
            [1, 2, 6, 30, 31, 32, 33],
            [1, 2, 6, 40, 41, 42, 43],
            [1, 2, 6, 50, 51, 52, 53]]
    seq = [7 * BS - 3] * 6
    return np.array(rows, np.int32), np.array(seq, np.int32)


def test_hand_worked_tree():
    bt, seq = _hand_table()
    nc = seq - 1
    segs, start = planner.plan_levels(bt, seq, nc, BS, max_levels=4)
    # level 0: keys 0-32 for all; level 1: requests 0-2 over keys 32-64 and requests 3-5
    # over keys 32-48; level 2: requests 0-1 over keys 64-80 (request 2 leaves at block 4)
    assert segs == [(0, 0, 6, 0, 32), (1, 0, 3, 32, 64), (2, 0, 2, 64, 80),
                    (1, 3, 6, 32, 48)]
    assert start == [80, 80, 64, 48, 48, 48]
    # depth limit: two levels keep level 0 and level 1 only
    segs2, start2 = planner.plan_levels(bt, seq, nc, BS, max_levels=2)
    assert segs2 == [(0, 0, 6, 0, 32), (1, 0, 3, 32, 64), (1, 3, 6, 32, 48)]
    assert start2 == [64, 64, 64, 48, 48, 48]


def test_hand_worked_tree_with_the_computed_cap():
    bt, seq = _hand_table()
    nc = seq - 1
    nc[4] = 40      # request 4 has computed only 40 tokens: its group's keys 32-48 are
    nc[1] = 70      # not all computed (cap 40, floor 32: no segment); request 1: 70 ->
    segs, start = planner.plan_levels(bt, seq, nc, BS, max_levels=4)
    # the level-2 segment of requests 0-1 is capped to 70 and floored to 64: gone
    assert segs == [(0, 0, 6, 0, 32), (1, 0, 3, 32, 64)]
    assert start == [64, 64, 64, 32, 32, 32]


def _random_tree(rng, n, bs):
    """A block table over a random prefix tree of consecutive requests."""
    rows = [[] for _ in range(n)]
    next_id = [100]

    def fresh():
        next_id[0] += 1
        return next_id[0]

    def grow(lo, hi, depth):
        if depth > 3 or hi - lo < 1:
            return
        cuts = sorted(set(rng.integers(lo + 1, hi, size=int(rng.integers(0, 3))).tolist())) \
            if hi - lo > 1 else []
        bounds = [lo] + cuts + [hi]
        for a, b in zip(bounds[:-1], bounds[1:]):
            k = int(rng.integers(0, 4))
            ids = [fresh() for _ in range(k)]
            for r in range(a, b):
                rows[r].extend(ids)
            grow(a, b, depth + 1)

    grow(0, n, 0)
    for r in range(n):
        rows[r].extend(fresh() for _ in range(int(rng.integers(1, 4))))
    width = max(len(x) for x in rows) + 2
    table = np.zeros((n, width), np.int32)
    for r in range(n):
        table[r, :len(rows[r])] = rows[r]
        table[r, len(rows[r]):] = 7   # padding past the used entries
    seq = np.array([len(x) * bs - int(rng.integers(0, bs)) for x in rows], np.int32)
    nc = np.array([int(rng.integers(max(0, s - 3 * bs), s + 1)) for s in seq], np.int32)
    return table, seq, nc


def _check_invariants(bt, seq, nc, bs, max_levels, segs, start):
    n = len(seq)
    used = [-(-int(s) // bs) for s in seq]
    for (lev, lo, hi, klo, khi) in segs:
        assert 0 <= lev < max_levels and hi - lo >= 2 and klo < khi
        assert klo % bs == 0 and khi % bs == 0
        assert khi <= min(int(nc[r]) for r in range(lo, hi))         # §八 Step 2 cap
        for col in range(klo // bs, khi // bs):                      # §八 Step 1 sharing
            assert all(col < used[r] for r in range(lo, hi))
            assert len({int(bt[r, col]) for r in range(lo, hi)}) == 1
        # maximal: one more block is not shared by all, or not within the cap
        col = khi // bs
        ext = all(col < used[r] for r in range(lo, hi)) and \
            len({int(bt[r, col]) for r in range(lo, hi)}) == 1 and \
            khi + bs <= min(int(nc[r]) for r in range(lo, hi))
        assert not ext
    for r in range(n):
        mine = sorted((s for s in segs if s[1] <= r < s[2]), key=lambda s: s[0])
        assert len({s[0] for s in mine}) == len(mine)                # one per level
        k = 0
        for s in mine:                                               # keys 0.. in order
            assert s[3] == k
            k = s[4]
        assert start[r] == k


@pytest.mark.parametrize("max_levels", [1, 2, 3, 8])
def test_random_trees_invariants(max_levels):
    rng = np.random.default_rng(700 + max_levels)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        bt, seq, nc = _random_tree(rng, n, BS)
        segs, start = planner.plan_levels(bt, seq, nc, BS, max_levels)
        _check_invariants(bt, seq, nc, BS, max_levels, segs, start)


def test_one_level_is_the_two_level_planner():
    rng = np.random.default_rng(711)
    for _ in range(300):
        n = int(rng.integers(2, 12))
        bt, seq, nc = _random_tree(rng, n, BS)
        cpl, _ = planner.plan(bt, seq, nc, BS)
        segs, start = planner.plan_levels(bt, seq, nc, BS, max_levels=1)
        assert segs == ([(0, 0, n, 0, cpl)] if cpl > 0 else [])
        assert start == [cpl] * n


