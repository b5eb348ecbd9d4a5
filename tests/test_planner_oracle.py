"""Planner oracle pins (CPU only): the worked example on the pages, a vectorised
restatement on random tables, invariants, padding, and planted faults."""

import json
import os

import numpy as np
import pytest

from oracle import planner

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def test_worked_example_from_the_pages():
    ex = _golden("planner_worked_example.json")
    ids = ex["block_ids"]
    table = [[ids[c] for c in row] for row in ex["block_table"]]
    bs = ex["block_size"]
    ncpb = planner.num_common_prefix_blocks(table, ex["seq_lens"], bs)
    assert ncpb == ex["expected"]["num_common_prefix_blocks"]
    cpl = planner.common_prefix_len(ncpb, bs, ex["num_computed_tokens"])
    assert cpl == ex["expected"]["common_prefix_len"]
    names = {v: k for k, v in ids.items()}
    assert [names[b] for b in table[0][:cpl]] == ex["expected"]["prefix_tokens"]
    for r, want in enumerate(ex["expected"]["suffix_tokens"]):
        assert [names[b] for b in table[r][cpl:ex["seq_lens"][r]]] == want
    for r, want in enumerate(ex["expected"]["query_tokens"]):
        nc = ex["num_computed_tokens"][r]
        assert [names[b] for b in table[r][nc:ex["seq_lens"][r]]] == want


def _vectorised_ncpb(table, seq_lens, bs):
    """Independent restatement: compare whole columns, first mismatch by argmin."""
    table = np.asarray(table)
    if len(seq_lens) == 0:
        return 0
    used = -(-np.asarray(seq_lens) // bs)
    limit = int(used.min())
    if limit == 0:
        return 0
    same = np.all(table[:, :limit] == table[0:1, :limit], axis=0)
    return limit if same.all() else int(np.argmin(same))


def _random_table(rng, n, bs):
    common = int(rng.integers(0, 6))
    seq = rng.integers(1, 10 * bs, size=n)
    width = int(-(-seq.max() // bs)) + 2
    table = rng.integers(0, 4, size=(n, width))    # small id range: accidental matches happen
    common = min(common, width)
    table[:, :common] = rng.integers(0, 50, size=common)[None, :]
    nc = np.array([int(rng.integers(0, s + 1)) for s in seq])
    return table, seq, nc


@pytest.mark.parametrize("bs", [1, 2, 16])
def test_random_tables_against_vectorised_statement(bs):
    rng = np.random.default_rng(bs)
    for _ in range(400):
        n = int(rng.integers(1, 7))
        table, seq, nc = _random_table(rng, n, bs)
        ncpb = planner.num_common_prefix_blocks(table.tolist(), seq.tolist(), bs)
        assert ncpb == _vectorised_ncpb(table, seq, bs)
        cpl = planner.common_prefix_len(ncpb, bs, nc.tolist())
        assert cpl % bs == 0
        assert cpl <= nc.min()
        assert cpl <= ncpb * bs
        assert cpl > min(ncpb * bs, nc.min()) - bs     # the floor drops less than one block


def test_padding_never_extends_the_run():
    bs = 4
    # both rows use 2 blocks, shared; the padding (same id in both rows) must not count
    table = [[7, 9, 3, 3, 3], [7, 9, 3, 3, 3]]
    assert planner.num_common_prefix_blocks(table, [8, 6], bs) == 2
    # a longer row cannot share more than the shortest row uses
    table = [[7, 9, 5, 1], [7, 9, 5, 1]]
    assert planner.num_common_prefix_blocks(table, [16, 5], bs) == 2


def test_empty_and_single_request():
    assert planner.num_common_prefix_blocks([], [], 16) == 0
    assert planner.common_prefix_len(0, 16, []) == 0
    # one request: its whole used run, capped to its computed tokens, floored
    assert planner.plan([[4, 5, 6, 0]], [40], [37], 16) == (32, False)
    assert planner.plan([[4, 5, 6, 0]], [40], [30], 16) == (16, False)


def test_thresholds_from_the_pages():
    assert planner.use_cascade_thresholds(256, 8)
    assert not planner.use_cascade_thresholds(255, 8)
    assert not planner.use_cascade_thresholds(256, 7)


# Planted planner faults: scanning one block past the shortest row (padding counted),
# no cap to the computed tokens, and no floor to whole blocks.
@pytest.mark.parametrize("fault", ["scan_padding", "no_cap", "no_floor"])
def test_planted_planner_faults_are_caught(fault, monkeypatch):
    if fault == "scan_padding":
        monkeypatch.setattr(planner, "_cdiv", lambda a, b: -(-a // b) + 1)
    elif fault == "no_cap":
        monkeypatch.setattr(planner, "common_prefix_len",
                            lambda k, bs, nc: (k * bs // bs) * bs)
    else:
        monkeypatch.setattr(planner, "common_prefix_len",
                            lambda k, bs, nc: min(k * bs, min(nc)) if len(nc) else 0)
    failed = False
    try:
        test_worked_example_from_the_pages()
        test_padding_never_extends_the_run()
        test_empty_and_single_request()
        for bs in (1, 2, 16):
            test_random_tables_against_vectorised_statement(bs)
    except AssertionError:
        failed = True
    assert failed, f"planted planner fault {fault} passed every pin"
