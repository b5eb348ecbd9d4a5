"""Oracle pins (CPU only): the oracle against library routines, closed forms and
invariants, and planted-fault builds of the oracle that the pins must catch."""

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin_passes_on_oracle(pin):
    fails = pin(mutant=0)
    assert not fails, fails


# Planted faults: scale dropped, causal off by one, GQA groups interleaved, base-2 LSE,
# slot off by one inside a page, feature index shifted, merge exponent sign flipped.
@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_planted_fault_is_caught(mutant):
    assert oracle._load(mutant).oracle_mutant_id() == mutant
    caught = [p.__name__ for p in pins.ALL_PINS if p(mutant=mutant)]
    assert caught, f"planted fault {mutant} passed every pin"


def test_real_oracle_build_has_no_planted_fault():
    assert oracle._load(0).oracle_mutant_id() == 0


def test_bad_block_id_is_an_error():
    paged, _ = pins.dense_problem(41, [8], [1], Hq=2, Hkv=1, D=8, bs=4)
    bt = paged["block_table"].copy()
    bt[0, 0] = paged["k_cache"].shape[0] + 5
    with pytest.raises(ValueError):
        oracle.attention(paged["q"], paged["k_cache"], paged["v_cache"], bt,
                         paged["cu_seqlens_q"], paged["seq_lens"], paged["scale"])


def test_sampled_rows_equal_full_run():
    paged, _ = pins.dense_problem(42, [30, 17], [4, 3], Hq=4, Hkv=2, D=16, bs=4,
                                  shared_tokens=8)
    o, l = oracle.attention(paged["q"], paged["k_cache"], paged["v_cache"],
                            paged["block_table"], paged["cu_seqlens_q"], paged["seq_lens"],
                            paged["scale"])
    rows = np.array([[0, 0], [3, 2], [6, 3], [4, 1]], np.int32)
    so, sl = oracle.attention(paged["q"], paged["k_cache"], paged["v_cache"],
                              paged["block_table"], paged["cu_seqlens_q"], paged["seq_lens"],
                              paged["scale"], rows=rows)
    for n, (t, h) in enumerate(rows):
        assert np.array_equal(so[n], o[t, h])
        assert sl[n] == l[t, h]
