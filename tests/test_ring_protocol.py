"""The single decode kernel's suffix ring, as a protocol, under random interleavings.

Host-logic test (no GPU).  The producer warp fills ring slot i % S with item i and the
consumer groups take items g, g + G, g + 2G, ...; a full barrier tells a group that an
item's copies have landed, an empty barrier tells the producer that a slot is free.  An
mbarrier's wait on a parity returns as soon as the barrier's current phase has the other
parity, so a waiter that is two phases behind sees a completion that is not its own.

The model keeps, per barrier, the number of completed phases; a wait for parity p passes
when (completed & 1) != p.  A copy lands some random time after it is issued.  A
consumer that passes its wait reads the slot: it must find its own item, landed.

The kept scheme gives every (group, slot) pair its own full and empty barrier, an item
i's barrier being (i % G) * S + i % S and its parity (i / lcm(G, S)) & 1.  The scheme it
replaced had one barrier per slot and parity (i / S) & 1; with G = 2 and S = 3 a group
could take the other group's phase for its own, and the model finds that.
"""

from __future__ import annotations

import math
import random

import pytest


class Barrier:
    def __init__(self, count: int):
        self.count = count
        self.pending = count
        self.completed = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passes(self, parity: int) -> bool:
        return (self.completed & 1) != parity


def per_group_scheme(groups: int, slots: int):
    period = groups * slots // math.gcd(groups, slots)
    n = groups * slots
    return n, (lambda i: (i % groups) * slots + i % slots), (lambda i: (i // period) & 1)


def per_slot_scheme(groups: int, slots: int):
    return slots, (lambda i: i % slots), (lambda i: (i // slots) & 1)


def simulate(scheme, groups: int, slots: int, items: int, rng: random.Random):
    """Runs one random interleaving; returns 'ok', or what went wrong."""
    n_bar, bar_of, parity_of = scheme(groups, slots)
    full = [Barrier(1) for _ in range(n_bar)]
    empty = [Barrier(1) for _ in range(n_bar)]  # one arrival per group, as in the kernel
    slot_item = [None] * slots    # which item a slot holds
    slot_landed = [False] * slots
    in_flight = []                # issued copies: (slot, item)
    produced = 0
    nxt = list(range(groups))     # the next item of each group
    consumed = 0
    steps = 0
    while consumed < items:
        steps += 1
        if steps > 200 * items:
            return "stuck"
        actors = []
        if produced < items:
            i = produced
            if i < slots or empty[bar_of(i - slots)].passes(parity_of(i - slots)):
                actors.append("produce")
        if in_flight:
            actors.append("land")
        for g in range(groups):
            i = nxt[g]
            if i < items and full[bar_of(i)].passes(parity_of(i)):
                actors.append(("consume", g))
        if not actors:
            return "deadlock"
        a = rng.choice(actors)
        if a == "produce":
            i = produced
            s = i % slots
            slot_item[s], slot_landed[s] = i, False
            in_flight.append((s, i))
            produced += 1
        elif a == "land":
            # copies may land out of order
            k = rng.randrange(len(in_flight))
            s, i = in_flight.pop(k)
            slot_landed[s] = True
            full[bar_of(i)].arrive()
        else:
            g = a[1]
            i = nxt[g]
            s = i % slots
            if slot_item[s] != i or not slot_landed[s]:
                return f"group {g} took item {i} while its slot held item {slot_item[s]}" \
                       f" (landed {slot_landed[s]})"
            empty[bar_of(i)].arrive()
            nxt[g] += groups
            consumed += 1
    return "ok"


@pytest.mark.parametrize("groups", [1, 2])
@pytest.mark.parametrize("slots", [2, 3, 4, 5, 6])
def test_per_group_barriers_never_skip_a_phase(groups, slots):
    rng = random.Random(1000 * groups + slots)
    for _ in range(300):
        assert simulate(per_group_scheme, groups, slots, 60, rng) == "ok"


def test_per_slot_barriers_fail_with_two_groups_over_three_slots():
    """The replaced scheme: some interleaving lets a group read a slot that is not its."""
    rng = random.Random(7)
    outcomes = {simulate(per_slot_scheme, 2, 3, 60, rng) for _ in range(300)}
    assert any(o.startswith("group") for o in outcomes), outcomes


@pytest.mark.parametrize("slots", [2, 4, 6])
def test_per_slot_barriers_hold_when_each_group_owns_its_slots(slots):
    """With an even slot count each slot only ever serves one group: no skipped phase."""
    rng = random.Random(slots)
    for _ in range(300):
        assert simulate(per_slot_scheme, 2, slots, 60, rng) == "ok"
