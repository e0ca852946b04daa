"""Pins of the oracle's cross-step residency rule (delta prefetch): hand-derived
cases, a hand-derived three-step sequence, structural invariants over long
random step sequences, and closed-form special cases.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLD, "resident_cases.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("i", range(3))
def test_assign_hand_cases(i):
    c = _cases()["assign_cases"][i]
    new, fetched, slot_of = orc.resident_assign(c["slots"], c["need"], c["keep"])
    assert new == c["new_slots"]
    assert [list(f) for f in fetched] == c["fetched"]
    assert slot_of == c["slot_of"]


def test_step_sequence_hand():
    seq = _cases()["step_sequence"]
    slots = [-1] * seq["cap"]
    for st in seq["steps"]:
        slots, urgent, sot, pref = orc.resident_step(slots, st["T"], st["P_cur"], st["P_next"])
        assert [list(f) for f in urgent] == st["urgent"]
        assert sot == st["slot_of_true"]
        assert [list(f) for f in pref] == st["pref"]
        assert slots == st["slots"]


def _sorted_sample(rng, n, k):
    return sorted(rng.choice(n, size=k, replace=False).tolist())


def _check_assign(before, need, keep, after, fetched, slot_of):
    cap = len(before)
    protect = set(need) | set(keep or [])
    held = [b for b in after if b >= 0]
    assert len(held) == len(set(held)), "a block sits in two slots"
    for x, s in zip(need, slot_of):                 # everything needed is resident where reported
        assert after[s] == x
    for s in range(cap):                            # protected residents never move or leave
        if before[s] >= 0 and before[s] in protect:
            assert after[s] == before[s]
    changed = [s for s in range(cap) if after[s] != before[s]]
    assert sorted(changed) == sorted(s for _, s in fetched)
    for s in changed:                               # only empty or unprotected slots are reused
        assert before[s] < 0 or before[s] not in protect
    missing = sorted(set(need) - set(b for b in before if b >= 0))
    assert [x for x, _ in fetched] == missing       # exactly the delta, ascending
    # minimality: the reused slots are the lowest reusable ones, taken in order
    reusable = [s for s in range(cap) if before[s] < 0 or before[s] not in protect]
    assert [s for _, s in fetched] == reusable[:len(fetched)]


@pytest.mark.parametrize("seed,k,n", [(0, 4, 20), (1, 16, 60), (2, 32, 40), (3, 8, 1000)])
def test_random_sequences_keep_the_invariants(seed, k, n):
    rng = np.random.default_rng(seed)
    slots = [-1] * (2 * k)
    P_cur = None
    total = 0
    for step in range(60):
        T = _sorted_sample(rng, n, k)
        P_next = _sorted_sample(rng, n, k) if step % 7 != 6 else None
        before = list(slots)
        s1, urgent, sot, _ = orc.resident_step(before, T, P_cur, None)
        _check_assign(before, T, P_cur, s1, urgent, sot)
        slots, urgent2, sot2, pref = orc.resident_step(before, T, P_cur, P_next)
        assert urgent2 == urgent and sot2 == sot
        if P_next is not None:
            a2, f2, _ = orc.resident_assign(s1, P_next, T)
            _check_assign(s1, P_next, T, a2, f2, [a2.index(x) for x in P_next])
            assert slots == a2 and pref == f2
        total += len(urgent) + len(pref)
        P_cur = P_next
    assert total > 0


def test_static_selection_fetches_once():
    k = 8
    T = list(range(3, 3 + k))
    slots = [-1] * (2 * k)
    fetched = []
    for step in range(5):
        slots, urgent, sot, pref = orc.resident_step(slots, T, T if step else None, T)
        fetched.append(len(urgent) + len(pref))
    assert fetched == [k, 0, 0, 0, 0]


def test_disjoint_selections_fetch_everything():
    k = 6
    slots = [-1] * (2 * k)
    for step in range(6):
        T = list(range(step * k, (step + 1) * k))
        slots, urgent, sot, pref = orc.resident_step(slots, T, None, None)
        assert len(urgent) == k and pref == []


def test_too_few_slots_raise():
    with pytest.raises(ValueError):
        orc.resident_assign([1, 2], [3, 4], [1])


def test_budget_admits_the_lowest_missing_ids_and_urgent_fills_the_rest():
    # hand case: 3 missing (5, 6, 8); budget 2 admits 5 and 6 only
    new, fetched, slot_of = orc.resident_assign([3, 9, -1, 4, -1, -1], [4, 5, 6, 8], [9], budget=2)
    assert fetched == [(5, 0), (6, 2)] and slot_of == [3, 0, 2, -1]
    assert new == [5, 9, 6, 4, -1, -1]
    # a capped prefetch never changes what the urgent phase leaves resident for T
    rng = np.random.default_rng(7)
    k, n = 8, 40
    s_free = s_cap = [-1] * (2 * k)
    P = None
    for step in range(30):
        T = _sorted_sample(rng, n, k)
        P_next = _sorted_sample(rng, n, k)
        s_free, u1, sot1, p1 = orc.resident_step(s_free, T, P, P_next)
        s_cap, u2, sot2, p2 = orc.resident_step(s_cap, T, P, P_next, budget=2)
        assert len(p2) <= 2
        assert all(s_free[s] == x for x, s in zip(T, sot1))
        assert all(s_cap[s] == x for x, s in zip(T, sot2))
        P = P_next
