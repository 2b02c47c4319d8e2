"""Pins of the oracle's per-layer LRU slot pool (page-table update).

Independent references: a trace worked by hand from the stated rules, a
textbook LRU cache (collections.OrderedDict) for the one-expert-per-step case,
and invariants of any correct pool.
"""
import collections

import numpy as np
import pytest


def _counts(E, used):
    c = np.zeros(E, np.int32)
    for e in used:
        c[e] = 1
    return c


# Hand trace, E=6 experts, S=3 slots.  Each entry: experts used, then the
# expected (page table entries, misses (expert, destination), working-buffer
# flag, slot->expert afterwards, last_use afterwards).
HAND_TRACE = [
    # step 0: two misses fill the lowest empty slots in ascending expert id
    ([0, 2], {0: 0, 2: 1}, [(0, 0), (2, 1)], False, [0, 2, -1], [0, 0, -1]),
    # step 1: hit on 2 refreshes slot 1; miss 3 takes the last empty slot
    ([2, 3], {2: 1, 3: 2}, [(3, 2)], False, [0, 2, 3], [0, 1, 1]),
    # step 2: no empty slot; least recently used is slot 0 (expert 0, step 0)
    ([4], {4: 0}, [(4, 0)], False, [4, 2, 3], [2, 1, 1]),
    # step 3: misses 0 then 5; slots 1 and 2 tie at last_use 1 -> lower index first
    ([0, 5], {0: 1, 5: 2}, [(0, 1), (5, 2)], False, [4, 0, 5], [2, 3, 3]),
    # step 4: 4 experts > 3 slots -> working buffer; resident 4 read in place,
    # non-resident 1, 2, 3 get working-buffer entries S+0, S+1, S+2; state untouched
    ([1, 2, 3, 4], {4: 0, 1: 3, 2: 4, 3: 5}, [(1, 3), (2, 4), (3, 5)], True, [4, 0, 5], [2, 3, 3]),
    # step 5: hit 4 (slot 0 -> 5); miss 1: slots 1 and 2 tie at 3 -> slot 1
    ([1, 4], {1: 1, 4: 0}, [(1, 1)], False, [4, 1, 5], [5, 5, 3]),
    # step 6: nothing routed
    ([], {}, [], False, [4, 1, 5], [5, 5, 3]),
    # step 7: hit 1; miss 0 -> slot 2 (last_use 3); miss 2 -> slot 0 (last_use 5)
    ([0, 1, 2], {0: 2, 1: 1, 2: 0}, [(0, 2), (2, 0)], False, [2, 1, 0], [7, 7, 7]),
]


def test_lru_hand_trace(orc):
    E, S = 6, 3
    lru = orc.LRU(E, S)
    for step, (used, table, misses, wb, slots, last) in enumerate(HAND_TRACE):
        pt, me, md, got_wb = lru.step(_counts(E, used))
        exp_pt = np.full(E, -1, np.int32)
        for e, d in table.items():
            exp_pt[e] = d
        assert np.array_equal(pt, exp_pt), step
        assert list(zip(me.tolist(), md.tolist())) == misses, step
        assert got_wb == wb, step
        se, lu, st = lru.state()
        assert se.tolist() == slots and lu.tolist() == last and st == step + 1, step


def test_lru_one_expert_per_step_is_textbook_lru(orc):
    # with one expert per step the pool is a plain LRU cache of capacity S
    E, S = 20, 5
    g = np.random.default_rng(11)
    seq = g.zipf(1.3, 2000) % E
    lru = orc.LRU(E, S)
    cache = collections.OrderedDict()
    for e in seq:
        pt, me, md, wb = lru.step(_counts(E, [int(e)]))
        hit_ref = e in cache
        if hit_ref:
            cache.move_to_end(e)
        else:
            if len(cache) == S:
                cache.popitem(last=False)
            cache[e] = True
        assert (len(me) == 0) == hit_ref
        se, _, _ = lru.state()
        assert sorted(x for x in se.tolist() if x >= 0) == sorted(cache.keys())


@pytest.mark.parametrize("E,S,maxk", [(256, 32, 12), (64, 64, 20), (16, 4, 6)])
def test_lru_invariants_random(orc, E, S, maxk):
    g = np.random.default_rng(E + S)
    lru = orc.LRU(E, S)
    ever = set()
    for step in range(300):
        used = g.choice(E, size=int(g.integers(0, maxk + 1)), replace=False)
        prev_se, _, _ = lru.state()
        pt, me, md, wb = lru.step(_counts(E, used))
        se, lu, _ = lru.state()
        res = [x for x in se.tolist() if x >= 0]
        assert len(res) == len(set(res)) <= S
        assert wb == (len(used) > S)
        for e in range(E):
            if e in used:
                assert pt[e] >= 0
                if pt[e] < S:
                    assert se[pt[e]] == e
                else:
                    assert wb and e not in res
            else:
                assert pt[e] == -1
        if wb:
            assert np.array_equal(se, prev_se)
            assert sorted(md.tolist()) == list(range(S, S + len(me)))
        else:
            assert set(used.tolist()) <= set(res)
            # misses are exactly the used experts that were not resident before
            assert set(me.tolist()) == set(used.tolist()) - set(prev_se.tolist())
        if S >= E:
            assert set(me.tolist()) == set(used.tolist()) - ever
        ever |= set(used.tolist())


def test_lru_all_resident_gives_identity(orc):
    # the tiny layer: slots = experts and every expert used at the first step
    E = 8
    lru = orc.LRU(E, E)
    pt, me, md, wb = lru.step(np.ones(E, np.int32))
    assert np.array_equal(pt, np.arange(E)) and not wb
    pt, me, md, wb = lru.step(np.ones(E, np.int32))
    assert np.array_equal(pt, np.arange(E)) and len(me) == 0


def test_lru_invalidate_hand(orc):
    # invalidation empties the slot; the next miss takes the lowest empty slot
    E, S = 6, 3
    lru = orc.LRU(E, S)
    lru.step(_counts(E, [0, 1, 2]))            # slots: 0 1 2
    lru.invalidate(1)
    se, lu, _ = lru.state()
    assert se.tolist() == [0, -1, 2] and lu.tolist() == [0, -1, 0]
    pt, me, md, wb = lru.step(_counts(E, [5]))
    assert list(zip(me.tolist(), md.tolist())) == [(5, 1)]
    lru.invalidate(4)                           # not resident: no change
    assert lru.state()[0].tolist() == [0, 5, 2]
