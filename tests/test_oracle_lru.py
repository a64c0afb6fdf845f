"""Oracle pins: the expert-slot cache replacement policy (CPU).

Pins: a trace worked by hand from the policy statement (golden fixture) and
invariants that hold on any trace.
"""
import numpy as np

import workloads as W
from conftest import golden_rows
from oracle.lru import LayerLRU


def test_hand_worked_trace():
    c = LayerLRU(3)
    for row in golden_rows("lru_trace.txt"):
        step, ids, slots, misses = (part.strip() for part in row.split("|"))
        ids = [int(v) for v in ids.split()]
        got_slots, got_misses = c.access(int(step), ids)
        assert got_slots == [int(v) for v in slots.split()], row
        want = [tuple(int(q) for q in m.split(":")) for m in misses.split()]
        assert got_misses == want, row


def test_invariants_on_cache_stream():
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=300)
    sets = W.cache_stream_sets(cfg, 0, 300)
    c = LayerLRU(cfg.slots)
    hits = 0
    prev = set()
    for s, ids in enumerate(sets):
        before = dict(c.slot_of)
        slots, misses = c.access(s, ids)
        assert len(set(slots)) == len(ids)                     # distinct slots per token
        assert all(c.expert_of[sl] == e for e, sl in zip(ids, slots))
        missed = {e for e, _ in misses}
        assert missed == {e for e in ids if e not in before}   # a miss is exactly a non-resident expert
        for e, sl in misses:
            if sl in before.values():
                evicted = [x for x, q in before.items() if q == sl][0]
                assert evicted not in ids                        # never evicts the current token's experts
        if len(before) == cfg.slots:
            # once full, everything shared with the previous token is a hit (capacity 32 >= 2k)
            assert set(ids) & prev <= set(ids) - missed
        hits += len(ids) - len(misses)
        prev = set(ids)
    assert hits > 0.5 * 8 * 300


def test_resize_hand_worked():
    """Worked by hand from the resize reading: keep the newest experts (lower old slot on equal stamps), in old-slot
    order, with their stamps."""
    c = LayerLRU(3)
    c.access(0, [1, 2])    # 1 -> slot 0, 2 -> slot 1
    c.access(1, [3])       # 3 -> slot 2
    c.access(2, [1])       # hit: slot 0 stamp 2
    c.access(3, [4, 2])    # 2 hit (stamp 3); 4 evicts expert 3 (slot 2, stamp 1)
    assert c.expert_of == [1, 2, 4] and c.stamp == [2, 3, 3]
    assert c.resize(2) == [1, 2]            # stamps 3, 3 beat 2; kept in old-slot order
    assert c.expert_of == [2, 4] and c.stamp == [3, 3] and c.slot_of == {2: 0, 4: 1}
    assert c.resize(4) == [0, 1, -1, -1]    # growing keeps everything in place
    assert c.access(4, [7]) == ([2], [(7, 2)])   # the lowest free slot
    assert c.resize(1) == [2]               # expert 7 (stamp 4) is the newest
    assert c.expert_of == [7] and c.access(5, [7]) == ([0], [])


def test_resize_ties_go_to_the_lower_old_slot():
    c = LayerLRU(4)
    c.access(0, [10, 11, 12, 13])   # one step: all four stamps equal
    assert c.resize(2) == [0, 1] and c.expert_of == [10, 11]


def test_resize_keeps_the_policy_on_a_long_stream():
    """After any resize the survivors are exactly the most recently used residents, and the model keeps serving
    accesses with the usual invariants (every id resident after its access, at most `slots` residents)."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=240)
    sets = W.cache_stream_sets(cfg, 1, 240)
    c = LayerLRU(cfg.slots)
    sizes = {40: 12, 80: 32, 120: 8, 160: 64, 200: 16}
    for s, ids in enumerate(sets):
        if s in sizes:
            before = {c.expert_of[q]: c.stamp[q] for q in range(c.slots) if c.expert_of[q] >= 0}
            n = sizes[s]
            c.resize(n)
            after = {e for e in c.expert_of if e >= 0}
            assert len(after) == min(n, len(before))
            if after:
                assert min(before[e] for e in after) >= max((before[e] for e in before if e not in after), default=-1)
        got, _ = c.access(s, list(ids))
        assert all(c.expert_of[q] == e for q, e in zip(got, ids))
        assert len(c.slot_of) <= c.slots


def test_resize_keeps_survivors_in_old_slot_order():
    """Worked by hand: stamps [1, 2, 0] make slot 1 the newest and slot 0 the next; a resize to two slots keeps
    both and places them in their old order (slot 0's expert first), not newest first."""
    c = LayerLRU(3)
    c.access(0, [10, 11, 12])   # 10, 11, 12 -> slots 0, 1, 2, stamps 0
    c.access(1, [10])           # slot 0 stamp 1
    c.access(2, [11])           # slot 1 stamp 2
    assert c.stamp == [1, 2, 0]
    assert c.resize(2) == [0, 1]
    assert c.expert_of == [10, 11] and c.stamp == [1, 2]


def test_prefetch_hand_worked():
    """Worked by hand from the prefetch reading.  Two slots: the second prediction may not displace the first one
    (both stamped step - 1 = 0 like the residents), and a resident expert is left with its own stamp."""
    c = LayerLRU(2)
    c.access(0, [1, 2])                          # 1 -> slot 0, 2 -> slot 1, stamps 0
    assert c.prefetch(1, [7, 5, 5]) == [(5, 0), (7, 1)]   # ascending, repeats ignored
    assert c.expert_of == [5, 7] and c.stamp == [0, 0] and c.fetched == [True, True]
    assert c.prefetch(1, [5]) == [] and c.stamp == [0, 0]  # resident: no fill, no restamp
    assert c.access(1, [7]) == ([1], []) and c.prefetch_used == 1 and c.prefetched == 2
    assert c.fetched == [True, False]
    assert c.access(2, [5, 9]) == ([0, 1], [(9, 1)]) and c.prefetch_used == 2


def test_prefetch_keeps_the_current_steps_experts():
    """Worked by hand: slot 0 holds expert 3, used at step 1; a prefetch at step 1 takes slot 1 (stamp 0) and then
    finds no slot for the second prediction."""
    c = LayerLRU(2)
    c.access(0, [1, 2])
    c.access(1, [3])                             # evicts expert 1 (slot 0); 3 stamped 1
    assert c.prefetch(1, [4, 5]) == [(4, 1)]     # 5 finds no slot older than step 1 that this call did not fill
    assert c.expert_of == [3, 4] and c.stamp == [1, 0]
    assert c.prefetch(2, [6]) == [(6, 1)]        # at step 2 both are older; stamp 0 < 1 picks slot 1


def test_perfect_prediction_leaves_no_miss_on_the_stream():
    """With the next token's experts predicted exactly, every access after the first is a hit: the k current experts
    stay (stamp == step) and the other slots - at least k of them - take the new ones (slots >= 2k)."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=200)
    sets = W.cache_stream_sets(cfg, 2, 200)
    assert cfg.slots >= 2 * cfg.k
    c = LayerLRU(cfg.slots)
    for s, ids in enumerate(sets):
        _, misses = c.access(s, list(ids))
        assert s == 0 or misses == []
        if s + 1 < len(sets):
            before = {c.expert_of[q] for q in range(c.slots)}
            fills = c.prefetch(s, list(sets[s + 1]))
            assert {e for e, _ in fills} == set(sets[s + 1]) - before
            assert all(c.expert_of[q] in ids for q in range(c.slots) if c.stamp[q] == s)
            assert set(ids) <= set(c.slot_of)
    assert 0 < c.prefetch_used == c.prefetched   # every exact prediction is used by the next token


def test_prefetch_keeps_a_predicted_resident():
    """Worked by hand: expert 1 (slot 0, stamp 0) is predicted again with expert 9; 9 must take slot 1 (stamp 0,
    tie broken to the lower slot would otherwise pick slot 0)."""
    c = LayerLRU(3)
    c.access(0, [1, 2])
    c.access(1, [3])                             # 3 -> slot 2, stamp 1
    assert c.prefetch(1, [1, 9]) == [(9, 1)]     # slot 0 holds a predicted expert, slot 2 is this step's
    assert c.expert_of == [1, 9, 3] and c.stamp == [0, 0, 1] and c.fetched == [False, True, False]
