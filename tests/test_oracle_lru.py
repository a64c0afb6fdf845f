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
