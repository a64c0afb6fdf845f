"""Host logic of the expert-slot cache through the C ABI (no device needed).

ft_expert_cache_lookup is pure host bookkeeping: it is checked against the
oracle's statement of the policy (oracle/lru.py) on the hand-worked trace and on
the cache decode stream's routing, for several layers at once.  The fill path's
host-side fault hook is checked here too: the injected failure returns before
any CUDA call.
"""
import pytest

import workloads as W
from conftest import golden_rows
from oracle.lru import LayerLRU

Q = pytest.importorskip("quantized_expert_ffn_06_b300")


def fake_cache(L, E, S, expert_bytes=4096):
    stride = (expert_bytes + 255) // 256 * 256
    # addresses are only stored, never dereferenced by lookup
    host = [0x10000000 + i * stride for i in range(L * E)]
    return Q.ExpertCacheHandle(L, E, S, expert_bytes, host, 0x40000000, stride, 0x80000000)


def test_hand_worked_trace_matches_oracle():
    c = fake_cache(1, 16, 3)
    o = LayerLRU(3)
    for row in golden_rows("lru_trace.txt"):
        step, ids, slots, misses = (part.strip() for part in row.split("|"))
        ids = [int(v) for v in ids.split()]
        got = c.lookup(0, int(step), ids)
        want = o.access(int(step), ids)
        assert got[0] == want[0] == [int(v) for v in slots.split()]
        assert got[1] == [tuple(m) for m in want[1]]


def test_cache_stream_trace_matches_oracle_on_three_layers():
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=200)
    L = 3
    c = fake_cache(L, cfg.E, cfg.slots)
    oracles = [LayerLRU(cfg.slots) for _ in range(L)]
    sets = [W.cache_stream_sets(cfg, l, 200) for l in range(L)]
    total_miss = 0
    for s in range(200):
        for l in range(L):  # layers interleave, as in a decode step
            got = c.lookup(l, s, list(sets[l][s]))
            want = oracles[l].access(s, list(sets[l][s]))
            assert got[0] == want[0] and got[1] == [tuple(m) for m in want[1]], (s, l)
            total_miss += len(want[1])
    hits, misses, filled = c.stats()
    assert misses == total_miss and hits + misses == 200 * L * cfg.k and filled == 0


@pytest.mark.parametrize("ids", [[1, 1], [-1], [16], [0, 1, 2, 3]])
def test_lookup_rejects_bad_token_sets(ids):
    c = fake_cache(1, 16, 3)
    with pytest.raises(Q.FtError) as ei:
        c.lookup(0, 0, ids)
    assert ei.value.status == Q.FT_ERR_INVALID_ARG


def test_create_rejects_bad_geometry():
    with pytest.raises(Q.FtError):
        fake_cache(1, 16, 17)        # more slots than experts
    with pytest.raises(Q.FtError):
        Q.ExpertCacheHandle(1, 4, 2, 1000, [0x1000] * 4, 0x40000000, 1000, 0x80000000)   # unaligned stride


def test_injected_fill_failure_is_reported_without_touching_the_device():
    c = fake_cache(2, 16, 4)
    c.inject_fill_failure(0)
    _, misses = c.lookup(1, 0, [3, 9])
    e, s = misses[0]
    with pytest.raises(Q.FtError) as ei:
        c.fill(1, e, s, stream=0)   # the legacy default stream handle; no torch device lookup
    assert ei.value.status == Q.FT_ERR_CUDA and "injected" in str(ei.value)


def test_resize_plan_matches_oracle_along_the_stream():
    """The library's resize plan (pure host) against the oracle's, at several points of the cache stream and for
    shrinking, equal and growing sizes, on three layers."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=120)
    L = 3
    c = fake_cache(L, cfg.E, cfg.slots)
    oracles = [LayerLRU(cfg.slots) for _ in range(L)]
    sets = [W.cache_stream_sets(cfg, l, 120) for l in range(L)]
    for s in range(120):
        for l in range(L):
            c.lookup(l, s, list(sets[l][s]))
            oracles[l].access(s, list(sets[l][s]))
        if s in (0, 3, 17, 60, 119):
            for n in (8, 9, 20, 32, 40, 128):
                want = []
                for o in oracles:
                    probe = LayerLRU(o.slots)
                    probe.expert_of, probe.stamp, probe.slot_of = list(o.expert_of), list(o.stamp), dict(o.slot_of)
                    want.append(probe.resize(n))
                assert c.resize_plan(n) == want, (s, n)


def test_resize_rejects_overlapping_pools_and_bad_sizes():
    c = fake_cache(2, 16, 4)          # pool at 0x40000000, 2 layers x 4 slots x 4096 B
    c.lookup(0, 0, [1, 2])
    for args in ((8, 0x40000000 + 4096, 4096),   # overlaps and is not a shrink in place
                 (8, 0x40000000, 4096),          # same base but growing
                 (0, 0x50000000, 4096),          # no slots
                 (17, 0x50000000, 4096),         # more slots than experts
                 (4, 0x50000000, 1000)):         # stride below expert_bytes / unaligned
        with pytest.raises(Q.FtError) as ei:
            c.resize(*args, stream=0)
        assert ei.value.status == Q.FT_ERR_INVALID_ARG, args
    assert c.S == 4 and c.lookup(0, 1, [1, 2])[1] == []   # nothing changed: both still resident


def test_injected_move_failure_empties_the_cache_with_the_new_geometry():
    """A move that cannot be enqueued (host-side hook, before any CUDA call) leaves an empty cache of the new size,
    so every access refills from host memory."""
    c = fake_cache(2, 16, 4)
    c.lookup(0, 0, [1, 2, 3])
    c.lookup(1, 0, [4])
    c.inject_fill_failure(0)
    with pytest.raises(Q.FtError) as ei:
        c.resize(2, 0x50000000, 4096, stream=0)   # a disjoint pool: every kept expert needs a move
    assert ei.value.status == Q.FT_ERR_CUDA and "injected" in str(ei.value)
    assert c.S == 2   # the handle is on the new pool
    c.inject_fill_failure(-1)
    assert c.lookup(0, 1, [2, 3]) == ([0, 1], [(2, 0), (3, 1)])
    assert c.lookup(1, 1, [4])[1] == [(4, 0)]
    with pytest.raises(Q.FtError):
        c.lookup(0, 2, [5, 6, 7])             # n > the new slot count


class _NeverReady:
    def __init__(self):
        self.queries = 0

    def query(self):
        self.queries += 1
        return False


class _ReadyAfter:
    def __init__(self, n):
        self.n = n

    def query(self):
        self.n -= 1
        return self.n < 0


def test_bounded_host_wait_gives_up_with_a_timeout_status():
    """The cached decode step waits for its routing result on the host; an event that never completes ends that
    wait with FT_ERR_TIMEOUT after the limit instead of blocking (a stand-in event, no GPU involved)."""
    import time

    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import wait_event
    ev = _NeverReady()
    t0 = time.monotonic()
    with pytest.raises(Q.FtError) as ei:
        wait_event(ev, 0.05, "routing result")
    assert ei.value.status == Q.FT_ERR_TIMEOUT
    assert 0.05 <= time.monotonic() - t0 < 1.0
    assert ev.queries > 1
    wait_event(_ReadyAfter(3), 1.0, "routing result")   # completes before the limit: returns


def test_prefetch_matches_oracle_along_the_stream():
    """Lookup + prefetch of a noisy predictor (the next token's experts, some replaced by random ids) through the
    library against the oracle, on two layers: the same fills, the same slots for every token, the same stats."""
    import numpy as np
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=150)
    L = 2
    c = fake_cache(L, cfg.E, cfg.slots)
    oracles = [LayerLRU(cfg.slots) for _ in range(L)]
    sets = [W.cache_stream_sets(cfg, 10 + l, 150) for l in range(L)]
    rng = np.random.default_rng(5)
    for s in range(150):
        for l in range(L):
            got = c.lookup(l, s, list(sets[l][s]))
            want = oracles[l].access(s, list(sets[l][s]))
            assert got[0] == want[0] and got[1] == [tuple(m) for m in want[1]], (s, l)
            if s + 1 < 150:
                pred = [int(e) for e in sets[l][s + 1]]
                pred = [e if rng.random() < 0.8 else int(rng.integers(cfg.E)) for e in pred] + [pred[0]]  # a repeat
                assert c.prefetch(l, s, pred) == [tuple(f) for f in oracles[l].prefetch(s, pred)], (s, l)
    assert c.prefetch_stats() == (sum(o.prefetched for o in oracles), sum(o.prefetch_used for o in oracles))
    assert c.prefetch_stats()[1] > 0


def test_prefetch_rejects_bad_ids():
    c = fake_cache(1, 16, 3)
    for ids in ([16], [-1]):
        with pytest.raises(Q.FtError) as ei:
            c.prefetch(0, 0, ids)
        assert ei.value.status == Q.FT_ERR_INVALID_ARG
    assert c.prefetch(0, 0, []) == []


def test_resize_plan_after_prefetches_matches_oracle():
    """Prefetched experts carry stamp step - 1, which decides who survives a resize: the library's plan against the
    oracle's along a stream with a prefetch after every token (the next token's experts plus one wrong guess)."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], steps=60)
    c = fake_cache(1, cfg.E, cfg.slots)
    o = LayerLRU(cfg.slots)
    sets = W.cache_stream_sets(cfg, 3, 61)
    for s in range(60):
        c.lookup(0, s, list(sets[s]))
        o.access(s, list(sets[s]))
        pred = [int(e) for e in sets[s + 1]] + [(s * 37) % cfg.E]
        assert c.prefetch(0, s, pred) == [tuple(f) for f in o.prefetch(s, pred)], s
        if s in (5, 30, 59):
            for n in (8, 16, 31, 64):
                probe = LayerLRU(o.slots)
                probe.expert_of, probe.stamp, probe.slot_of = list(o.expert_of), list(o.stamp), dict(o.slot_of)
                probe.fetched = list(o.fetched)
                assert c.resize_plan(n) == [probe.resize(n)], (s, n)
