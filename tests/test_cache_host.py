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
