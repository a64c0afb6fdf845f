"""GPU tests of the expert-slot cache: fills, the cached decode stream, and fill failures.

The decode stream uses the cache workload's routing (E = 128, k = 8, 32 slots, 60 % of each token's experts shared
with the previous token), once on a reduced expert shape (hidden 512, intermediate 256; also through three elastic
resizes) and once at the workload's own shape (hidden 4096, intermediate 1536).  Every layer output read through
the cache slots must equal, bit for bit, the output of the same kernel on the resident weights (same bytes, same
arithmetic, only the weight index differs), and outputs are checked against the oracle, which reads the device's
own canonical NVFP4 bytes.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import OracleExperts, assert_layer_close
from oracle.lru import LayerLRU

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import (CachedDecodeLayer, ExpertSlotPool, FusedDecodeLayer,
                                                     LayerWeights, MoEWeights)

CFG = W.scaled(W.CONFIGS["cache_stream"], H=512, I=256, layers=2, steps=24)


class Resident:
    """One layer's experts resident on the device: canonical row-layout NVFP4 bytes drawn and quantised there, the
    handle's decode-tile copy of them (w, what the pool is loaded from and the resident kernel reads), and the
    oracle's experts read from the canonical bytes."""

    def __init__(self, cfg, layer):
        canon = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_ROWS)
        canon.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
        self.canon = canon
        self.handle = MoEWeights(canon, Q.FT_WEIGHTS_DECODE_TILES)
        self.w = self.handle.view(Q.FT_LAYOUT_DECODE_TILES)
        self.oracle = OracleExperts(canon)


def make_pool(cfg):
    pool = ExpertSlotPool(cfg.layers, cfg.E, cfg.H, cfg.I, cfg.slots, DEV)
    resident = []
    for l in range(cfg.layers):
        r = Resident(cfg, l)
        pool.load_layer(l, r.w)
        resident.append(r)
    torch.cuda.synchronize()
    return pool, resident


@pytest.fixture(scope="module")
def pool_and_resident():
    return make_pool(CFG)


def run_stream(cfg, pool, resident, oracle_steps, prefetch=0):
    """The cached decode stream over cfg.steps tokens and cfg.layers layers: misses (and, with prefetch = P, the
    prefetch fills of the router's next P ranks) as the oracle LRU predicts, outputs bit-equal to the resident
    weights, and equal to the oracle within the tolerance at oracle_steps."""
    layers = [CachedDecodeLayer(pool, l, cfg.k, cfg.T, prefetch=prefetch) for l in range(cfg.layers)]
    ref_mods = [FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV) for _ in range(cfg.layers)]
    oracles = [LayerLRU(cfg.slots) for _ in range(cfg.layers)]
    want_miss_total = 0
    stream = torch.cuda.current_stream()
    for step in range(cfg.steps):
        for l in range(cfg.layers):
            logits_np = W.router_logits(cfg, l, step)
            x_np = W.activations_bf16(cfg, l, step)
            logits = torch.from_numpy(logits_np).to(DEV)
            x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(DEV)
            out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
            misses = layers[l](logits, x, out, step, stream=stream)
            ref = torch.empty_like(out)
            ref_mods[l](resident[l].w, logits, x, ref)
            torch.cuda.synchronize()
            assert Q.ft_device_status() == 0
            ids = sorted(W.cache_stream_sets(cfg, l, step + 1)[step])
            _, want_misses = oracles[l].access(step, ids)
            assert misses == [tuple(m) for m in want_misses], (step, l)
            want_miss_total += len(want_misses)
            if prefetch:
                ranked = [int(e) for e in O.route(logits_np, cfg.k + prefetch)[0][0]]
                assert sorted(ranked[:cfg.k]) == ids
                want_fills = oracles[l].prefetch(step, sorted(set(ranked[cfg.k:]) - set(ids)))
                assert layers[l].prefetched == [tuple(f) for f in want_fills], (step, l)
            assert torch.equal(out, ref), (step, l)
            if step in oracle_steps:
                r = O.moe_layer(logits_np, x_np, cfg.k, resident[l].oracle, O.MODE_A16)
                assert_layer_close(out.float().cpu().numpy(), r["out"], f"cached layer {l} step {step}")
    return want_miss_total, oracles


def test_fill_copies_the_host_block_into_the_slot(pool_and_resident):
    pool, _ = pool_and_resident
    c = Q.ExpertCacheHandle(pool.L, pool.E, pool.S, pool.expert_bytes,
                            [pool.host.data_ptr() + i * pool.slot_stride for i in range(pool.L * pool.E)],
                            pool.slots.data_ptr(), pool.slot_stride, pool.tables.data_ptr())
    _, misses = c.lookup(1, 0, [5, 77])
    s = torch.cuda.Stream()
    for e, slot in misses:
        c.fill(1, e, slot, stream=s)
    c.publish(1, stream=s)
    s.synchronize()
    for e, slot in misses:
        off = (1 * pool.S + slot) * pool.slot_stride
        assert torch.equal(pool.slots[off:off + pool.expert_bytes].cpu(), pool.host_expert(1, e))
    table = pool.tables[1].cpu().numpy()
    assert table[5] == dict(misses)[5] and table[77] == dict(misses)[77] and (table >= 0).sum() == 2
    c.close()
    pool.tables.fill_(-1)


def test_cached_decode_stream_equals_resident_weights(pool_and_resident):
    pool, resident = pool_and_resident
    want_miss_total, _ = run_stream(CFG, pool, resident, oracle_steps=(0, 11, 23))
    hits, miss, filled = pool.cache.stats()
    assert miss == want_miss_total
    assert filled == miss * pool.expert_bytes
    assert hits > miss   # 60 % sharing between consecutive tokens


def test_cached_decode_stream_at_the_workload_shape():
    """Hidden 4096, intermediate 1536, 128 experts, top-8, 32 VRAM slots per layer, experts from a pinned host
    pool (two layers, 16 tokens): misses as the oracle LRU predicts, every output bit-equal to the resident
    weights, and against the oracle on the first, a middle and the last token."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], layers=2, steps=16)
    assert (cfg.H, cfg.I, cfg.E, cfg.k, cfg.slots) == (4096, 1536, 128, 8, 32)
    pool, resident = make_pool(cfg)
    want_miss_total, _ = run_stream(cfg, pool, resident, oracle_steps=(0, 7, 15))
    hits, miss, filled = pool.cache.stats()
    assert miss == want_miss_total and filled == miss * pool.expert_bytes
    assert hits > miss


def test_cached_decode_stream_with_router_driven_prefetch():
    """Prefetch of the router's next 4 ranks after each token: the prefetch fills (copied on the copy stream behind
    the token's misses while later layers compute) and the demand misses follow the oracle LRU with its prefetch
    reading, the outputs stay bit-equal to the resident weights, and the library's prefetch counters equal the
    oracle's."""
    cfg = CFG
    pool, resident = make_pool(cfg)
    want_miss_total, oracles = run_stream(cfg, pool, resident, oracle_steps=(0, 23), prefetch=4)
    hits, miss, filled = pool.cache.stats()
    prefetched, used = pool.cache.prefetch_stats()
    assert miss == want_miss_total
    assert prefetched == sum(o.prefetched for o in oracles) > 0
    assert used == sum(o.prefetch_used for o in oracles)
    assert filled == (miss + prefetched) * pool.expert_bytes


def test_injected_fill_failure_leaves_the_device_usable(pool_and_resident):
    pool, _ = pool_and_resident
    c = Q.ExpertCacheHandle(pool.L, pool.E, pool.S, pool.expert_bytes,
                            [pool.host.data_ptr() + i * pool.slot_stride for i in range(pool.L * pool.E)],
                            pool.slots.data_ptr(), pool.slot_stride, pool.tables.data_ptr())
    c.inject_fill_failure(1)
    _, misses = c.lookup(0, 0, [1, 2, 3])
    s = torch.cuda.Stream()
    c.fill(0, *misses[0], stream=s)
    with pytest.raises(Q.FtError) as ei:
        c.fill(0, *misses[1], stream=s)
    assert ei.value.status == Q.FT_ERR_CUDA
    c.inject_fill_failure(-1)
    c.fill(0, *misses[1], stream=s)
    s.synchronize()
    assert Q.ft_device_status() == 0
    c.close()


def test_elastic_resize_keeps_the_cached_stream_exact(pool_and_resident):
    """The cached decode stream with three resizes at safe points: a shrink into a new pool, a growth into a new
    pool, and a shrink compacted in place.  At each resize the plan equals the oracle's, every kept slot holds its
    expert's bytes (moved device to device, not reloaded), the published tables map exactly the kept experts, and
    the stream goes on with misses as the oracle predicts and outputs bit-equal to the resident weights."""
    _, resident = pool_and_resident
    cfg = CFG
    pool = ExpertSlotPool(cfg.layers, cfg.E, cfg.H, cfg.I, cfg.slots, DEV)
    for l in range(cfg.layers):
        pool.load_layer(l, resident[l].w)
    layers = [CachedDecodeLayer(pool, l, cfg.k, cfg.T) for l in range(cfg.layers)]
    ref_mods = [FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV) for _ in range(cfg.layers)]
    oracles = [LayerLRU(cfg.slots) for _ in range(cfg.layers)]
    resizes = {6: (16, False), 12: (40, False), 18: (12, True)}
    stream = torch.cuda.current_stream()
    _, _, filled0 = pool.cache.stats()
    for step in range(cfg.steps):
        if step in resizes:
            n, in_place = resizes[step]
            torch.cuda.synchronize()   # safe point: fills and layer kernels are done
            plan = pool.cache.resize_plan(n)
            assert plan == [o.resize(n) for o in oracles], step
            pool.resize(n, in_place=in_place, stream=stream)
            torch.cuda.synchronize()
            _, _, filled = pool.cache.stats()
            assert filled == filled0   # no host bytes moved by a resize
            tables = pool.tables.cpu().numpy()
            for l, o in enumerate(oracles):
                want_table = np.full(cfg.E, -1, np.int32)
                for i, e in enumerate(o.expert_of):
                    if e < 0:
                        continue
                    want_table[e] = i
                    off = (l * n + i) * pool.slot_stride
                    assert torch.equal(pool.slots[off:off + pool.expert_bytes].cpu(), pool.host_expert(l, e)), (step, l, i)
                assert np.array_equal(tables[l], want_table), (step, l)
        for l in range(cfg.layers):
            logits_np = W.router_logits(cfg, l, step)
            x_np = W.activations_bf16(cfg, l, step)
            logits = torch.from_numpy(logits_np).to(DEV)
            x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(DEV)
            out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
            misses = layers[l](logits, x, out, step, stream=stream)
            ref = torch.empty_like(out)
            ref_mods[l](resident[l].w, logits, x, ref)
            torch.cuda.synchronize()
            assert Q.ft_device_status() == 0
            ids = sorted(W.cache_stream_sets(cfg, l, step + 1)[step])
            _, want_misses = oracles[l].access(step, ids)
            assert misses == [tuple(m) for m in want_misses], (step, l)
            assert torch.equal(out, ref), (step, l)
        _, _, filled0 = pool.cache.stats()
    assert pool.S == 12
