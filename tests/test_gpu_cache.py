"""GPU tests of the expert-slot cache: fills, the cached decode stream, and fill failures.

The decode stream uses the cache workload's routing (E = 128, k = 8, 32 slots,
60 % of each token's experts shared with the previous token) on a reduced
expert shape so that the pinned host pool stays small.  Every layer output
read through the cache slots must equal, bit for bit, the output of the same
kernel on the resident weights (same bytes, same arithmetic, only the weight
index differs), and the first step is checked against the oracle as well.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import assert_layer_close, oracle_expert
from oracle.lru import LayerLRU

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import (CachedDecodeLayer, ExpertSlotPool, FusedDecodeLayer,
                                                     LayerWeights)

CFG = W.scaled(W.CONFIGS["cache_stream"], H=512, I=256, layers=2, steps=24)


def resident_weights(cfg, layer):
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_DECODE_TILES)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
    return lw


@pytest.fixture(scope="module")
def pool_and_resident():
    cfg = CFG
    pool = ExpertSlotPool(cfg.layers, cfg.E, cfg.H, cfg.I, cfg.slots, DEV)
    resident = []
    for l in range(cfg.layers):
        lw = resident_weights(cfg, l)
        pool.load_layer(l, lw)
        resident.append(lw)
    torch.cuda.synchronize()
    return pool, resident


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
    cfg = CFG
    layers = [CachedDecodeLayer(pool, l, cfg.k, cfg.T) for l in range(cfg.layers)]
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
            ref_mods[l](resident[l], logits, x, ref)
            torch.cuda.synchronize()
            assert Q.ft_device_status() == 0
            ids = sorted(W.cache_stream_sets(cfg, l, step + 1)[step])
            _, want_misses = oracles[l].access(step, ids)
            assert misses == [tuple(m) for m in want_misses], (step, l)
            want_miss_total += len(want_misses)
            assert torch.equal(out, ref), (step, l)
            if step == 0:
                r = O.moe_layer(logits_np, x_np, cfg.k, lambda e: oracle_expert(cfg, l, e), O.MODE_A16)
                assert_layer_close(out.float().cpu().numpy(), r["out"], f"cached layer {l}")
    hits, miss, filled = pool.cache.stats()
    assert miss == want_miss_total
    assert filled == miss * pool.expert_bytes
    assert hits > miss   # 60 % sharing between consecutive tokens


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
        pool.load_layer(l, resident[l])
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
            ref_mods[l](resident[l], logits, x, ref)
            torch.cuda.synchronize()
            assert Q.ft_device_status() == 0
            ids = sorted(W.cache_stream_sets(cfg, l, step + 1)[step])
            _, want_misses = oracles[l].access(step, ids)
            assert misses == [tuple(m) for m in want_misses], (step, l)
            assert torch.equal(out, ref), (step, l)
        _, _, filled0 = pool.cache.stats()
    assert pool.S == 12
