"""GPU parity of the prefill expert FFN on the block-scaled FP4 tensor cores.

The tensor-core path quantises the activations (x, and h after its bf16
rounding) to NVFP4 with unit tensor scale; the oracle's A4 mode states the same
arithmetic in fp64.  Routing and grouping are bit-exact; outputs within relative
L2 5e-3 and max |err| 2e-2 * RMS per layer output.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import OracleExperts, assert_layer_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights, MoEWeights, PrefillLayer


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


class DeviceLayer:
    """Canonical row-layout NVFP4 weights of one layer on the device (drawn and quantised there, or uploaded from the
    host generator and quantised there), the handle's tensor-core layout of them (w), and the oracle's experts read
    from the same canonical bytes."""

    def __init__(self, cfg, layer, generated=True):
        self.canon = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_ROWS)
        if generated:
            self.canon.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
        else:
            for e in range(cfg.E):
                self.canon.set_expert(e, *(to_dev(W.weights_fp32(cfg, layer, e, p)) for p in range(3)))
        self.handle = MoEWeights(self.canon, Q.FT_WEIGHTS_UMMA_TILES)
        self.w = self.handle.view(Q.FT_LAYOUT_UMMA_TILES)
        self.oracle = OracleExperts(self.canon)


def weights(cfg, layer, generated=True):
    return DeviceLayer(cfg, layer, generated)


def run(cfg, lw, logits, x_bits):
    T = logits.shape[0]
    mod = PrefillLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    w = lw.w if isinstance(lw, DeviceLayer) else lw
    mod(w, to_dev(logits), to_dev(x_bits.view(np.int16), torch.bfloat16), out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return mod, out


def check(cfg, dl, mod, out, logits, x_bits, rows=None):
    ref = O.moe_layer(logits, x_bits, cfg.k, dl.oracle, O.MODE_A4, rows=rows)
    assert np.array_equal(mod.ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(mod.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(mod.perm.cpu().numpy(), ref["perm"])
    assert np.array_equal(mod.inv.cpu().numpy(), ref["inv"])
    got = out.float().cpu().numpy()
    if rows is not None:
        got = got[rows]
    return assert_layer_close(got, ref["out"], f"prefill {cfg.name}")


def test_tiny_layer_every_output():
    cfg = W.CONFIGS["tiny"]
    lw = weights(cfg, 0, generated=False)
    logits, x_bits = W.router_logits(cfg, 0, 0), W.activations_bf16(cfg, 0, 0)
    mod, out = run(cfg, lw, logits, x_bits)
    check(cfg, lw, mod, out, logits, x_bits)


@pytest.mark.parametrize("T", [1, 13, 37, 200])
def test_ragged_token_counts(T):
    cfg = W.scaled(W.CONFIGS["tiny"], T=T)
    lw = weights(cfg, 0, generated=False)
    logits, x_bits = W.router_logits(cfg, 0, 1), W.activations_bf16(cfg, 0, 1)
    mod, out = run(cfg, lw, logits, x_bits)
    check(cfg, lw, mod, out, logits, x_bits)


def test_one_expert_spanning_several_tiles():
    """k = 1 and every token routed to expert 5: 300 rows = three 128-row tiles, the last one partial."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=300, k=1)
    lw = weights(cfg, 0, generated=False)
    logits = W.router_logits(cfg, 0, 2).copy()
    logits[:, 5] = 50.0
    x_bits = W.activations_bf16(cfg, 0, 2)
    mod, out = run(cfg, lw, logits, x_bits)
    assert (mod.ids.cpu().numpy() == 5).all()
    check(cfg, lw, mod, out, logits, x_bits)


@pytest.mark.parametrize("I", [1536, 2048])
def test_wide_intermediate(I):
    """Intermediate 1536 (the down GEMM's token tile leaves room for two ring stages and the combine's
    shared-memory transpose in 16-column passes; the other shapes here take 32-column passes) and 2048 (no room:
    the combine reduces straight from the thread's row)."""
    cfg = W.scaled(W.CONFIGS["tiny"], I=I, E=4, T=200)
    lw = weights(cfg, 0)
    logits, x_bits = W.router_logits(cfg, 0, 3), W.activations_bf16(cfg, 0, 3)
    mod, out = run(cfg, lw, logits, x_bits)
    check(cfg, lw, mod, out, logits, x_bits)


def boundary_tokens(offsets, perm, k, heavy=10, extra=256, seed=0):
    """Tokens whose expert rows include every expert's first and last permuted row and every row of the last
    (partial) 128-row tile of the `heavy` experts with the most rows, plus a seeded sample up to `extra` more."""
    offsets = np.asarray(offsets)
    perm = np.asarray(perm)
    rows = set()
    counts = np.diff(offsets)
    for e in np.nonzero(counts)[0]:
        rows.add(int(offsets[e]))
        rows.add(int(offsets[e + 1]) - 1)
    for e in np.argsort(-counts, kind="stable")[:heavy]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        last_tile = lo + 128 * ((hi - lo - 1) // 128)
        rows.update(range(last_tile, hi))
    toks = set(int(perm[p]) // k for p in rows)
    T = len(perm) // k
    rng = np.random.default_rng(seed)
    toks.update(int(t) for t in rng.choice(T, size=min(extra, T), replace=False))
    return sorted(toks)


def test_prefill_35b_zipf_boundary_tokens():
    """4096 tokens with Zipf(1.1) expert popularity.  Checked against the oracle: every token owning some
    expert's first or last permuted row, every token in the last partial 128-row tile of the ten heaviest
    experts, and 256 more drawn at random (several hundred tokens, every expert's tile boundaries)."""
    cfg = W.CONFIGS["prefill_35b"]
    lw = weights(cfg, 0)
    logits, x_bits = W.router_logits(cfg, 0, 0), W.activations_bf16(cfg, 0, 0)
    mod, out = run(cfg, lw, logits, x_bits)
    offsets = mod.offsets.cpu().numpy()
    counts = np.diff(offsets)
    assert counts.max() > 1000 and counts.min() < 100   # skewed groups, as Zipf(1.1) popularity gives
    rows = boundary_tokens(offsets, mod.perm.cpu().numpy(), cfg.k)
    assert len(rows) >= 256
    check(cfg, lw, mod, out, logits, x_bits, rows=rows)


def test_umma_packing_places_every_byte_where_the_layout_says():
    cfg = W.CONFIGS["tiny"]
    rows = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_ROWS)
    umma = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_UMMA_TILES)
    for lw in (rows, umma):
        lw.set_expert(2, *(to_dev(W.weights_fp32(cfg, 0, 2, p)) for p in range(3)))
    torch.cuda.synchronize()
    codes = rows.gu_codes[2].cpu().numpy()    # [2I][H/2]
    scales = rows.gu_scales[2].cpu().numpy()  # [2I][H/16]
    blob = umma.gu_codes[2].cpu().numpy()
    N, K = 2 * cfg.I, cfg.H
    KSN = K // 128
    for n in range(0, N, 7):
        rt, r = divmod(n, 128)
        for kk in range(0, K // 2, 5):
            ks, b = divmod(kk, 64)
            base = (rt * KSN + ks) * 9216
            assert blob[base + (b // 16) * 2048 + (r // 8) * 128 + (r % 8) * 16 + b % 16] == codes[n, kk]
        for j in range(K // 16):
            ks, jj = divmod(j, 8)
            base = (rt * KSN + ks) * 9216
            assert blob[base + 8192 + (jj // 4) * 512 + (r % 32) * 16 + (r // 32) * 4 + jj % 4] == scales[n, j]


def test_hidden_beyond_resident_token_tile_streams_both_operands():
    """H = 2304 (18 K blocks of 128) is too long for the resident token tile, so the gate/up GEMM
    streams both operands; the down GEMM (I = 128) keeps its token tile resident."""
    cfg = W.scaled(W.CONFIGS["tiny"], H=2304, T=40)
    lw = weights(cfg, 0, generated=False)
    logits, x_bits = W.router_logits(cfg, 0, 3), W.activations_bf16(cfg, 0, 3)
    mod, out = run(cfg, lw, logits, x_bits)
    check(cfg, lw, mod, out, logits, x_bits)


@pytest.mark.parametrize("case", ["short_total", "decreasing", "negative_start"])
def test_offsets_that_do_not_partition_the_rows_are_reported_and_add_nothing(case):
    """offsets must split [0, T*k) into consecutive per-expert ranges; anything else is flagged on the
    device and no expert row is computed, so no tile index can run past the workspace."""
    cfg = W.CONFIGS["tiny"]
    lw = weights(cfg, 0)
    logits, x_bits = W.router_logits(cfg, 0, 3), W.activations_bf16(cfg, 0, 3)
    mod, out = run(cfg, lw, logits, x_bits)
    bad = mod.offsets.clone()
    if case == "short_total":
        bad[-1] -= 1
    elif case == "decreasing":
        bad[2] = int(bad[3].item()) + 1  # expert 2 would end before it starts
    else:
        bad[0] = -128
    out.fill_(1.0)
    Q.ft_moe_expert_ffn_nvfp4_prefill(lw.w, to_dev(x_bits.view(np.int16), torch.bfloat16), cfg.k, bad, mod.perm,
                                      mod.w, out, mod.ws)
    assert Q.ft_device_status() == Q.FT_DEVERR_BAD_INDEX
    assert not out.float().abs().sum().item()
    # the workspace stays usable: a valid call after the failed one is exact again
    mod2, out2 = run(cfg, lw, logits, x_bits)
    check(cfg, lw, mod2, out2, logits, x_bits)


def test_streamed_layers_equal_resident_weights():
    """Three layers of a k = 2 prefill whose experts stream from pinned host memory through two device buffers,
    called twice: every layer's output equals, bit for bit, the same call on resident weights (with k = 2 each
    output element receives two fp32 additions onto zero, so their order cannot matter), and layer 0 also agrees
    with the oracle."""
    from quantized_expert_ffn_06_b300.layer import StreamedPrefill
    cfg = W.scaled(W.CONFIGS["tiny"], T=200)
    L = 3
    lws = [weights(cfg, l) for l in range(L)]
    sp = StreamedPrefill(L, cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    for l in range(L):
        sp.load_layer(l, lws[l].w)
    logits = [W.router_logits(cfg, l, 5) for l in range(L)]
    xs = [W.activations_bf16(cfg, l, 5) for l in range(L)]
    lg_d = [to_dev(a) for a in logits]
    x_d = [to_dev(a.view(np.int16), torch.bfloat16) for a in xs]
    for call in range(2):
        outs = [torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
        sp(lg_d, x_d, outs)
        torch.cuda.synchronize()
        assert Q.ft_device_status() == 0
        for l in range(L):
            mod, ref = run(cfg, lws[l], logits[l], xs[l])
            assert torch.equal(outs[l], ref), (call, l)
            if l == 0 and call == 0:
                check(cfg, lws[0], mod, outs[0], logits[0], xs[0])


def test_per_row_outputs_and_slot_table():
    """The per-row expert outputs y (fp32, no routing weight) against the oracle's y; the same call through a slot
    table that stores expert e at slot perm[e] gives bit-identical outputs (k = 2: two fp32 additions onto zero per
    output element, so their order cannot matter); an expert mapped to an invalid slot is flagged and contributes
    nothing (the oracle with that expert's weights all zero)."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=200)
    dl = weights(cfg, 0)
    logits, x_bits = W.router_logits(cfg, 0, 6), W.activations_bf16(cfg, 0, 6)
    mod, out = run(cfg, dl, logits, x_bits)
    x_dev = to_dev(x_bits.view(np.int16), torch.bfloat16)
    y = torch.full((cfg.T * cfg.k, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    Q.ft_moe_expert_ffn_nvfp4_prefill(dl.w, x_dev, cfg.k, mod.offsets, mod.perm, mod.w, None, mod.ws, y=y)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    ref = O.moe_layer(logits, x_bits, cfg.k, dl.oracle, O.MODE_A4)
    assert_layer_close(y.cpu().numpy(), ref["y"], "prefill y")

    slots = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, n_weights=cfg.E, layout=Q.FT_LAYOUT_UMMA_TILES)
    perm = np.random.default_rng(5).permutation(cfg.E)
    for e in range(cfg.E):
        s = int(perm[e])
        slots.gu_codes[s].copy_(dl.w.gu_codes[e])
        slots.d_codes[s].copy_(dl.w.d_codes[e])
        slots.tscale[s].copy_(dl.w.tscale[e])
    slots.expert_to_slot = to_dev(perm.astype(np.int32))
    out_s = torch.empty_like(out)
    Q.ft_moe_expert_ffn_nvfp4_prefill(slots, x_dev, cfg.k, mod.offsets, mod.perm, mod.w, out_s, mod.ws)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    assert torch.equal(out_s, out)

    counts = np.diff(mod.offsets.cpu().numpy())
    bad = int(np.argmax(counts))   # an expert with rows
    table = perm.astype(np.int32).copy()
    table[bad] = -1
    slots.expert_to_slot = to_dev(table)
    Q.ft_moe_expert_ffn_nvfp4_prefill(slots, x_dev, cfg.k, mod.offsets, mod.perm, mod.w, out_s, mod.ws)
    assert Q.ft_device_status() == Q.FT_DEVERR_BAD_INDEX
    H, I = cfg.H, cfg.I
    zero = O.QuantizedExpert((np.zeros((I, H // 2), np.uint8), np.zeros((I, H // 16), np.uint8), 1.0),
                             (np.zeros((I, H // 2), np.uint8), np.zeros((I, H // 16), np.uint8), 1.0),
                             (np.zeros((H, I // 2), np.uint8), np.zeros((H, I // 16), np.uint8), 1.0))
    ref_bad = O.moe_layer(logits, x_bits, cfg.k, lambda e: zero if e == bad else dl.oracle(e), O.MODE_A4)
    assert_layer_close(out_s.float().cpu().numpy(), ref_bad["out"], "prefill without the unmapped expert")
