"""GPU parity of the decode layer step (route -> permute -> NVFP4 expert FFN -> combine).

The weights are drawn and quantised on the device (or, for the small layers, uploaded from the host generator and
quantised there) into canonical row-layout NVFP4 bytes; the layer weights handle (ft_moe_weights_create) repacks
those bytes into the kernel layouts, and the oracle reads the very same canonical bytes, copied to the host.  ids,
offsets, perm and inv are compared bit for bit; outputs within relative L2 5e-3 and max |err| 2e-2 * RMS.

Three paths are checked:
  rows  -- route / permute / expert FFN / combine as separate calls, row-major weights
  tiles -- the same separate calls on tiled weights (the fused kernel in grouped mode)
  fused -- the single-launch layer step on tiled weights
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import OracleExperts, assert_layer_close, oracle_expert

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import FusedDecodeLayer, LayerWeights, MoEDecodeLayer, MoEWeights
DEV = "cuda:0"
PATHS = ["rows", "tiles", "fused"]


def layout_of(path):
    return Q.FT_LAYOUT_ROWS if path == "rows" else Q.FT_LAYOUT_DECODE_TILES


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


class DeviceLayer:
    """Canonical row-layout NVFP4 weights of one layer on the device, and the handle's kernel layouts of them."""

    def __init__(self, cfg, layer, from_host=False):
        self.canon = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_ROWS)
        if from_host:
            for e in range(cfg.E):
                self.canon.set_expert(e, *(to_dev(W.weights_fp32(cfg, layer, e, p)) for p in range(3)))
        else:
            self.canon.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
        self.handle = MoEWeights(self.canon, Q.FT_WEIGHTS_ROWS | Q.FT_WEIGHTS_DECODE_TILES)
        self.oracle = OracleExperts(self.canon)

    def view(self, path):
        return self.handle.view(layout_of(path))


def device_weights_from_host(cfg, layer, experts=None, layout=0):
    """Upload the host generator's fp32 weights and quantise them on the device (one layout, no handle)."""
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=layout)
    for e in (range(cfg.E) if experts is None else experts):
        lw.set_expert(e, *(to_dev(W.weights_fp32(cfg, layer, e, p)) for p in range(3)))
    return lw


def device_weights_generated(cfg, layer, layout=0):
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=layout)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
    return lw


def run_layer(cfg, lw, layer, step, T=None, want_y=False, path="rows"):
    T = cfg.T if T is None else T
    logits = W.router_logits(cfg, layer, step, T=T)
    x_bits = W.activations_bf16(cfg, layer, step, T=T)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    y = None
    if path == "fused":
        mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
        mod(lw, to_dev(logits), to_dev(x_bits.view(np.int16), torch.bfloat16), out)
    else:
        mod = MoEDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
        y = torch.empty((T * cfg.k, cfg.H), dtype=torch.float32, device=DEV) if want_y else None
        mod(lw, to_dev(logits), to_dev(x_bits.view(np.int16), torch.bfloat16), out, y=y)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return logits, x_bits, mod, out, y


def oracle_layer(cfg, dl, logits, x_bits, rows=None):
    """The oracle on the device's own bytes (dl: a DeviceLayer)."""
    return O.moe_layer(logits, x_bits, cfg.k, dl.oracle, O.MODE_A16, rows=rows)


def check_routing(mod, ref):
    assert np.array_equal(mod.ids.cpu().numpy(), ref["ids"])
    if hasattr(mod, "perm"):
        assert np.array_equal(mod.offsets.cpu().numpy(), ref["offsets"])
        assert np.array_equal(mod.perm.cpu().numpy(), ref["perm"])
        assert np.array_equal(mod.inv.cpu().numpy(), ref["inv"])
    w = mod.w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w - ref["w"]) <= 1e-5 * ref["w"] + 1e-7)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_layer_every_output(path):
    cfg = W.CONFIGS["tiny"]
    dl = DeviceLayer(cfg, 0, from_host=True)
    logits, x_bits, mod, out, y = run_layer(cfg, dl.view(path), 0, 0, want_y=True, path=path)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "tiny out")
    if y is not None:
        # every per-row expert output as well (y is not rounded)
        assert_layer_close(y.cpu().numpy(), ref["y"], "tiny y")


def test_device_weights_equal_oracle_weights_on_samples():
    """Device generator + device quantiser reproduce the oracle's NVFP4 bytes (sampled experts)."""
    cfg = W.CONFIGS["decode_35b"]
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_ROWS)
    experts = [0, 77, 255]
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, 5, e, p), sigma=cfg.w_sigma, experts=experts)
    torch.cuda.synchronize()
    for e in experts:
        ex = oracle_expert(cfg, 5, e)
        (gc, gs, gts), (uc, us, uts), (dc, ds, dts) = ex.q
        gu_c = lw.gu_codes[e].cpu().numpy()
        gu_s = lw.gu_scales[e].cpu().numpy()
        ts = lw.tscale[e].cpu().numpy()
        assert ts[0] == gts and ts[1] == uts and ts[2] == dts
        # allow a rare fp32 rounding difference of the generator to flip one code
        for got, want in ((gu_c[0::2], gc), (gu_c[1::2], uc), (lw.d_codes[e].cpu().numpy(), dc)):
            assert (got != want).sum() <= 2
        for got, want in ((gu_s[0::2], gs), (gu_s[1::2], us), (lw.d_scales[e].cpu().numpy(), ds)):
            assert (got != want).sum() <= 2


def test_tile_packing_is_a_permutation_of_row_bytes():
    """Every code and scale byte of a row-major matrix lands once in the tiled layout, where the doc says."""
    cfg = W.CONFIGS["tiny"]
    rows = device_weights_from_host(cfg, 0, experts=[3], layout=Q.FT_LAYOUT_ROWS)
    tiles = device_weights_from_host(cfg, 0, experts=[3], layout=Q.FT_LAYOUT_DECODE_TILES)
    codes = rows.d_codes[3].cpu().numpy()      # [H][I/2]
    scales = rows.d_scales[3].cpu().numpy()    # [H][I/16]
    tb = tiles.d_codes[3].cpu().numpy()
    N, K = cfg.H, cfg.I
    KB = K // 128
    for n in range(0, N, 5):
        tile, rr = divmod(n, 16)
        h, g = divmod(rr, 8)
        base = tile * KB * 1152
        for b in range(0, K // 2, 3):
            kb, within = divmod(b, 64)
            q, i = divmod(within, 16)
            assert tb[base + kb * 1024 + h * 512 + (g * 4 + q) * 16 + i] == codes[n, b]
        for blk in range(K // 16):
            kb, j = divmod(blk, 8)
            q, bb = divmod(j, 2)
            assert tb[base + KB * 1024 + kb * 128 + (g * 4 + q) * 4 + 2 * h + bb] == scales[n, blk]


@pytest.fixture(scope="module")
def layers35():
    cfg = W.CONFIGS["decode_35b"]
    return {layer: DeviceLayer(cfg, layer) for layer in (0, 7, 47)}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("layer,step", [(0, 0), (7, 3), (47, 255)])
def test_decode_35b_layer(layers35, layer, step, path):
    cfg = W.CONFIGS["decode_35b"]
    dl = layers35[layer]
    logits, x_bits, mod, out, _ = run_layer(cfg, dl.view(path), layer, step, path=path)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], f"35B layer {layer} step {step}")


@pytest.fixture(scope="module")
def layer753():
    return DeviceLayer(W.CONFIGS["decode_753b_b1"], 3)


@pytest.mark.parametrize("path", PATHS)
def test_decode_753b_batch1_layer(layer753, path):
    cfg = W.CONFIGS["decode_753b_b1"]
    logits, x_bits, mod, out, _ = run_layer(cfg, layer753.view(path), 3, 11, path=path)
    ref = oracle_layer(cfg, layer753, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "753B b1")


@pytest.mark.parametrize("path", ["rows", "fused"])
def test_decode_753b_batch16_every_token(layer753, path):
    """Batch 16 of hidden 6144, all 16 tokens against the oracle: the fused step runs as launches over token
    chunks that fit its shared memory."""
    cfg = W.CONFIGS["decode_753b_b16"]
    logits, x_bits, mod, out, _ = run_layer(cfg, layer753.view(path), 3, 2, path=path)
    ref = oracle_layer(cfg, layer753, logits, x_bits)
    check_routing(mod, ref)
    got = out.float().cpu().numpy()
    for t in range(cfg.T):
        assert_layer_close(got[t:t + 1], ref["out"][t:t + 1], f"753B b16 token {t} ({path})")


def test_fused_token_chunks_agree_with_single_token_launches():
    """A batch run as token chunks agrees with one launch per token.  The chunk size changes how the
    down tiles are split across warps (so the fp32 summation order), hence a last-bf16-bit tolerance."""
    cfg = W.scaled(W.CONFIGS["decode_753b_b16"], T=5)
    lw = device_weights_generated(cfg, 1, layout=Q.FT_LAYOUT_DECODE_TILES)
    logits = to_dev(W.router_logits(cfg, 1, 4))
    x = to_dev(W.activations_bf16(cfg, 1, 4).view(np.int16), torch.bfloat16)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    mod(lw, logits, x, out)
    one = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, 1, DEV)
    for t in range(cfg.T):
        o1 = torch.empty((1, cfg.H), dtype=torch.bfloat16, device=DEV)
        one(lw, logits[t:t + 1].contiguous(), x[t:t + 1].contiguous(), o1)
        torch.cuda.synchronize()
        assert torch.equal(one.ids[0], mod.ids[t])
        a, b = out[t].float(), o1[0].float()
        rms = b.pow(2).mean().sqrt()
        assert ((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-3 * rms).all(), t
    assert Q.ft_device_status() == 0


def test_tiled_grouped_kernel_reports_unsupported_staging_size():
    """The grouped-mode launch (separate route and permute) stages the whole batch: 16 tokens of hidden 6144
    do not fit, and the call says so without launching."""
    cfg = W.CONFIGS["decode_753b_b16"]
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_DECODE_TILES, n_weights=cfg.E)
    with pytest.raises(Q.FtError) as ei:
        run_layer(cfg, lw, 1, 2, path="tiles")
    assert ei.value.status == Q.FT_ERR_UNSUPPORTED


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [13, 16])
def test_ragged_token_counts_and_single_expert_segments(path, T):
    """T tokens over 8 experts with k = 2: segments of uneven length, several token groups."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=T)
    dl = DeviceLayer(cfg, 0, from_host=True)
    logits, x_bits, mod, out, _ = run_layer(cfg, dl.view(path), 0, 4, path=path)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "ragged")


def test_empty_batch_is_a_no_op():
    cfg = W.CONFIGS["tiny"]
    lw = device_weights_from_host(cfg, 0, experts=[0])
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device=DEV)
    offsets = torch.zeros(cfg.E + 1, dtype=torch.int32, device=DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    y, out = Q.ft_moe_expert_ffn_nvfp4_decode(lw, x, cfg.k, offsets, e, e, y=e)
    assert y.numel() == 0


@pytest.mark.parametrize("path", PATHS)
def test_slot_table_indirection(path):
    """Weights addressed through expert_to_slot give the same output as direct addressing."""
    cfg = W.CONFIGS["tiny"]
    lay = layout_of(path)
    direct = device_weights_from_host(cfg, 0, layout=lay)
    slots = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, n_weights=cfg.E, layout=lay)
    perm = np.random.default_rng(3).permutation(cfg.E)
    for e in range(cfg.E):   # expert e lives in slot perm[e]
        s = int(perm[e])
        for a, b in ((slots.gu_codes, direct.gu_codes), (slots.gu_scales, direct.gu_scales),
                     (slots.d_codes, direct.d_codes), (slots.d_scales, direct.d_scales),
                     (slots.tscale, direct.tscale)):
            if a is not None:
                a[s].copy_(b[e])
    slots.expert_to_slot = to_dev(perm.astype(np.int32))
    _, _, _, out_a, _ = run_layer(cfg, direct, 0, 0, path=path)
    _, _, _, out_b, _ = run_layer(cfg, slots, 0, 0, path=path)
    assert torch.equal(out_a, out_b)


def test_fused_and_grouped_tiled_paths_agree_bitwise():
    """Same kernel, same routing numerics, same summation order: identical outputs."""
    cfg = W.CONFIGS["decode_35b"]
    lw = device_weights_generated(cfg, 2, layout=Q.FT_LAYOUT_DECODE_TILES)
    _, _, _, out_f, _ = run_layer(cfg, lw, 2, 5, path="fused")
    _, _, _, out_t, _ = run_layer(cfg, lw, 2, 5, path="tiles")
    assert torch.equal(out_f, out_t)


def test_fused_repeated_calls_share_workspace():
    """The grid-barrier counter in the workspace stays consistent across many calls."""
    cfg = W.CONFIGS["tiny"]
    lw = device_weights_from_host(cfg, 0, layout=Q.FT_LAYOUT_DECODE_TILES)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    logits = to_dev(W.router_logits(cfg, 0, 0))
    x = to_dev(W.activations_bf16(cfg, 0, 0).view(np.int16), torch.bfloat16)
    outs = []
    for _ in range(50):
        out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
        mod(lw, logits, x, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    assert all(torch.equal(o, outs[0]) for o in outs)


def test_fused_nan_logits_flag_and_stay_in_bounds():
    cfg = W.CONFIGS["tiny"]
    lw = device_weights_from_host(cfg, 0, layout=Q.FT_LAYOUT_DECODE_TILES)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    logits = W.router_logits(cfg, 0, 0).copy()
    logits[1, :] = np.nan
    x = to_dev(W.activations_bf16(cfg, 0, 0).view(np.int16), torch.bfloat16)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod(lw, to_dev(logits), x, out)
    assert Q.ft_device_status() & Q.FT_DEVERR_NAN_LOGIT
    ids = mod.ids.cpu().numpy()
    assert ids.min() >= 0 and ids.max() < cfg.E


def fused_run(cfg, lw, logits_dev, x_bits):
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, logits_dev.shape[0], DEV)
    out = torch.empty((logits_dev.shape[0], cfg.H), dtype=torch.bfloat16, device=DEV)
    mod(lw, logits_dev, to_dev(x_bits.view(np.int16), torch.bfloat16), out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return mod, out


@pytest.mark.parametrize("E,k,T", [(8, 2, 4), (10, 3, 3), (512, 8, 3)])
@pytest.mark.parametrize("offset", [0, 1])
def test_fused_router_on_wide_odd_and_unaligned_logits(E, k, T, offset):
    """E = 512 spans 16 router blocks of 32 logits; E = 10 leaves most of a block empty; logits at a 4-byte offset
    (offset 1) are not 16-byte aligned."""
    cfg = W.scaled(W.CONFIGS["tiny"], E=E, k=k, T=T)
    dl = DeviceLayer(cfg, 0)
    lw = dl.view("fused")
    logits = W.router_logits(cfg, 0, 1)
    x_bits = W.activations_bf16(cfg, 0, 1)
    buf = torch.zeros(T * E + 4, dtype=torch.float32, device=DEV)
    lg = buf[offset:offset + T * E].view(T, E)
    lg.copy_(to_dev(logits))
    mod, out = fused_run(cfg, lw, lg, x_bits)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], f"E={E} offset={offset}")


def test_fused_router_ties_and_infinities():
    """Equal logits go to the lower expert id; a row of -inf gives every slot weight 1/k."""
    cfg = W.scaled(W.CONFIGS["tiny"], E=16, k=3)
    dl = DeviceLayer(cfg, 0)
    lw = dl.view("fused")
    logits = np.zeros((4, 16), np.float32)
    logits[1, [9, 3, 12]] = 2.0
    logits[2] = -np.inf
    logits[3, :] = -np.inf
    logits[3, [5, 7]] = [0.0, -0.0]
    x_bits = W.activations_bf16(cfg, 0, 3)
    mod, out = fused_run(cfg, lw, to_dev(logits), x_bits)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "ties")


@pytest.mark.parametrize("T,big_row", [(4, 1), (1, 0)])
def test_fused_activations_beyond_f16_range_are_rescaled(T, big_row):
    """A token row scaled by 2^20 overflows f16 staging: x and its h rows take the exact
    power-of-two rescaling path (one token: the one-warp router and per-warp h slices; four tokens: the
    general router).  Each token row is checked on its own scale."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=T)
    dl = DeviceLayer(cfg, 0, from_host=True)
    lw = dl.view("fused")
    logits = W.router_logits(cfg, 0, 2)
    x32 = W.bf16_bits_to_f32(W.activations_bf16(cfg, 0, 2)).copy()
    x32[big_row] *= 2.0 ** 20
    x_bits = (x32.view(np.uint32) >> 16).astype(np.uint16)   # exact: only exponents changed
    mod, out = fused_run(cfg, lw, to_dev(logits), x_bits)
    ref = oracle_layer(cfg, dl, logits, x_bits)
    check_routing(mod, ref)
    got = out.float().cpu().numpy()
    for t in range(cfg.T):
        assert_layer_close(got[t:t + 1], ref["out"][t:t + 1], f"token {t}")
