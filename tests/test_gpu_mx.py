"""GPU tests of the MX expert weights (MXFP4 and MXFP8): the quantisers and the tile packings bit for bit against the
oracle's statement of the formats (oracle/mx.py) and of the layouts, and the fused decode layer step on MX tiles
against the oracle layer reading the device's own row-layout MX bytes (relative L2 5e-3, max |err| 2e-2 * RMS), on
the one-token path (routing by one warp) and the multi-token path.  MXFP4 weights on the tensor-core prefill: the
re-encoded tiles dequantise (by the oracle's NVFP4 reading) to exactly the MX values, and the prefill layer matches
the oracle's A4-mode layer on the MX bytes.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import assert_layer_close
from oracle import mx as MX

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import FusedDecodeLayer, LayerWeights, PrefillLayer


FMTS = ["mxfp4", "mxfp8"]


def quantize_on_device(w: np.ndarray, fmt: str = "mxfp4"):
    N, K = w.shape
    codes = torch.empty((N, K // 2 if fmt == "mxfp4" else K), dtype=torch.uint8, device=DEV)
    scales = torch.empty((N, K // 32), dtype=torch.uint8, device=DEV)
    quant = Q.ft_mxfp4_quantize_weight if fmt == "mxfp4" else Q.ft_mxfp8_quantize_weight
    quant(torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), codes, scales)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return codes.cpu().numpy(), scales.cpu().numpy()


def special_matrix(rng):
    """Blocks that reach every branch of the format: all zeros, subnormal-only amax, the largest fp32 values, exact
    grid points, the midpoints between grid values (ties), values above 6 * 2^X (saturation) and signed zeros."""
    K = 32 * 12
    w = rng.normal(0, 0.02, (16, K)).astype(np.float32)
    w[0, :32] = 0.0
    w[1, :32] = -0.0
    w[1, 32:64] = rng.uniform(-1, 1, 32).astype(np.float32) * np.float32(1e-42)    # subnormal amax
    w[2, :32] = np.float32(3.0e38) * rng.choice([-1, 1], 32)                       # X = 125
    w[2, 32:64] = np.float32(2.0 ** -130) * rng.integers(1, 8, 32)                  # X clamped to -127
    grid = np.concatenate([MX.E2M1_MAG, -MX.E2M1_MAG[1:]])
    w[3, :32] = rng.choice(grid, 32).astype(np.float32) * 4                         # exact grid points, amax 24
    w[3, 0] = 24.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    w[4, :32] = rng.choice(np.concatenate([mids, -mids]), 32).astype(np.float32)   # ties, amax 5 -> X = 0
    w[4, 31] = 5.0
    w[5, :32] = rng.normal(0, 1, 32).astype(np.float32)
    w[5, 0] = 7.9                                                                  # above 6 * 2^X: saturates
    w[6, :32] = -1e-30                                                             # negative, rounds to -0
    w[6, 0] = 1.0
    return w


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("which", ["normal", "special", "wide"])
def test_quantiser_bit_exact_against_oracle(which, fmt):
    rng = np.random.default_rng({"normal": 0, "special": 1, "wide": 2}[which])
    if which == "normal":
        w = rng.normal(0, 0.02, (512, 2048)).astype(np.float32)
    elif which == "special":
        w = special_matrix(rng)
    else:  # magnitudes over the whole fp32 range, one decade per block
        w = (rng.normal(0, 1, (256, 1024)) * 10.0 ** rng.integers(-40, 37, (256, 32)).repeat(32, axis=1)).astype(np.float32)
    if fmt == "mxfp8" and which == "special":   # E4M3 ties and saturation at its own grid
        w[4, :32] = np.float32(256.0 + 16.0) * np.sign(w[4, :32])   # halfway between 256 and 288
        w[4, 31] = 416.0                                            # amax 416: X = 0; 416 = 448 - 32 exact
        w[5, 0] = 470.0                                             # above 448 * 2^X: saturates
    codes, scales = quantize_on_device(w, fmt)
    want_c, want_s = MX.quantize(w, fmt)
    assert np.array_equal(scales, want_s)
    assert np.array_equal(codes, want_c)


def unpack_mx_tiles(tiles: np.ndarray, N: int, K: int, fmt: str = "mxfp4"):
    """Rows-layout codes and scales read back from MX decode tiles by the layout statements of ft_mxfp4_pack_tiles
    and ft_mxfp8_pack_tiles: with P code bytes per lane and half tile (16 for MXFP4, 32 for MXFP8) and C = 32 P
    code bytes per half tile, the codes of row 8h+g, bytes Pq..Pq+P-1 of K-block kb, at kb*2C + h*C + (g*4+q)*P;
    the scale of block 4kb+q of row 8h+g at (K/128)*2C + kb*64 + (g*4+q)*2 + h."""
    KB = K // 128
    P = 16 if fmt == "mxfp4" else 32
    C = 32 * P
    t = tiles.reshape(N // 16, KB * (2 * C + 64))
    codes = np.empty((N, KB * 4 * P), np.uint8)
    scales = np.empty((N, K // 32), np.uint8)
    for kb in range(KB):
        for h in range(2):
            for g in range(8):
                for q in range(4):
                    off = kb * 2 * C + h * C + (g * 4 + q) * P
                    codes[8 * h + g::16, kb * 4 * P + P * q:kb * 4 * P + P * q + P] = t[:, off:off + P]
                    scales[8 * h + g::16, kb * 4 + q] = t[:, KB * 2 * C + kb * 64 + (g * 4 + q) * 2 + h]
    return codes, scales


@pytest.mark.parametrize("fmt", FMTS)
def test_pack_tiles_places_every_byte(fmt):
    rng = np.random.default_rng(3)
    N, K = 48, 384
    cb = K // 2 if fmt == "mxfp4" else K
    codes = torch.from_numpy(rng.integers(0, 256, (N, cb), dtype=np.uint8)).to(DEV)
    scales = torch.from_numpy(rng.integers(0, 255, (N, K // 32), dtype=np.uint8)).to(DEV)
    tiles = torch.empty(N * K * (17 if fmt == "mxfp4" else 33) // 32, dtype=torch.uint8, device=DEV)
    pack = Q.ft_mxfp4_pack_tiles if fmt == "mxfp4" else Q.ft_mxfp8_pack_tiles
    pack(codes, cb, scales, K // 32, N, K, tiles)
    got_c, got_s = unpack_mx_tiles(tiles.cpu().numpy(), N, K, fmt)
    assert np.array_equal(got_c, codes.cpu().numpy())
    assert np.array_equal(got_s, scales.cpu().numpy())


class MxOracleExperts:
    """expert(e) for O.moe_layer: the device's row-layout MXFP4 bytes (gate and up are the even and odd rows of the
    interleaved gate/up matrix), dequantised by the oracle."""

    def __init__(self, rows, fmt="mxfp4"):
        self.rows, self.fmt = rows, fmt

    def __call__(self, e):
        r, f = self.rows, self.fmt
        gc, gs = r.gu_codes[e].cpu().numpy(), r.gu_scales[e].cpu().numpy()
        dc, ds = r.d_codes[e].cpu().numpy(), r.d_scales[e].cpu().numpy()

        class Ex:
            pass

        ex = Ex()
        ex.Wg = MX.dequantize(gc[0::2], gs[0::2], f)
        ex.Wu = MX.dequantize(gc[1::2], gs[1::2], f)
        ex.Wd = MX.dequantize(dc, ds, f)
        return ex


def mx_layer(cfg, layer, fmt="mxfp4"):
    """The same fp32 draws quantised twice on the device: row layout (what the oracle reads) and decode tiles."""
    stream_of = lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p)  # noqa: E731
    lr, lt = ((Q.FT_LAYOUT_MXFP4_ROWS, Q.FT_LAYOUT_MXFP4_DECODE_TILES) if fmt == "mxfp4" else
              (Q.FT_LAYOUT_MXFP8_ROWS, Q.FT_LAYOUT_MXFP8_DECODE_TILES))
    rows = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=lr)
    rows.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    tiles = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=lt)
    tiles.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    torch.cuda.synchronize()
    return rows, tiles


def check_fused(cfg, rows, tiles, layer, step, T, fmt="mxfp4"):
    logits = W.router_logits(cfg, layer, step, T=T)
    x_bits = W.activations_bf16(cfg, layer, step, T=T)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
    mod(tiles, torch.from_numpy(logits).to(DEV),
        torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).to(DEV), out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    r = O.moe_layer(logits, x_bits, cfg.k, MxOracleExperts(rows, fmt), O.MODE_A16)
    assert np.array_equal(mod.ids.cpu().numpy(), r["ids"])
    assert_layer_close(out.float().cpu().numpy(), r["out"], f"{fmt} layer {layer} step {step} T={T}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fused_decode_mx_tiny(fmt):
    cfg = W.CONFIGS["tiny"]
    rows, tiles = mx_layer(cfg, 0, fmt)
    for T in (1, 4):
        check_fused(cfg, rows, tiles, 0, 0, T, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_fused_decode_mx_35b_shape(fmt):
    """Hidden 2048, 256 experts, top-8, intermediate 512: one token (one-warp routing) at several steps, and 16
    tokens (the multi-token path)."""
    cfg = W.CONFIGS["decode_35b"]
    rows, tiles = mx_layer(cfg, 0, fmt)
    for step in range(3):
        check_fused(cfg, rows, tiles, 0, step, 1, fmt)
    check_fused(cfg, rows, tiles, 0, 5, 16, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_tiles_equal_repacked_rows(fmt):
    """The decode tiles drawn directly equal the row-layout bytes packed by the pack call (the quantiser is
    deterministic), so the oracle's bytes are the kernel's bytes."""
    cfg = W.scaled(W.CONFIGS["tiny"], E=3)
    rows, tiles = mx_layer(cfg, 1, fmt)
    H, I = cfg.H, cfg.I
    for e in range(cfg.E):
        gc, gs = unpack_mx_tiles(tiles.gu_codes[e].cpu().numpy(), 2 * I, H, fmt)
        dc, ds = unpack_mx_tiles(tiles.d_codes[e].cpu().numpy(), H, I, fmt)
        assert np.array_equal(gc, rows.gu_codes[e].cpu().numpy()) and np.array_equal(gs, rows.gu_scales[e].cpu().numpy())
        assert np.array_equal(dc, rows.d_codes[e].cpu().numpy()) and np.array_equal(ds, rows.d_scales[e].cpu().numpy())


@pytest.mark.parametrize("fmt", FMTS)
def test_fused_decode_mx_large_shape(fmt):
    """Hidden 4096, intermediate 1536, 128 experts, top-8 (the cache workload's layer shape, K-blocks of several
    tiles per warp and a down phase split across warps), one token at two steps."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], routing="normal", T=1)
    rows, tiles = mx_layer(cfg, 0, fmt)
    for step in range(2):
        check_fused(cfg, rows, tiles, 0, step, 1, fmt)


# ---------------------------------------------------------------- MXFP4 on the tensor-core prefill

def unpack_umma(blob: np.ndarray, N: int, K: int):
    """Row-major NVFP4 codes [N][K/2] and E4M3 scales [N][K/16] read back from FT_LAYOUT_UMMA_TILES (code byte b of
    row r of a 128 x 128 block at (b/16)*2048 + (r/8)*128 + (r%8)*16 + b%16, scale j at 8192 + (j/4)*512 +
    (r%32)*16 + (r/32)*4 + j%4)."""
    KSN = K // 128
    t = blob.reshape(N // 128, KSN, 9216)
    c = t[:, :, :8192].reshape(N // 128, KSN, 4, 16, 8, 16).transpose(0, 3, 4, 1, 2, 5).reshape(N, K // 2)
    s = t[:, :, 8192:].reshape(N // 128, KSN, 2, 32, 4, 4).transpose(0, 4, 3, 1, 2, 5).reshape(N, K // 16)
    return c, s


def mx_umma_layer(cfg, layer):
    """The same fp32 draws as MXFP4 rows (what the oracle reads) and as tensor-core tiles re-encoded from MXFP4."""
    stream_of = lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p)  # noqa: E731
    rows = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_MXFP4_ROWS)
    rows.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    umma = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_UMMA_TILES, source="mxfp4")
    umma.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return rows, umma


def test_mxfp4_umma_tiles_dequantise_to_the_mx_values():
    """Every expert's gate/up and down tiles: the codes are the MX codes, and E4M3 scale x tensor scale reproduces
    each block's 2^(s-127) exactly (two independent oracle dequantisers agree bit for bit)."""
    cfg = W.scaled(W.CONFIGS["tiny"], E=3)
    rows, umma = mx_umma_layer(cfg, 2)
    H, I = cfg.H, cfg.I
    ts = umma.tscale.cpu().numpy()
    for e in range(cfg.E):
        for blob, codes, scales, N, K, t in ((umma.gu_codes[e], rows.gu_codes[e], rows.gu_scales[e], 2 * I, H, ts[e, 0]),
                                             (umma.d_codes[e], rows.d_codes[e], rows.d_scales[e], H, I, ts[e, 2])):
            c, s = unpack_umma(blob.cpu().numpy(), N, K)
            mc, ms = codes.cpu().numpy(), scales.cpu().numpy()
            assert np.array_equal(c, mc)
            got = O.dequantize(c, s, float(t))
            want = MX.dequantize(mc, ms, "mxfp4")
            assert np.array_equal(got, want)
        assert ts[e, 0] == ts[e, 1]


@pytest.mark.parametrize("spread", [17, 18])
def test_mxfp4_umma_exponent_span(spread):
    """Non-zero blocks 17 octaves below the largest are still exact; 18 set FT_DEVERR_RANGE.  All-zero blocks (any
    scale byte) get scale 0 and do not count."""
    rng = np.random.default_rng(spread)
    N, K = 128, 256
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(124, 130, (N, K // 32), dtype=np.uint8)
    scales[0, 0] = 140                 # the largest: s0 = 132, tensor scale 2^5
    scales[5, 3] = 140 - spread        # 2^-9 (the smallest E4M3 power of two) or beyond
    codes[5, 48:64] = 0x31             # that block holds non-zero codes
    codes[9, 16:32] = 0x80            # an all-zero block (signed zeros) with an out-of-span scale
    scales[9, 1] = 3
    tiles = torch.empty(N * K * 9 // 16, dtype=torch.uint8, device=DEV)
    ts = torch.zeros(1, dtype=torch.float32, device=DEV)
    assert Q.ft_device_status() == 0
    Q.ft_mxfp4_pack_umma(torch.from_numpy(codes).to(DEV), K // 2, torch.from_numpy(scales).to(DEV), K // 32, N, K,
                         tiles, ts, 1)
    torch.cuda.synchronize()
    st = Q.ft_device_status()
    if spread == 17:
        assert st == 0
        c, s = unpack_umma(tiles.cpu().numpy(), N, K)
        assert np.array_equal(O.dequantize(c, s, float(ts.item())), MX.dequantize(codes, scales, "mxfp4"))
        assert s[9, 2] == 0 and s[9, 3] == 0
    else:
        assert st == Q.FT_DEVERR_RANGE


def test_mxfp4_umma_nan_scale_is_reported():
    """A UE8M0 scale byte of 255 (NaN) sets FT_DEVERR_BAD_SCALE; the packing still finishes."""
    rng = np.random.default_rng(5)
    N, K = 128, 128
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = np.full((N, K // 32), 127, np.uint8)
    scales[7, 2] = 255
    tiles = torch.empty(N * K * 9 // 16, dtype=torch.uint8, device=DEV)
    ts = torch.zeros(1, dtype=torch.float32, device=DEV)
    assert Q.ft_device_status() == 0
    Q.ft_mxfp4_pack_umma(torch.from_numpy(codes).to(DEV), K // 2, torch.from_numpy(scales).to(DEV), K // 32, N, K,
                         tiles, ts, 1)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == Q.FT_DEVERR_BAD_SCALE


def run_prefill(cfg, umma, logits, x_bits):
    T = logits.shape[0]
    mod = PrefillLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod(umma, torch.from_numpy(logits).to(DEV),
        torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).to(DEV), out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return mod, out


@pytest.mark.parametrize("name,T", [("tiny", 200), ("prefill_35b", 384)])
def test_prefill_on_mxfp4_weights_matches_oracle(name, T):
    """The tensor-core prefill on MXFP4 weights (tiny layer, every output; 35B layer shape, 384 tokens) against the
    oracle's A4-mode layer on the MX-dequantised row bytes."""
    cfg = W.scaled(W.CONFIGS[name], T=T)
    rows, umma = mx_umma_layer(cfg, 0)
    logits, x_bits = W.router_logits(cfg, 0, 4), W.activations_bf16(cfg, 0, 4)
    mod, out = run_prefill(cfg, umma, logits, x_bits)
    r = O.moe_layer(logits, x_bits, cfg.k, MxOracleExperts(rows), O.MODE_A4)
    assert np.array_equal(mod.ids.cpu().numpy(), r["ids"])
    assert_layer_close(out.float().cpu().numpy(), r["out"], f"mxfp4 prefill {name} T={T}")
