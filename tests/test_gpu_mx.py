"""GPU tests of the MXFP4 expert weights: the quantiser and the tile packing bit for bit against the oracle's
statement of the format (oracle/mx.py) and of the layout, and the fused decode layer step on MXFP4 tiles against the
oracle layer reading the device's own row-layout MXFP4 bytes (relative L2 5e-3, max |err| 2e-2 * RMS), on the
one-token path (routing by one warp) and the multi-token path.
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
    from quantized_expert_ffn_06_b300.layer import FusedDecodeLayer, LayerWeights


def quantize_on_device(w: np.ndarray):
    N, K = w.shape
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=DEV)
    scales = torch.empty((N, K // 32), dtype=torch.uint8, device=DEV)
    Q.ft_mxfp4_quantize_weight(torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), codes, scales)
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


@pytest.mark.parametrize("which", ["normal", "special", "wide"])
def test_quantiser_bit_exact_against_oracle(which):
    rng = np.random.default_rng({"normal": 0, "special": 1, "wide": 2}[which])
    if which == "normal":
        w = rng.normal(0, 0.02, (512, 2048)).astype(np.float32)
    elif which == "special":
        w = special_matrix(rng)
    else:  # magnitudes over the whole fp32 range, one decade per block
        w = (rng.normal(0, 1, (256, 1024)) * 10.0 ** rng.integers(-40, 37, (256, 32)).repeat(32, axis=1)).astype(np.float32)
    codes, scales = quantize_on_device(w)
    want_c, want_s = MX.quantize(w, "mxfp4")
    assert np.array_equal(scales, want_s)
    assert np.array_equal(codes, want_c)


def unpack_mx_tiles(tiles: np.ndarray, N: int, K: int):
    """Rows-layout codes and scales read back from MXFP4 decode tiles by the layout statement of
    ft_mxfp4_pack_tiles: codes of row 8h+g, bytes 16q..16q+15 of K-block kb, at kb*1024 + h*512 + (g*4+q)*16; the
    scale of block 4kb+q of row 8h+g at (K/128)*1024 + kb*64 + (g*4+q)*2 + h."""
    KB = K // 128
    t = tiles.reshape(N // 16, KB * 1088)
    codes = np.empty((N, K // 2), np.uint8)
    scales = np.empty((N, K // 32), np.uint8)
    for kb in range(KB):
        for h in range(2):
            for g in range(8):
                for q in range(4):
                    off = kb * 1024 + h * 512 + (g * 4 + q) * 16
                    codes[8 * h + g::16, kb * 64 + 16 * q:kb * 64 + 16 * q + 16] = t[:, off:off + 16]
                    scales[8 * h + g::16, kb * 4 + q] = t[:, KB * 1024 + kb * 64 + (g * 4 + q) * 2 + h]
    return codes, scales


def test_pack_tiles_places_every_byte():
    rng = np.random.default_rng(3)
    N, K = 48, 384
    codes = torch.from_numpy(rng.integers(0, 256, (N, K // 2), dtype=np.uint8)).to(DEV)
    scales = torch.from_numpy(rng.integers(0, 255, (N, K // 32), dtype=np.uint8)).to(DEV)
    tiles = torch.empty(N * K * 17 // 32, dtype=torch.uint8, device=DEV)
    Q.ft_mxfp4_pack_tiles(codes, K // 2, scales, K // 32, N, K, tiles)
    got_c, got_s = unpack_mx_tiles(tiles.cpu().numpy(), N, K)
    assert np.array_equal(got_c, codes.cpu().numpy())
    assert np.array_equal(got_s, scales.cpu().numpy())


class MxOracleExperts:
    """expert(e) for O.moe_layer: the device's row-layout MXFP4 bytes (gate and up are the even and odd rows of the
    interleaved gate/up matrix), dequantised by the oracle."""

    def __init__(self, rows):
        self.rows = rows

    def __call__(self, e):
        r = self.rows
        gc, gs = r.gu_codes[e].cpu().numpy(), r.gu_scales[e].cpu().numpy()
        dc, ds = r.d_codes[e].cpu().numpy(), r.d_scales[e].cpu().numpy()

        class Ex:
            pass

        ex = Ex()
        ex.Wg = MX.dequantize(gc[0::2], gs[0::2], "mxfp4")
        ex.Wu = MX.dequantize(gc[1::2], gs[1::2], "mxfp4")
        ex.Wd = MX.dequantize(dc, ds, "mxfp4")
        return ex


def mx_layer(cfg, layer):
    """The same fp32 draws quantised twice on the device: row layout (what the oracle reads) and decode tiles."""
    stream_of = lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p)  # noqa: E731
    rows = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_MXFP4_ROWS)
    rows.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    tiles = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_MXFP4_DECODE_TILES)
    tiles.fill_synthetic(stream_of, sigma=cfg.w_sigma)
    torch.cuda.synchronize()
    return rows, tiles


def check_fused(cfg, rows, tiles, layer, step, T):
    logits = W.router_logits(cfg, layer, step, T=T)
    x_bits = W.activations_bf16(cfg, layer, step, T=T)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
    mod(tiles, torch.from_numpy(logits).to(DEV),
        torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).to(DEV), out)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    r = O.moe_layer(logits, x_bits, cfg.k, MxOracleExperts(rows), O.MODE_A16)
    assert np.array_equal(mod.ids.cpu().numpy(), r["ids"])
    assert_layer_close(out.float().cpu().numpy(), r["out"], f"mxfp4 layer {layer} step {step} T={T}")


def test_fused_decode_mxfp4_tiny():
    cfg = W.CONFIGS["tiny"]
    rows, tiles = mx_layer(cfg, 0)
    for T in (1, 4):
        check_fused(cfg, rows, tiles, 0, 0, T)


def test_fused_decode_mxfp4_35b_shape():
    """Hidden 2048, 256 experts, top-8, intermediate 512: one token (one-warp routing) at several steps, and 16
    tokens (the multi-token path)."""
    cfg = W.CONFIGS["decode_35b"]
    rows, tiles = mx_layer(cfg, 0)
    for step in range(3):
        check_fused(cfg, rows, tiles, 0, step, 1)
    check_fused(cfg, rows, tiles, 0, 5, 16)


def test_mx_tiles_equal_repacked_rows():
    """The decode tiles drawn directly equal the row-layout bytes packed by ft_mxfp4_pack_tiles (the quantiser is
    deterministic), so the oracle's bytes are the kernel's bytes."""
    cfg = W.scaled(W.CONFIGS["tiny"], E=3)
    rows, tiles = mx_layer(cfg, 1)
    H, I = cfg.H, cfg.I
    for e in range(cfg.E):
        gc, gs = unpack_mx_tiles(tiles.gu_codes[e].cpu().numpy(), 2 * I, H)
        dc, ds = unpack_mx_tiles(tiles.d_codes[e].cpu().numpy(), H, I)
        assert np.array_equal(gc, rows.gu_codes[e].cpu().numpy()) and np.array_equal(gs, rows.gu_scales[e].cpu().numpy())
        assert np.array_equal(dc, rows.d_codes[e].cpu().numpy()) and np.array_equal(ds, rows.d_scales[e].cpu().numpy())


def test_fused_decode_mxfp4_large_shape():
    """Hidden 4096, intermediate 1536, 128 experts, top-8 (the cache workload's layer shape, K-blocks of several
    tiles per warp and a down phase split across warps), one token at two steps."""
    cfg = W.scaled(W.CONFIGS["cache_stream"], routing="normal", T=1)
    rows, tiles = mx_layer(cfg, 0)
    for step in range(2):
        check_fused(cfg, rows, tiles, 0, step, 1)
