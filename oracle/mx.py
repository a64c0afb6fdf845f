"""Oracle of the MX expert-weight formats (MXFP4 and MXFP8), plain numpy in fp64.

TEST INFRASTRUCTURE ONLY: the tests use it; the CUDA library never does.

The page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier MoE 拉回本地"
(section 局限) names MXFP4 and FP8 beside NVFP4 as weight formats, without
their bit layout.  The plainest reading is the published OCP Microscaling
(MX) v1.0 definition, restated here:

* a block is 32 consecutive elements along the reduction dimension, sharing
  one UE8M0 scale byte s: the power of two 2^(s - 127) (s = 255 is NaN);
* MXFP4 elements are E2M1 (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), MXFP8
  elements E4M3 (largest finite 448);
* quantising a block: X = floor(log2(max |v|)) - emax, where emax is the
  exponent of the element format's largest normal (2 for E2M1, 8 for E4M3),
  clamped to the scale's range [-127, 127]; each element is v / 2^X rounded
  to the nearest element value, ties to the even code, saturating at the
  largest finite value;
* an all-zero block takes scale byte 0 and zero codes; a negative value that
  rounds to zero is stored as +0 (as the NVFP4 encoder here does).

There is no tensor scale.  Codes: E2M1 two per byte, the even element in the
low nibble; E4M3 one per byte with the sign in bit 7.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32

# magnitude of each non-negative code, in code order (code order is value order)
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_EMAX = 2


def _e4m3_magnitudes() -> np.ndarray:
    mags = []
    for c in range(0x7F):  # 0x7F is NaN
        e, m = c >> 3, c & 7
        mags.append(m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8))
    return np.array(mags)


E4M3_MAG = _e4m3_magnitudes()   # codes 0 .. 0x7E, largest 448
E4M3_EMAX = 8

FORMATS = {"mxfp4": (E2M1_MAG, E2M1_EMAX, 3), "mxfp8": (E4M3_MAG, E4M3_EMAX, 7)}  # grid, emax, sign bit


def ue8m0_value(s: int) -> float:
    """The scale a UE8M0 byte stands for: 2^(s - 127); NaN for 255."""
    return float("nan") if s == 255 else float(np.ldexp(1.0, s - 127))


def round_to_grid(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Code of the grid value nearest to each magnitude a >= 0 (fp64), ties to the even code, saturating at the
    last grid value."""
    a = np.asarray(a, np.float64)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo, d_hi = np.abs(a - grid[lo]), np.abs(grid[hi] - a)
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    return np.where(a >= grid[-1], len(grid) - 1, code)


def block_exponent(amax: np.ndarray, emax: int) -> np.ndarray:
    """X = floor(log2(amax)) - emax, clamped to [-127, 127]; -127 where amax is 0."""
    amax = np.asarray(amax, np.float64)
    _, e = np.frexp(amax)            # amax = f * 2^e with f in [0.5, 1): floor(log2(amax)) = e - 1
    x = np.where(amax > 0, e - 1 - emax, -127)
    return np.clip(x, -127, 127).astype(np.int64)


def quantize(w: np.ndarray, fmt: str):
    """fp32 [N, K] (K a multiple of 32) -> (codes, scales u8 [N, K/32]).

    codes: u8 [N, K/2] for mxfp4, u8 [N, K] for mxfp8."""
    grid, emax, sign_bit = FORMATS[fmt]
    w = np.asarray(w, np.float32).astype(np.float64)
    N, K = w.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = w.reshape(N, K // BLOCK, BLOCK)
    x = block_exponent(np.abs(blocks).max(axis=2), emax)            # [N, K/32]
    a = np.abs(blocks) / np.ldexp(1.0, x)[:, :, None]              # exact: division by a power of two
    mag = round_to_grid(a, grid)
    neg = (blocks < 0) & (mag > 0)                                  # -0 is stored as +0
    code = (mag | (neg.astype(np.int64) << sign_bit)).reshape(N, K).astype(np.uint8)
    scales = (x + 127).astype(np.uint8)
    if fmt == "mxfp4":
        code = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return code, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, fmt: str) -> np.ndarray:
    """fp64 [N, K] from quantize()'s output."""
    grid, _, sign_bit = FORMATS[fmt]
    codes = np.asarray(codes, np.uint8)
    if fmt == "mxfp4":
        c = np.empty((codes.shape[0], codes.shape[1] * 2), np.int64)
        c[:, 0::2], c[:, 1::2] = codes & 0xF, codes >> 4
    else:
        c = codes.astype(np.int64)
    mag_code = c & ((1 << sign_bit) - 1)
    if fmt == "mxfp8" and np.any(mag_code == 0x7F):
        raise ValueError("E4M3 NaN code")
    val = grid[mag_code] * np.where(c >> sign_bit, -1.0, 1.0)
    s = np.asarray(scales, np.int64)
    if np.any(s == 255):
        raise ValueError("UE8M0 NaN scale")
    return val * np.repeat(np.ldexp(1.0, s - 127), BLOCK, axis=1)
