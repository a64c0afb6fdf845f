"""Oracle pins: the MX weight formats (MXFP4 = E2M1 elements, MXFP8 = E4M3 elements, one UE8M0 scale per 32).

Pins: the scale byte's closed form over all 256 values, the element grids against the hand-written E2M1 table and
the published E4M3 landmarks, the block exponent on worked amax values, the E2M1 tie table (golden fixture),
rounding against a brute-force nearest search, saturation, round trips of values on the grid, and the error bound
that follows from the grid spacing.
"""
import math

import numpy as np
import pytest

from conftest import golden_rows
from oracle import mx


def test_ue8m0_is_a_power_of_two_per_byte():
    for s in range(255):
        assert mx.ue8m0_value(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(mx.ue8m0_value(255))
    assert mx.ue8m0_value(127) == 1.0 and mx.ue8m0_value(0) == 2.0 ** -127 and mx.ue8m0_value(254) == 2.0 ** 127


def test_element_grids():
    assert list(mx.E2M1_MAG) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    g = mx.E4M3_MAG
    assert len(g) == 127 and np.all(np.diff(g) > 0)
    assert g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6 and g[0x7E] == 448.0   # min subnormal, min normal, max
    assert g[0x38] == 1.0 and g[0x3C] == 1.5


@pytest.mark.parametrize("fmt,emax,top", [("mxfp4", 2, 6.0), ("mxfp8", 8, 448.0)])
def test_block_exponent_on_worked_values(fmt, emax, top):
    # amax in [2^(emax+s), 2^(emax+s+1)) gives X = s: the block's largest value lands in [2^emax, 2^(emax+1))
    for s in (-20, -3, 0, 5, 40):
        for amax in (2.0 ** (emax + s), top * 2.0 ** s, 2.0 ** (emax + s + 1) * (1 - 2 ** -20)):
            assert mx.block_exponent(np.array(amax), emax) == s, (amax, s)
        assert mx.block_exponent(np.array(2.0 ** (emax + s + 1)), emax) == s + 1
    assert mx.block_exponent(np.array(0.0), emax) == -127
    assert mx.block_exponent(np.array(2.0 ** -140), emax) == -127       # clamped to the scale's range
    assert mx.block_exponent(np.array(2.0 ** 200), emax) == 127


def test_e2m1_ties_go_to_the_even_code():
    """The tie table's inputs as elements of a block whose scale is 1 (a 6.0 fixes X = 0): same codes, sign in
    bit 3, negatives that round to zero stored as +0."""
    for row in golden_rows("e2m1_ties.txt"):
        v, want = row.split()[:2]
        w = np.zeros((1, 32), np.float32)
        w[0, 0], w[0, 1] = 6.0, float(v)
        codes, scales = mx.quantize(w, "mxfp4")
        if abs(float(v)) < 8:               # a larger input raises the block's scale; its code still saturates
            assert scales[0, 0] == 127, row
        assert (codes[0, 0] >> 4) == int(want), row


@pytest.mark.parametrize("grid", [mx.E2M1_MAG, mx.E4M3_MAG])
def test_rounding_equals_brute_force_nearest(grid):
    rng = np.random.default_rng(3)
    top = grid[-1]
    mids = (grid[1:] + grid[:-1]) / 2
    a = np.concatenate([rng.uniform(0, top * 1.2, 4000), mids, grid, [top * 1.1, top * 2]])
    got = mx.round_to_grid(a, grid)
    for ai, gi in zip(a, got):
        d = np.abs(grid - min(ai, top))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert gi == want, ai


def test_saturation_and_zero_blocks():
    w = np.zeros((1, 64), np.float32)
    w[0, 0], w[0, 1] = 7.0, -7.9           # amax 7.9 -> X = 0; both beyond 6 saturate
    codes, scales = mx.quantize(w, "mxfp4")
    d = mx.dequantize(codes, scales, "mxfp4")
    assert scales[0, 0] == 127 and d[0, 0] == 6.0 and d[0, 1] == -6.0
    assert scales[0, 1] == 0 and np.all(d[0, 32:] == 0) and np.all(codes[0, 16:] == 0)
    w8 = np.zeros((1, 32), np.float32)
    w8[0, 0], w8[0, 1] = 500.0, -1e-30     # X = 0: 500 saturates to 448; a tiny negative becomes +0
    c8, s8 = mx.quantize(w8, "mxfp8")
    d8 = mx.dequantize(c8, s8, "mxfp8")
    assert s8[0, 0] == 127 and d8[0, 0] == 448.0 and c8[0, 1] == 0


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_values_on_the_grid_round_trip(fmt):
    grid, emax, sign_bit = mx.FORMATS[fmt]
    rng = np.random.default_rng(11)
    N, K = 16, 256
    mag = rng.integers(0, len(grid), size=(N, K))
    mag[:, ::mx.BLOCK] = len(grid) - 1     # each block holds the top value, so amax fixes X = s
    sign = rng.integers(0, 2, size=(N, K)) * (mag > 0)
    s = rng.integers(-30, 30, size=(N, K // mx.BLOCK))
    w = (grid[mag] * np.where(sign, -1, 1) * np.repeat(np.ldexp(1.0, s), mx.BLOCK, axis=1)).astype(np.float32)
    codes, scales = mx.quantize(w, fmt)
    assert np.array_equal(scales.astype(np.int64), s + 127)
    assert np.array_equal(mx.dequantize(codes, scales, fmt), w.astype(np.float64))
    assert np.array_equal(mx.quantize(mx.dequantize(codes, scales, fmt), fmt)[0], codes)


@pytest.mark.parametrize("fmt,half_step", [("mxfp4", 2.0), ("mxfp8", 64.0)])
def test_error_bound_from_the_grid(fmt, half_step):
    """Within a block, v / 2^X lies below 2^(emax+1); the grid's largest gap below that (rounding) or the distance
    past the largest value (saturation) bounds the error: 2 for E2M1 (6 .. 8), 64 for E4M3 (448 .. 512)."""
    rng = np.random.default_rng(5)
    N, K = 64, 1024
    mag = np.exp(rng.uniform(-10, 10, size=(N, K // mx.BLOCK, 1)))
    w = (rng.standard_normal((N, K // mx.BLOCK, mx.BLOCK)) * mag).reshape(N, K).astype(np.float32)
    codes, scales = mx.quantize(w, fmt)
    d = mx.dequantize(codes, scales, fmt)
    step = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), mx.BLOCK, axis=1)
    assert np.all(np.abs(d - w.astype(np.float64)) <= half_step * step)
    assert np.all(np.sign(d) * np.sign(w) >= 0)   # never the wrong sign


def test_byte_layout():
    """MXFP4: element 2j in the low nibble of byte j, sign in bit 3; MXFP8: one E4M3 byte per element, sign in
    bit 7 (E4M3 1.0 is 0x38); the scale byte is the exponent + 127."""
    w = np.zeros((1, 32), np.float32)
    w[0, :4] = [0.5, 1.0, -6.0, 3.0]       # amax 6 -> X = 0 (scale byte 127)
    codes, scales = mx.quantize(w, "mxfp4")
    assert scales.tolist() == [[127]] and codes[0, 0] == 0x21 and codes[0, 1] == 0x5F
    w8 = np.zeros((1, 32), np.float32)
    w8[0, :3] = [1.0, -1.0, 256.0]         # amax 256 -> X = 0
    c8, s8 = mx.quantize(w8, "mxfp8")
    assert s8.tolist() == [[127]] and c8[0, :3].tolist() == [0x38, 0xB8, 0x78]


def test_e4m3_holds_exactly_the_powers_of_two_the_mxfp4_reencoding_uses():
    """The MXFP4 tensor-core packing writes each block scale 2^(s - s0) as an E4M3 byte: (d + 7) << 3 for
    d = -6 .. 8 and 1 << (d + 9) for the subnormals d = -9 .. -7.  Those bytes decode (the oracle's E4M3 table) to
    exactly 2^d, and no E4M3 value is a power of two outside -9 .. 8: the 18 exponents s0 - 9 .. s0 + 8, a span
    of 17 octaves."""
    import oracle as O
    for d in range(-9, 9):
        b = (d + 7) << 3 if d >= -6 else 1 << (d + 9)
        assert O.e4m3_value(b) == 2.0 ** d, d
    vals = [O.e4m3_value(b) for b in range(0x7F)]            # every finite non-negative E4M3 value
    pow2 = sorted({math.log2(v) for v in vals if v > 0 and math.log2(v).is_integer()})
    assert pow2 == list(range(-9, 9))
