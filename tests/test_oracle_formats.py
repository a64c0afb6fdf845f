"""Oracle pins: NVFP4 element and scale formats, their encoders, bf16 rounding (CPU).

Pinned against the published format tables (golden fixtures), against an
independent library (torch's float8_e4m3fn and bfloat16 conversions), and by
brute force over the grid.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_rows

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table_matches_published_values():
    rows = golden_rows("e2m1_values.txt")
    assert len(rows) == 16
    for row in rows:
        code, val = row.split()
        got = O.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_all_codes_match_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for code in range(256):
        got = O.e4m3_value(code)
        if np.isnan(ref[code]):
            assert np.isnan(got), code
        else:
            assert got == ref[code], code


def test_e4m3_landmarks():
    for row in golden_rows("e4m3_landmarks.txt"):
        h, v = row.split()
        got = O.e4m3_value(int(h, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v)


def test_exhaustive_code_times_scale_table():
    """All 16 x 254 (code, non-NaN scale) products are exact and equal the closed form."""
    for s in range(256):
        if (s & 0x7F) == 0x7F:
            continue
        sv = O.e4m3_value(s)
        for c in range(16):
            prod = O.e2m1_value(c) * sv
            e = (s >> 3) & 15
            m = s & 7
            mag = (m * 2.0 ** -9) if e == 0 else 2.0 ** (e - 7) * (1 + m / 8)
            ce, cm = (c >> 1) & 3, c & 1
            cmag = 0.5 * cm if ce == 0 else 2.0 ** (ce - 1) * (1 + cm / 2)
            sign = (-1) ** (((s >> 7) ^ (c >> 3)) & 1)
            assert abs(prod) == cmag * mag
            if prod != 0:
                assert math.copysign(1.0, prod) == sign


def test_e2m1_ties_and_saturation():
    for row in golden_rows("e2m1_ties.txt"):
        v, code = row.split()
        assert O.e2m1_encode(float(v)) == int(code), v


def _f32(x):
    return struct.unpack("f", struct.pack("f", x))[0]


def test_e2m1_encode_is_nearest_on_random_inputs():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-7, 7, 20000), rng.normal(0, 2, 20000)]).astype(np.float32)
    for v in vals:
        c = O.e2m1_encode(float(v))
        got = O.e2m1_value(c)
        target = min(abs(float(v)), 6.0)
        best = min(abs(g - target) for g in E2M1_GRID)
        assert abs(abs(got) - target) == best
        if got != 0:
            assert (got < 0) == (v < 0)
        else:
            assert c == 0


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(2)
    vals = [O.e4m3_value(c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    samples = np.concatenate([
        np.exp(rng.uniform(np.log(1e-4), np.log(448.0), 50000)),
        np.array(vals + mids),
        rng.uniform(0, 0.02, 5000),
    ]).astype(np.float32)
    ref = torch.from_numpy(samples).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in samples], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    for v in (448.0, 449.0, 464.0, 470.0, 1e6, float("inf")):
        assert O.e4m3_encode(v) == 0x7E


def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(3)
    f = np.concatenate([
        rng.normal(0, 1, 20000),
        rng.normal(0, 1e-38, 2000),           # bf16 subnormals
        np.exp(rng.uniform(-80, 80, 5000)),
    ]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([O.bf16_round(float(v)) for v in f])
    assert np.array_equal(got, ref)


def test_bf16_round_ties_and_overflow():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16_round(one + ulp / 2) == one            # tie -> even (1.0)
    assert O.bf16_round(one + 3 * ulp / 2) == one + 2 * ulp  # tie -> even
    assert O.bf16_round(one + ulp / 2 + 2.0 ** -40) == one + ulp  # just above the tie (fp64-only input)
    r = O.bf16_round(3.0e38)
    assert math.isfinite(r) and abs(r - 3.0e38) <= 2.0 ** (127 - 7) / 2
    assert O.bf16_round(2.0 ** 128 * (1 - 2.0 ** -9)) == float("inf")
    assert O.bf16_round(-(2.0 ** 127) * (2 - 2.0 ** -7)) == -(2.0 ** 127) * (2 - 2.0 ** -7)
    assert O.bf16_round(2.0 ** -134) == 0.0      # below half the smallest subnormal: tie to even (0)
    assert O.bf16_round(2.0 ** -134 * 1.5) == 2.0 ** -133


@pytest.mark.parametrize("v", [0.0, -0.0, 1.0, -2.5, 1e-30])
def test_bf16_round_fixed_points(v):
    r = O.bf16_round(v)
    assert O.bf16_round(r) == r
