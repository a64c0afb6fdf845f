"""Oracle pins: NVFP4 block quantisation of weights and activations (CPU).

Pins: round trip of grid-exact tensors (quantise(dequantise(q)) == q), the
closed-form error bound, the tensor-scale definition, degenerate tensors, and
dequantisation checked against an independent decoder (the published E2M1
table and torch's float8_e4m3fn).
"""
import numpy as np
import pytest
import torch

import oracle as O

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def independent_dequant(codes, scales, ts):
    """Decoder written from the published tables, sharing nothing with the oracle."""
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    s = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return E2M1[c] * np.repeat(s, 16, axis=1) * float(ts)


def grid_tensor(rng, N, K, ts_exp=-12):
    """Random grid-exact weights: each block holds a +-6 code; one block has scale 448."""
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    codes[:, ::16] = rng.choice([7, 15], size=(N, K // 16))          # a +-6 in every block
    scales = rng.integers(0x08, 0x7F, size=(N, K // 16)).astype(np.uint8)  # normal E4M3, not NaN
    scales[0, 0] = 0x7E                                               # global amax = 6*448*ts
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    ts = 2.0 ** ts_exp
    return packed, scales, ts


@pytest.mark.parametrize("shape", [(4, 64), (32, 256), (7, 512)])
def test_weight_round_trip_of_grid_values(shape):
    rng = np.random.default_rng(shape[1])
    packed, scales, ts = grid_tensor(rng, *shape)
    w = independent_dequant(packed, scales, ts).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), independent_dequant(packed, scales, ts))  # exact in fp32
    c2, s2, ts2 = O.quantize_weight(w)
    assert ts2 == ts
    assert np.array_equal(s2, scales)
    # -0 codes come back canonical (+0); compare values
    assert np.array_equal(independent_dequant(c2, s2, ts2), independent_dequant(packed, scales, ts))


def test_oracle_dequantize_matches_independent_decoder():
    rng = np.random.default_rng(5)
    w = (rng.normal(0, 0.02, size=(64, 512))).astype(np.float32)
    c, s, ts = O.quantize_weight(w)
    assert np.array_equal(O.dequantize(c, s, ts), independent_dequant(c, s, ts))


def test_tensor_scale_definition():
    rng = np.random.default_rng(6)
    w = rng.normal(0, 0.02, size=(16, 256)).astype(np.float32)
    _, _, ts = O.quantize_weight(w)
    assert ts == float(np.float32(np.abs(w).max()) / np.float32(2688.0))


def test_weight_error_bound():
    """|w - deq| <= eff and eff <= (1 + 2^-4) amax_b / 6 for blocks with normal E4M3 scales."""
    rng = np.random.default_rng(7)
    w = rng.normal(0, 0.02, size=(128, 1024)).astype(np.float32)
    c, s, ts = O.quantize_weight(w)
    deq = O.dequantize(c, s, ts)
    sv = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    eff = sv * ts
    amax_b = np.abs(w.astype(np.float64)).reshape(128, 64, 16).max(axis=2)
    err = np.abs(w.astype(np.float64) - deq).reshape(128, 64, 16).max(axis=2)
    assert np.all(err <= eff * (1 + 1e-6))
    normal = s >= 0x08
    assert np.all(eff[normal] <= (1 + 2.0 ** -4) * amax_b[normal] / 6 * (1 + 1e-6))
    # relative quantisation noise of NVFP4 on Gaussian data is a few percent
    rel = np.linalg.norm(w - deq) / np.linalg.norm(w)
    assert 0.02 < rel < 0.15


def test_degenerate_tensors():
    z = np.zeros((2, 32), np.float32)
    c, s, ts = O.quantize_weight(z)
    assert ts == 1.0 and not c.any() and not s.any()
    tiny = np.full((1, 16), 1e-45, np.float32)        # amax/2688 underflows: unit tensor scale
    c, s, ts = O.quantize_weight(tiny)
    assert ts == 1.0 and not c.any()
    with pytest.raises(O.OracleError):
        O.quantize_weight(np.full((1, 16), np.nan, np.float32))
    with pytest.raises(O.OracleError):
        O.quantize_weight(np.zeros((1, 8), np.float32))   # K not a multiple of 16


def test_negative_zero_is_canonical():
    w = np.zeros((1, 16), np.float32)
    w[0, 0] = 1.0
    w[0, 1] = -1e-3      # rounds to zero
    c, s, ts = O.quantize_weight(w)
    assert (c[0, 0] >> 4) == 0


def test_activation_quantizer_round_trip_and_bound():
    rng = np.random.default_rng(8)
    # grid-exact activations with unit tensor scale
    codes = rng.integers(0, 16, size=(3, 256)).astype(np.uint8)
    codes[:, ::16] = 7
    scales = rng.integers(0x20, 0x60, size=(3, 16)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    x = independent_dequant(packed, scales, 1.0).astype(np.float32)
    c2, s2 = O.quantize_act(x)
    assert np.array_equal(s2, scales)
    assert np.array_equal(independent_dequant(c2, s2, 1.0), x.astype(np.float64))
    # bound on Gaussian activations
    xa = rng.normal(0, 1, size=(8, 512)).astype(np.float32)
    c, s = O.quantize_act(xa)
    d = independent_dequant(c, s, 1.0)
    sv = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    err = np.abs(xa - d).reshape(8, 32, 16).max(axis=2)
    assert np.all(err <= sv)


def test_weight_and_activation_quantizers_agree_at_unit_scale():
    """The activation quantiser is the weight quantiser with tensor scale fixed at 1."""
    rng = np.random.default_rng(9)
    x = rng.normal(0, 1, size=(4, 64)).astype(np.float32)
    x[0, 0] = 2688.0   # forces amax/2688 == 1 so the weight path's tensor scale is exactly 1
    cw, sw, ts = O.quantize_weight(x)
    assert ts == 1.0
    ca, sa = O.quantize_act(x)
    assert np.array_equal(cw, ca) and np.array_equal(sw, sa)
