"""Oracle pins: expert SwiGLU FFN, combine and the composed layer (CPU).

Pins: one expert with k = 1 reduces the layer to a dense SwiGLU FFN, checked
against a NumPy matmul on independently dequantised weights; combine weights
(1, 0) select one expert exactly; linearity of the combine; A4 mode reduces
to A16 on activations that are already on the NVFP4 grid.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def indep_deq(codes, scales, ts):
    lo, hi = codes & 0xF, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    s = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return E2M1[c] * np.repeat(s, 16, axis=1) * float(ts)


def make_expert(cfg, layer, e):
    return O.QuantizedExpert.from_fp32(*(W.weights_fp32(cfg, layer, e, p) for p in range(3)))


def bf16_values(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def test_single_expert_k1_is_dense_swiglu():
    cfg = W.scaled(W.CONFIGS["tiny"], E=1, k=1)
    ex = make_expert(cfg, 0, 0)
    Wg, Wu, Wd = (indep_deq(*q) for q in ex.q)
    x_bits = W.activations_bf16(cfg, 0, 0)
    logits = np.zeros((cfg.T, 1), np.float32)
    res = O.moe_layer(logits, x_bits, 1, lambda e: ex)
    x = bf16_values(x_bits)
    g = x @ Wg.T
    u = x @ Wu.T
    hraw = g / (1 + np.exp(-g)) * u
    h = res["h"]
    # h is hraw rounded to bf16: within half a bf16 ulp, i.e. at most 2^-8 relative
    assert np.all(np.abs(h - hraw) <= np.abs(hraw) * 2.0 ** -8 * (1 + 1e-9))
    assert np.array_equal(h, O.bf16_round_array(hraw))
    y_ref = h @ Wd.T
    assert np.allclose(res["y"], y_ref, rtol=1e-12, atol=1e-14)
    assert np.array_equal(res["w"], np.ones((cfg.T, 1)))
    # the output is y rounded to bf16
    assert np.array_equal(res["out"], O.bf16_round_array(res["y"]))
    assert np.allclose(res["out"], y_ref, rtol=2.0 ** -8, atol=0)


def test_combine_weights_one_zero_select_one_expert():
    cfg = W.CONFIGS["tiny"]
    experts = {e: make_expert(cfg, 0, e) for e in range(2)}
    x_bits = W.activations_bf16(cfg, 0, 0)
    logits = np.full((cfg.T, 2), -np.inf, np.float32)
    logits[:, 1] = 0.0       # expert 1 gets weight 1, expert 0 weight exp(-inf) = 0
    res = O.moe_layer(logits, x_bits, 2, lambda e: experts[e])
    assert np.array_equal(res["w"][:, 0], np.ones(cfg.T)) and np.array_equal(res["w"][:, 1], np.zeros(cfg.T))
    solo = O.moe_layer(np.zeros((cfg.T, 1), np.float32), x_bits, 1, lambda e: experts[1])
    assert np.array_equal(res["out"], solo["out"])


def test_combine_is_the_weighted_sum_in_slot_order():
    rng = np.random.default_rng(21)
    T, k, H = 3, 4, 32
    y = rng.normal(size=(T * k, H))
    inv = rng.permutation(T * k).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T)
    out, pre = O.combine(y, inv, w, T, k)
    ref = np.stack([sum(w[t, j] * y[inv[t * k + j]] for j in range(k)) for t in range(T)])
    assert np.array_equal(pre, ref)
    assert np.array_equal(out, O.bf16_round_array(ref))


def test_a4_mode_on_grid_exact_activations_matches_a16_through_gate_up():
    """x already on the unit-scale NVFP4 grid: A4 quantisation of x is exact, so g, u agree."""
    cfg = W.CONFIGS["tiny"]
    ex = make_expert(cfg, 0, 3)
    rng = np.random.default_rng(22)
    codes = rng.integers(0, 16, size=(cfg.T, cfg.H)).astype(np.uint8)
    codes[:, ::16] = 7
    scales = rng.integers(0x20, 0x40, size=(cfg.T, cfg.H // 16)).astype(np.uint8)
    x = indep_deq((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), scales, 1.0)
    h16, _ = O.expert_ffn(ex.Wg, ex.Wu, ex.Wd, x, O.MODE_A16)
    h4, y4 = O.expert_ffn(ex.Wg, ex.Wu, ex.Wd, x, O.MODE_A4)
    assert np.array_equal(h16, h4)
    # the down projection in A4 mode uses the quantised h
    hq_c, hq_s = O.quantize_act(h4.astype(np.float32))
    assert np.allclose(y4, indep_deq(hq_c, hq_s, 1.0) @ ex.Wd.T, rtol=1e-12, atol=1e-14)


def test_a4_mode_quantises_x_before_gate_up():
    """Off the grid: A4's h on x equals A16's h on x quantised per 16 with unit scale and decoded independently,
    and differs from A16's h on x itself."""
    cfg = W.CONFIGS["tiny"]
    ex = make_expert(cfg, 0, 5)
    x = W.bf16_bits_to_f32(W.activations_bf16(cfg, 0, 4)).astype(np.float64)
    xc, xs = O.quantize_act(x.astype(np.float32))
    xq = indep_deq(xc, xs, 1.0)
    h4, _ = O.expert_ffn(ex.Wg, ex.Wu, ex.Wd, x, O.MODE_A4)
    h16q, _ = O.expert_ffn(ex.Wg, ex.Wu, ex.Wd, xq, O.MODE_A16)
    h16, _ = O.expert_ffn(ex.Wg, ex.Wu, ex.Wd, x, O.MODE_A16)
    assert np.array_equal(h4, h16q)
    assert not np.array_equal(h4, h16)


def test_a4_vs_a16_deviation_is_small_on_gaussian_inputs():
    cfg = W.CONFIGS["tiny"]
    experts = {e: make_expert(cfg, 0, e) for e in range(cfg.E)}
    x_bits = W.activations_bf16(cfg, 0, 0)
    logits = W.router_logits(cfg, 0, 0)
    a16 = O.moe_layer(logits, x_bits, cfg.k, lambda e: experts[e], O.MODE_A16)
    a4 = O.moe_layer(logits, x_bits, cfg.k, lambda e: experts[e], O.MODE_A4)
    rel = np.linalg.norm(a4["out_pre"] - a16["out_pre"]) / np.linalg.norm(a16["out_pre"])
    assert 1e-3 < rel < 0.2   # NVFP4 activation noise: informational, not a parity bound


def test_layer_rows_subset_equals_full_layer_rows():
    cfg = W.scaled(W.CONFIGS["tiny"], T=6)
    experts = {e: make_expert(cfg, 0, e) for e in range(cfg.E)}
    x_bits = W.activations_bf16(cfg, 0, 0)
    logits = W.router_logits(cfg, 0, 0)
    full = O.moe_layer(logits, x_bits, cfg.k, lambda e: experts[e])
    part = O.moe_layer(logits, x_bits, cfg.k, lambda e: experts[e], rows=[1, 4])
    assert np.array_equal(part["out"], full["out"][[1, 4]])


def test_expert_ffn_rejects_bad_shapes():
    with pytest.raises(O.OracleError):
        O.expert_ffn(np.zeros((8, 20)), np.zeros((8, 20)), np.zeros((20, 8)), np.zeros((1, 20)))
