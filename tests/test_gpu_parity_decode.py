"""GPU parity of the decode layer step (route -> permute -> NVFP4 expert FFN -> combine).

The device quantises fp32 weights drawn by its own generator (or uploaded from
the host generator for the tiny layer); the oracle quantises the host
generator's weights itself.  ids, offsets, perm and inv are compared bit for
bit; outputs within relative L2 5e-3 and max |err| 2e-2 * RMS.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from helpers import assert_layer_close, oracle_expert, parity_metrics

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights, MoEDecodeLayer
DEV = "cuda:0"


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


def device_weights_from_host(cfg, layer, experts=None):
    """Upload the host generator's fp32 weights and quantise them on the device."""
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV)
    for e in (range(cfg.E) if experts is None else experts):
        for p in range(3):
            lw.quantize_projection(e, p, to_dev(W.weights_fp32(cfg, layer, e, p)))
    return lw


def device_weights_generated(cfg, layer):
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
    return lw


def run_layer(cfg, lw, layer, step, T=None, want_y=False):
    T = cfg.T if T is None else T
    logits = W.router_logits(cfg, layer, step, T=T)
    x_bits = W.activations_bf16(cfg, layer, step, T=T)
    mod = MoEDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, T, DEV)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T * cfg.k, cfg.H), dtype=torch.float32, device=DEV) if want_y else None
    mod(lw, to_dev(logits), to_dev(x_bits.view(np.int16), torch.bfloat16), out, y=y)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    return logits, x_bits, mod, out, y


def oracle_layer(cfg, layer, logits, x_bits, rows=None):
    return O.moe_layer(logits, x_bits, cfg.k, lambda e: oracle_expert(cfg, layer, e), O.MODE_A16, rows=rows)


def check_routing(mod, ref):
    assert np.array_equal(mod.ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(mod.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(mod.perm.cpu().numpy(), ref["perm"])
    assert np.array_equal(mod.inv.cpu().numpy(), ref["inv"])
    w = mod.w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w - ref["w"]) <= 1e-5 * ref["w"] + 1e-7)


def test_tiny_layer_every_output():
    cfg = W.CONFIGS["tiny"]
    lw = device_weights_from_host(cfg, 0)
    logits, x_bits, mod, out, y = run_layer(cfg, lw, 0, 0, want_y=True)
    ref = oracle_layer(cfg, 0, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "tiny out")
    # every per-row expert output as well (y is not rounded)
    assert_layer_close(y.cpu().numpy(), ref["y"], "tiny y")


def test_device_weights_equal_oracle_weights_on_samples():
    """Device generator + device quantiser reproduce the oracle's NVFP4 bytes (sampled experts)."""
    cfg = W.CONFIGS["decode_35b"]
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV)
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


@pytest.mark.parametrize("layer,step", [(0, 0), (7, 3), (47, 255)])
def test_decode_35b_layer(layer, step):
    cfg = W.CONFIGS["decode_35b"]
    lw = device_weights_generated(cfg, layer)
    logits, x_bits, mod, out, _ = run_layer(cfg, lw, layer, step)
    ref = oracle_layer(cfg, layer, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], f"35B layer {layer} step {step}")


def test_decode_753b_batch1_layer():
    cfg = W.CONFIGS["decode_753b_b1"]
    lw = device_weights_generated(cfg, 3)
    logits, x_bits, mod, out, _ = run_layer(cfg, lw, 3, 11)
    ref = oracle_layer(cfg, 3, logits, x_bits)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy(), ref["out"], "753B b1")


def test_decode_753b_batch16_sampled_tokens():
    cfg = W.CONFIGS["decode_753b_b16"]
    lw = device_weights_generated(cfg, 1)
    logits, x_bits, mod, out, _ = run_layer(cfg, lw, 1, 2)
    rows = [0, 9]
    ref = oracle_layer(cfg, 1, logits, x_bits, rows=rows)
    check_routing(mod, ref)
    assert_layer_close(out.float().cpu().numpy()[rows], ref["out"], "753B b16 sampled")


def test_ragged_token_counts_and_single_expert_segments():
    """T = 13 tokens over 8 experts with k = 2: segments of uneven length, several token chunks."""
    cfg = W.scaled(W.CONFIGS["tiny"], T=13)
    lw = device_weights_from_host(cfg, 0)
    logits, x_bits, mod, out, _ = run_layer(cfg, lw, 0, 4)
    ref = oracle_layer(cfg, 0, logits, x_bits)
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


def test_slot_table_indirection():
    """Weights addressed through expert_to_slot give the same output as direct addressing."""
    cfg = W.CONFIGS["tiny"]
    direct = device_weights_from_host(cfg, 0)
    slots = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, n_weights=cfg.E)
    perm = np.random.default_rng(3).permutation(cfg.E)
    for e in range(cfg.E):   # expert e lives in slot perm[e]
        s = int(perm[e])
        for a, b in ((slots.gu_codes, direct.gu_codes), (slots.gu_scales, direct.gu_scales),
                     (slots.d_codes, direct.d_codes), (slots.d_scales, direct.d_scales),
                     (slots.tscale, direct.tscale)):
            a[s].copy_(b[e])
    slots.expert_to_slot = to_dev(perm.astype(np.int32))
    _, _, _, out_a, _ = run_layer(cfg, direct, 0, 0)
    _, _, _, out_b, _ = run_layer(cfg, slots, 0, 0)
    assert torch.equal(out_a, out_b)
