"""Failure detection on the device, made to happen without faulting anything.

A bounded device wait runs out when it waits for h words of a tag no CTA writes (the library's test hook, with a
1 ms limit): the kernel must return on its own, report FT_DEVERR_TIMEOUT through the device error word, and leave the
workspace usable, so that the next call is bit-equal to a clean one.  The same for the tensor-core prefill, whose
gate/up MMA issuer is made to wait on a barrier nothing completes: the next call matches a clean one (its fp32
reductions have no fixed order, so within the layer tolerance rather than bit for bit).  The workspace's 64-bit call counter is also
started just before its tag wraps (2^32 - 1 tags, never 0): the calls across the wrap must equal a clean call.
"""
import time

import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_layer_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

if torch.cuda.is_available():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import FusedDecodeLayer, LayerWeights, PrefillLayer


def layer_and_inputs(cfg):
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_DECODE_TILES)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, 0, e, p), sigma=cfg.w_sigma)
    logits = torch.from_numpy(W.router_logits(cfg, 0, 0)).to(DEV)
    x = torch.from_numpy(W.activations_bf16(cfg, 0, 0).view(np.int16)).view(torch.bfloat16).to(DEV)
    return lw, logits, x


@pytest.mark.parametrize("shape", ["decode_35b", "hidden_4096"])
def test_expired_wait_reports_timeout_and_the_next_call_is_exact(shape):
    """On the 35B layer shape and on hidden 4096 / intermediate 1536 (several tiles per warp, the down phase
    split across warps)."""
    cfg = (W.CONFIGS["decode_35b"] if shape == "decode_35b" else
           W.scaled(W.CONFIGS["cache_stream"], routing="normal", T=1))
    lw, logits, x = layer_and_inputs(cfg)
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    clean = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod(lw, logits, x, clean)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    out = torch.empty_like(clean)
    Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_DECODE_H, 1_000_000)  # 1 ms
    try:
        t0 = time.perf_counter()
        mod(lw, logits, x, out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_NONE)
    assert Q.ft_device_status() & Q.FT_DEVERR_TIMEOUT
    assert elapsed < 0.5, elapsed   # each wait gave up after ~1 ms, far below the default 2 s
    again = torch.empty_like(clean)
    mod(lw, logits, x, again)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    assert torch.equal(again, clean)


def test_prefill_expired_wait_reports_timeout_and_the_next_call_is_clean():
    """The 35B layer shape with 512 prompt tokens: the gate/up GEMM's MMA issuer gives up after 1 ms, every role of
    the kernel winds down (no trap, TMEM freed), the down GEMM and the output conversion still run, and the next
    call without the hook equals a clean call."""
    cfg = W.scaled(W.CONFIGS["prefill_35b"], T=512)
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_UMMA_TILES)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, 0, e, p), sigma=cfg.w_sigma)
    logits = torch.from_numpy(W.router_logits(cfg, 0, 0)).to(DEV)
    x = torch.from_numpy(W.activations_bf16(cfg, 0, 0).view(np.int16)).view(torch.bfloat16).to(DEV)
    mod = PrefillLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    clean = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    mod(lw, logits, x, clean)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    out = torch.empty_like(clean)
    Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_PREFILL_TOKEN, 1_000_000)  # 1 ms
    try:
        t0 = time.perf_counter()
        mod(lw, logits, x, out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_NONE)
    assert Q.ft_device_status() & Q.FT_DEVERR_TIMEOUT
    assert elapsed < 0.5, elapsed
    again = torch.empty_like(clean)
    mod(lw, logits, x, again)
    torch.cuda.synchronize()
    assert Q.ft_device_status() == 0
    assert_layer_close(again.float().cpu().numpy(), clean.float().cpu().numpy().astype(np.float64), "prefill after expiry")


def test_wait_hook_rejects_bad_arguments():
    with pytest.raises(Q.FtError):
        Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_DECODE_H, 0)
    with pytest.raises(Q.FtError):
        Q.ft_debug_inject_wait_expiry(Q.FT_WAIT_SITE_DECODE_H, 3_000_000_000)
    with pytest.raises(Q.FtError):
        Q.ft_debug_inject_wait_expiry(99, 1000)


def test_call_counter_wrap_keeps_the_hand_off_exact():
    """Start the 64-bit counter so that this call's h tag is the last one (2^32 - 1) and the next call's wraps to 1;
    both equal a call on a fresh workspace."""
    cfg = W.CONFIGS["decode_35b"]
    lw, logits, x = layer_and_inputs(cfg)
    fresh = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    clean = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    fresh(lw, logits, x, clean)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    mod = FusedDecodeLayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.T, DEV)
    start = (2 ** 32 - 2) * G   # call number 2^32 - 2 -> tag 2^32 - 1; the next call -> tag 1
    mod.ws[:8].copy_(torch.tensor([start], dtype=torch.int64).view(torch.uint8).to(DEV))
    for _ in range(3):
        out = torch.empty_like(clean)
        mod(lw, logits, x, out)
        torch.cuda.synchronize()
        assert Q.ft_device_status() == 0
        assert torch.equal(out, clean)
    count = int(mod.ws[:8].cpu().view(torch.int64).item())
    assert count == start + 3 * G
