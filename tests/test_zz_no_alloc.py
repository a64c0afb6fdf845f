"""The fused decode layer step without a caller workspace (ft_moe_layer_decode_noalloc).

Some callers cannot allocate device memory: plugins handed only their input and
output buffers, applications whose own pool allocator owns the device, decode
loops that must not take the allocator's locks.  The no-allocation entry point
uses a scratch array built into the library instead of a workspace.  Here it is
called through the C ABI and its output is compared with ft_moe_layer_decode's
(the entry point that takes a workspace) on the same inputs, for two calls in a
row, within the layer tolerance the parity tests use.  The file is collected
last so that a stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_layer_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(cfg, layer, step):
    logits = torch.from_numpy(W.router_logits(cfg, layer, step)).to(DEV)
    x = torch.from_numpy(W.activations_bf16(cfg, layer, step).view(np.int16)).view(torch.bfloat16).to(DEV)
    return logits, x


@pytest.mark.parametrize("cfg_name,layer", [("tiny", 0), ("decode_35b", 3)])
def test_no_alloc_matches_workspace_entry_point_on_two_calls(cfg_name, layer):
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights

    cfg = W.CONFIGS[cfg_name]
    lw = LayerWeights(cfg.E, cfg.H, cfg.I, DEV, layout=Q.FT_LAYOUT_DECODE_TILES)
    lw.fill_synthetic(lambda e, p: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
    T, k = cfg.T, cfg.k
    ws = torch.zeros(Q.ft_moe_layer_decode_workspace_size(T, k, cfg.H, cfg.I), dtype=torch.uint8, device=DEV)
    for step in (0, 1):  # two calls in a row: the second must not see the first's leftovers
        logits, x = _inputs(cfg, layer, step)
        ref_out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
        ref_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        ref_w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        Q.ft_moe_layer_decode(lw, logits, x, k, ref_out, ws, ids=ref_ids, w=ref_w)
        out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
        ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        Q.ft_moe_layer_decode_noalloc(lw, logits, x, k, out, ids=ids, w=w)
        torch.cuda.synchronize()
        assert Q.ft_device_status() == 0
        assert torch.equal(ids, ref_ids)
        assert torch.allclose(w, ref_w, rtol=1e-5, atol=1e-7)
        assert_layer_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), f"{cfg_name} call {step}")


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights

    # T*k*I = 16 * 32 * 1024 = 524288 > 262144: refused before anything is enqueued
    lw = LayerWeights(64, 256, 1024, DEV, layout=Q.FT_LAYOUT_DECODE_TILES)
    logits = torch.zeros((16, 64), dtype=torch.float32, device=DEV)
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((16, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(Q.FtError) as ei:
        Q.ft_moe_layer_decode_noalloc(lw, logits, x, 32, out)
    assert ei.value.status == Q.FT_ERR_INVALID_ARG
    assert "scratch" in str(ei.value)
