"""Device-side containers for one MoE layer: NVFP4 expert weights in the
layout the kernels read, and the ABI-level decode step (route -> permute ->
expert FFN -> combine) with its buffers allocated once.
"""
from __future__ import annotations

import ctypes

import torch

from . import (ft_gen_normal_f32, ft_moe_layer_weights, ft_moe_permute_workspace_size, ft_moe_decode_workspace_size,
               ft_nvfp4_quantize_weight, ft_moe_route, ft_moe_permute, ft_moe_expert_ffn_nvfp4_decode, lib, _check,
               _s)

PROJ_GATE, PROJ_UP, PROJ_DOWN = 0, 1, 2


class LayerWeights:
    """NVFP4 weights of one layer (E experts, or n_weights cache slots).

    gu_codes  [n, 2I, H/2]  rows 2i / 2i+1 = gate row i / up row i
    gu_scales [n, 2I, H/16]
    d_codes   [n, H, I/2]
    d_scales  [n, H, I/16]
    tscale    [n, 4] fp32   (gate, up, down, pad)
    """

    def __init__(self, E: int, H: int, I: int, device, n_weights: int | None = None):
        self.E, self.H, self.I = E, H, I
        self.n = E if n_weights is None else n_weights
        u8 = torch.uint8
        self.gu_codes = torch.empty((self.n, 2 * I, H // 2), dtype=u8, device=device)
        self.gu_scales = torch.empty((self.n, 2 * I, H // 16), dtype=u8, device=device)
        self.d_codes = torch.empty((self.n, H, I // 2), dtype=u8, device=device)
        self.d_scales = torch.empty((self.n, H, I // 16), dtype=u8, device=device)
        self.tscale = torch.zeros((self.n, 4), dtype=torch.float32, device=device)
        self.expert_to_slot: torch.Tensor | None = None
        self._qws = torch.empty(256, dtype=u8, device=device)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.gu_codes, self.gu_scales, self.d_codes, self.d_scales))

    def desc(self) -> ft_moe_layer_weights:
        d = ft_moe_layer_weights()
        d.E, d.H, d.I, d.n_weights = self.E, self.H, self.I, self.n
        d.gu_codes, d.gu_codes_stride = self.gu_codes.data_ptr(), self.gu_codes.stride(0)
        d.gu_scales, d.gu_scales_stride = self.gu_scales.data_ptr(), self.gu_scales.stride(0)
        d.d_codes, d.d_codes_stride = self.d_codes.data_ptr(), self.d_codes.stride(0)
        d.d_scales, d.d_scales_stride = self.d_scales.data_ptr(), self.d_scales.stride(0)
        d.tscale, d.tscale_stride = self.tscale.data_ptr(), self.tscale.stride(0)
        d.expert_to_slot = None if self.expert_to_slot is None else self.expert_to_slot.data_ptr()
        return d

    def quantize_projection(self, wi: int, proj: int, w: torch.Tensor, stream=None) -> None:
        """Quantise an fp32 [N, K] matrix into weight index wi (proj 0 gate, 1 up, 2 down)."""
        H, I = self.H, self.I
        ts = self.tscale[wi, proj:proj + 1]
        if proj in (PROJ_GATE, PROJ_UP):
            assert tuple(w.shape) == (I, H)
            codes = self.gu_codes[wi].data_ptr() + proj * (H // 2)
            scales = self.gu_scales[wi].data_ptr() + proj * (H // 16)
            ft_nvfp4_quantize_weight(w, codes, scales, ts, codes_ld=H, scales_ld=H // 8, ws=self._qws, stream=stream)
        else:
            assert tuple(w.shape) == (H, I)
            ft_nvfp4_quantize_weight(w, self.d_codes[wi], self.d_scales[wi], ts, ws=self._qws, stream=stream)

    def fill_synthetic(self, stream_of, seed: int = 0, sigma: float = 0.02, experts=None, stream=None) -> None:
        """Draw each expert's fp32 weights on the device (Philox4x32-10 + Box-Muller) and quantise them.

        stream_of(expert, proj) -> 64-bit stream id; weight index = expert id.
        """
        H, I = self.H, self.I
        dev = self.gu_codes.device
        tmp = torch.empty(H * I, dtype=torch.float32, device=dev)
        for e in (range(self.n) if experts is None else experts):
            for proj in (PROJ_GATE, PROJ_UP, PROJ_DOWN):
                ft_gen_normal_f32(seed, stream_of(e, proj), H * I, sigma, tmp, stream=stream)
                shape = (I, H) if proj != PROJ_DOWN else (H, I)
                self.quantize_projection(e, proj, tmp.view(*shape), stream=stream)


class MoEDecodeLayer:
    """route -> permute -> decode expert FFN (+ combine) through the C ABI, buffers allocated once."""

    def __init__(self, E: int, H: int, I: int, k: int, T: int, device):
        self.E, self.H, self.I, self.k, self.T = E, H, I, k, T
        i32 = torch.int32
        self.ids = torch.empty((T, k), dtype=i32, device=device)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.offsets = torch.empty(E + 1, dtype=i32, device=device)
        self.perm = torch.empty(T * k, dtype=i32, device=device)
        self.inv = torch.empty(T * k, dtype=i32, device=device)
        self.active = torch.empty(E + 1, dtype=i32, device=device)
        pw = ft_moe_permute_workspace_size(T, E, k)
        self.ws_perm = torch.empty(max(pw, 256), dtype=torch.uint8, device=device)
        self.ws = torch.empty(ft_moe_decode_workspace_size(T, k, H, I), dtype=torch.uint8, device=device)

    def __call__(self, weights: LayerWeights, logits: torch.Tensor, x: torch.Tensor, out: torch.Tensor,
                 y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        ft_moe_route(logits, self.k, self.ids, self.w, stream=stream)
        ft_moe_permute(self.ids, self.E, self.offsets, self.perm, self.inv, self.active, self.ws_perm, stream=stream)
        ft_moe_expert_ffn_nvfp4_decode(weights, x, self.k, self.offsets, self.perm, self.active, self.inv, self.w,
                                       y=y, out=out, ws=self.ws, stream=stream)
        return out
