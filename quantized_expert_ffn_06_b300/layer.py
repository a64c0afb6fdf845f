"""Device-side containers for one MoE layer: NVFP4 expert weights in the
layout the kernels read, and the decode step through the C ABI (separate
route -> permute -> expert FFN -> combine calls, or the fused launch), with
buffers allocated once.
"""
from __future__ import annotations

import torch

from . import (FT_LAYOUT_DECODE_TILES, FT_LAYOUT_ROWS, ft_gen_normal_f32, ft_moe_decode_workspace_size,
               ft_moe_expert_ffn_nvfp4_decode, ft_moe_layer_decode, ft_moe_layer_decode_workspace_size,
               ft_moe_layer_weights, ft_moe_permute, ft_moe_permute_workspace_size, ft_moe_route, ft_nvfp4_pack_tiles,
               ft_nvfp4_quantize_weight)

PROJ_GATE, PROJ_UP, PROJ_DOWN = 0, 1, 2


class LayerWeights:
    """NVFP4 weights of one layer (E experts, or n_weights cache slots).

    layout ROWS:   gu_codes [n, 2I, H/2], gu_scales [n, 2I, H/16] (rows 2i / 2i+1 = gate / up row i),
                   d_codes [n, H, I/2], d_scales [n, H, I/16]
    layout TILES:  gu_codes [n, 2I*H*9/16], d_codes [n, H*I*9/16] (16-row tiles, see ft_nvfp4_pack_tiles)
    tscale [n, 4] fp32 (gate, up, down, pad)
    """

    def __init__(self, E: int, H: int, I: int, device, n_weights: int | None = None, layout: int = FT_LAYOUT_ROWS):
        self.E, self.H, self.I = E, H, I
        self.n = E if n_weights is None else n_weights
        self.layout = layout
        self.device = torch.device(device)
        u8 = torch.uint8
        if layout == FT_LAYOUT_ROWS:
            self.gu_codes = torch.empty((self.n, 2 * I, H // 2), dtype=u8, device=device)
            self.gu_scales = torch.empty((self.n, 2 * I, H // 16), dtype=u8, device=device)
            self.d_codes = torch.empty((self.n, H, I // 2), dtype=u8, device=device)
            self.d_scales = torch.empty((self.n, H, I // 16), dtype=u8, device=device)
        else:
            self.gu_codes = torch.empty((self.n, 2 * I * H * 9 // 16), dtype=u8, device=device)
            self.d_codes = torch.empty((self.n, H * I * 9 // 16), dtype=u8, device=device)
            self.gu_scales = self.d_scales = None
        self._tmp = None
        self.tscale = torch.zeros((self.n, 4), dtype=torch.float32, device=device)
        self.expert_to_slot: torch.Tensor | None = None
        self._qws = torch.empty(256, dtype=u8, device=device)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.gu_codes, self.gu_scales, self.d_codes, self.d_scales)
                   if t is not None)

    def desc(self) -> ft_moe_layer_weights:
        d = ft_moe_layer_weights()
        d.E, d.H, d.I, d.n_weights, d.layout = self.E, self.H, self.I, self.n, self.layout
        d.gu_codes, d.gu_codes_stride = self.gu_codes.data_ptr(), self.gu_codes.stride(0)
        d.d_codes, d.d_codes_stride = self.d_codes.data_ptr(), self.d_codes.stride(0)
        if self.layout == FT_LAYOUT_ROWS:
            d.gu_scales, d.gu_scales_stride = self.gu_scales.data_ptr(), self.gu_scales.stride(0)
            d.d_scales, d.d_scales_stride = self.d_scales.data_ptr(), self.d_scales.stride(0)
        d.tscale, d.tscale_stride = self.tscale.data_ptr(), self.tscale.stride(0)
        d.expert_to_slot = None if self.expert_to_slot is None else self.expert_to_slot.data_ptr()
        return d

    def _rows_target(self, wi: int):
        """Row-major destination for expert wi: the weights themselves (ROWS) or a staging copy (TILES)."""
        if self.layout == FT_LAYOUT_ROWS:
            return self.gu_codes[wi], self.gu_scales[wi], self.d_codes[wi], self.d_scales[wi]
        if self._tmp is None:
            H, I, u8, dev = self.H, self.I, torch.uint8, self.device
            self._tmp = (torch.empty((2 * I, H // 2), dtype=u8, device=dev),
                         torch.empty((2 * I, H // 16), dtype=u8, device=dev),
                         torch.empty((H, I // 2), dtype=u8, device=dev),
                         torch.empty((H, I // 16), dtype=u8, device=dev))
        return self._tmp

    def set_expert(self, wi: int, wg: torch.Tensor, wu: torch.Tensor, wd: torch.Tensor, stream=None) -> None:
        """Quantise fp32 gate [I,H], up [I,H], down [H,I] into weight index wi."""
        H, I = self.H, self.I
        guc, gus, dc, ds = self._rows_target(wi)
        for proj, w in ((PROJ_GATE, wg), (PROJ_UP, wu)):
            assert tuple(w.shape) == (I, H)
            ft_nvfp4_quantize_weight(w, guc.data_ptr() + proj * (H // 2), gus.data_ptr() + proj * (H // 16),
                                     self.tscale[wi, proj:proj + 1], codes_ld=H, scales_ld=H // 8, ws=self._qws,
                                     stream=stream)
        assert tuple(wd.shape) == (H, I)
        ft_nvfp4_quantize_weight(wd, dc, ds, self.tscale[wi, 2:3], ws=self._qws, stream=stream)
        if self.layout == FT_LAYOUT_DECODE_TILES:
            ft_nvfp4_pack_tiles(guc, H // 2, gus, H // 16, 2 * I, H, self.gu_codes[wi], stream=stream)
            ft_nvfp4_pack_tiles(dc, I // 2, ds, I // 16, H, I, self.d_codes[wi], stream=stream)

    def fill_synthetic(self, stream_of, seed: int = 0, sigma: float = 0.02, experts=None, stream=None) -> None:
        """Draw each expert's fp32 weights on the device (Philox4x32-10 + Box-Muller) and quantise them.

        stream_of(expert, proj) -> 64-bit stream id; weight index = expert id.
        """
        H, I = self.H, self.I
        tmp = [torch.empty(H * I, dtype=torch.float32, device=self.device) for _ in range(3)]
        for e in (range(self.n) if experts is None else experts):
            for proj in (PROJ_GATE, PROJ_UP, PROJ_DOWN):
                ft_gen_normal_f32(seed, stream_of(e, proj), H * I, sigma, tmp[proj], stream=stream)
            self.set_expert(e, tmp[0].view(I, H), tmp[1].view(I, H), tmp[2].view(H, I), stream=stream)


class MoEDecodeLayer:
    """route -> permute -> decode expert FFN (+ combine) as separate C-ABI calls, buffers allocated once."""

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
        self.ws = torch.zeros(ft_moe_decode_workspace_size(T, k, H, I), dtype=torch.uint8, device=device)

    def __call__(self, weights: LayerWeights, logits: torch.Tensor, x: torch.Tensor, out: torch.Tensor,
                 y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        ft_moe_route(logits, self.k, self.ids, self.w, stream=stream)
        ft_moe_permute(self.ids, self.E, self.offsets, self.perm, self.inv, self.active, self.ws_perm, stream=stream)
        ft_moe_expert_ffn_nvfp4_decode(weights, x, self.k, self.offsets, self.perm, self.active, self.inv, self.w,
                                       y=y, out=out, ws=self.ws, stream=stream)
        return out


class FusedDecodeLayer:
    """The fused decode launch (route + group + FFN + combine) with its zero-initialised workspace."""

    def __init__(self, E: int, H: int, I: int, k: int, T: int, device):
        self.E, self.H, self.I, self.k, self.T = E, H, I, k, T
        self.ids = torch.empty((T, k), dtype=torch.int32, device=device)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.ws = torch.zeros(ft_moe_layer_decode_workspace_size(T, k, H, I), dtype=torch.uint8, device=device)

    def __call__(self, weights: LayerWeights, logits: torch.Tensor, x: torch.Tensor, out: torch.Tensor,
                 routing: bool = True, stream=None) -> torch.Tensor:
        ft_moe_layer_decode(weights, logits, x, self.k, out, self.ws, ids=self.ids if routing else None,
                            w=self.w if routing else None, stream=stream)
        return out
