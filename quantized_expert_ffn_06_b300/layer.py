"""Device-side containers for one MoE layer: NVFP4 expert weights in the
layout the kernels read, and the decode step through the C ABI (separate
route -> permute -> expert FFN -> combine calls, or the fused launch), with
buffers allocated once.
"""
from __future__ import annotations

import time

import torch

from . import (FT_LAYOUT_DECODE_TILES, FT_LAYOUT_MXFP4_DECODE_TILES, FT_LAYOUT_MXFP4_ROWS, FT_LAYOUT_MXFP8_DECODE_TILES,
               FT_LAYOUT_MXFP8_ROWS, FT_LAYOUT_ROWS, FT_LAYOUT_UMMA_TILES, ft_gen_normal_f32, ft_mxfp4_pack_tiles,
               ft_mxfp4_pack_umma, ft_mxfp4_quantize_weight, ft_mxfp8_pack_tiles, ft_mxfp8_quantize_weight,
               ft_moe_decode_workspace_size, ft_moe_expert_ffn_nvfp4_decode, ft_moe_expert_ffn_nvfp4_prefill,
               ft_moe_layer_decode, ft_moe_layer_decode_workspace_size, ft_moe_layer_weights, ft_moe_permute,
               ft_moe_permute_workspace_size, ft_moe_prefill_workspace_size, ft_moe_route, ft_nvfp4_pack_tiles,
               ft_nvfp4_pack_umma, ft_nvfp4_quantize_weight)

PROJ_GATE, PROJ_UP, PROJ_DOWN = 0, 1, 2


def wait_event(event, timeout_s: float, what: str) -> None:
    """Host wait for a CUDA event (anything with query()), bounded: raises FtError(FT_ERR_TIMEOUT) once timeout_s
    seconds have passed without the event completing, instead of blocking for ever."""
    from . import FT_ERR_TIMEOUT, FtError
    deadline = time.monotonic() + timeout_s
    while not event.query():
        if time.monotonic() > deadline:
            raise FtError(FT_ERR_TIMEOUT, f"{what}: not complete after {timeout_s} s")


class LayerWeights:
    """NVFP4 weights of one layer (E experts, or n_weights cache slots).

    layout ROWS:   gu_codes [n, 2I, H/2], gu_scales [n, 2I, H/16] (rows 2i / 2i+1 = gate / up row i),
                   d_codes [n, H, I/2], d_scales [n, H, I/16]
    layout TILES:  gu_codes [n, 2I*H*9/16], d_codes [n, H*I*9/16] (16-row tiles, see ft_nvfp4_pack_tiles)
    layout UMMA:   the same sizes in 128x128 blocks for the tensor-core prefill (see ft_nvfp4_pack_umma)
    tscale [n, 4] fp32 (gate, up, down, pad)
    layout UMMA with source="mxfp4": MXFP4 weights re-encoded exactly into the UMMA tiles (E4M3 power-of-two
                   block scales and a power-of-two tensor scale per matrix, see ft_mxfp4_pack_umma)
    MXFP4 layouts (UE8M0 scales per 32, no tensor scale):
    layout MXFP4_ROWS:  as ROWS with gu_scales [n, 2I, H/32], d_scales [n, H, I/32]
    layout MXFP4_TILES: gu_codes [n, 2I*H*17/32], d_codes [n, H*I*17/32] (see ft_mxfp4_pack_tiles)
    layout MXFP8_ROWS:  codes of one byte per element: gu_codes [n, 2I, H], d_codes [n, H, I]; scales as MXFP4
    layout MXFP8_TILES: gu_codes [n, 2I*H*33/32], d_codes [n, H*I*33/32] (see ft_mxfp8_pack_tiles)
    """

    def __init__(self, E: int, H: int, I: int, device, n_weights: int | None = None, layout: int = FT_LAYOUT_ROWS,
                 source: str = "nvfp4"):
        assert source in ("nvfp4", "mxfp4") and (source == "nvfp4" or layout == FT_LAYOUT_UMMA_TILES)
        self.mx_src = source == "mxfp4"
        self.E, self.H, self.I = E, H, I
        self.n = E if n_weights is None else n_weights
        self.layout = layout
        self.device = torch.device(device)
        u8 = torch.uint8
        self.mx8 = layout in (FT_LAYOUT_MXFP8_ROWS, FT_LAYOUT_MXFP8_DECODE_TILES)
        self.mx = self.mx8 or layout in (FT_LAYOUT_MXFP4_ROWS, FT_LAYOUT_MXFP4_DECODE_TILES)
        self.sblock = 32 if self.mx or self.mx_src else 16  # elements per scale (of the row-layout staging)
        self.cpe = 1 if self.mx8 else 2      # code elements per byte
        if layout in (FT_LAYOUT_ROWS, FT_LAYOUT_MXFP4_ROWS, FT_LAYOUT_MXFP8_ROWS):
            self.gu_codes = torch.empty((self.n, 2 * I, H // self.cpe), dtype=u8, device=device)
            self.gu_scales = torch.empty((self.n, 2 * I, H // self.sblock), dtype=u8, device=device)
            self.d_codes = torch.empty((self.n, H, I // self.cpe), dtype=u8, device=device)
            self.d_scales = torch.empty((self.n, H, I // self.sblock), dtype=u8, device=device)
        elif layout in (FT_LAYOUT_MXFP4_DECODE_TILES, FT_LAYOUT_MXFP8_DECODE_TILES):
            num = 33 if self.mx8 else 17
            self.gu_codes = torch.empty((self.n, 2 * I * H * num // 32), dtype=u8, device=device)
            self.d_codes = torch.empty((self.n, H * I * num // 32), dtype=u8, device=device)
            self.gu_scales = self.d_scales = None
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
        if self.gu_scales is not None:
            d.gu_scales, d.gu_scales_stride = self.gu_scales.data_ptr(), self.gu_scales.stride(0)
            d.d_scales, d.d_scales_stride = self.d_scales.data_ptr(), self.d_scales.stride(0)
        if not self.mx:  # MXFP4 has no tensor scale: the descriptor carries none
            d.tscale, d.tscale_stride = self.tscale.data_ptr(), self.tscale.stride(0)
        d.expert_to_slot = None if self.expert_to_slot is None else self.expert_to_slot.data_ptr()
        return d

    def _rows_target(self, wi: int):
        """Row-major destination for expert wi: the weights themselves (ROWS) or a staging copy (TILES)."""
        if self.layout in (FT_LAYOUT_ROWS, FT_LAYOUT_MXFP4_ROWS, FT_LAYOUT_MXFP8_ROWS):
            return self.gu_codes[wi], self.gu_scales[wi], self.d_codes[wi], self.d_scales[wi]
        if self._tmp is None:
            H, I, u8, dev, sb, c = self.H, self.I, torch.uint8, self.device, self.sblock, self.cpe
            self._tmp = (torch.empty((2 * I, H // c), dtype=u8, device=dev),
                         torch.empty((2 * I, H // sb), dtype=u8, device=dev),
                         torch.empty((H, I // c), dtype=u8, device=dev),
                         torch.empty((H, I // sb), dtype=u8, device=dev))
        return self._tmp

    def set_expert(self, wi: int, wg: torch.Tensor, wu: torch.Tensor, wd: torch.Tensor, stream=None) -> None:
        """Quantise fp32 gate [I,H], up [I,H], down [H,I] into weight index wi."""
        H, I = self.H, self.I
        guc, gus, dc, ds = self._rows_target(wi)
        if self.mx_src:  # MXFP4 rows, then re-encoded into the tensor-core tiles with a tensor scale per matrix
            for proj, w in ((PROJ_GATE, wg), (PROJ_UP, wu)):
                assert tuple(w.shape) == (I, H)
                ft_mxfp4_quantize_weight(w, guc.data_ptr() + proj * (H // 2), gus.data_ptr() + proj * (H // 32),
                                         codes_ld=H, scales_ld=H // 16, stream=stream)
            assert tuple(wd.shape) == (H, I)
            ft_mxfp4_quantize_weight(wd, dc, ds, stream=stream)
            ft_mxfp4_pack_umma(guc, H // 2, gus, H // 32, 2 * I, H, self.gu_codes[wi], self.tscale[wi, 0:2], 2,
                               stream=stream)
            ft_mxfp4_pack_umma(dc, I // 2, ds, I // 32, H, I, self.d_codes[wi], self.tscale[wi, 2:3], 1, stream=stream)
            return
        if self.mx:
            quant, pack, c = ((ft_mxfp8_quantize_weight, ft_mxfp8_pack_tiles, 1) if self.mx8 else
                              (ft_mxfp4_quantize_weight, ft_mxfp4_pack_tiles, 2))
            for proj, w in ((PROJ_GATE, wg), (PROJ_UP, wu)):
                assert tuple(w.shape) == (I, H)
                quant(w, guc.data_ptr() + proj * (H // c), gus.data_ptr() + proj * (H // 32),
                      codes_ld=2 * H // c, scales_ld=H // 16, stream=stream)
            assert tuple(wd.shape) == (H, I)
            quant(wd, dc, ds, stream=stream)
            if self.layout in (FT_LAYOUT_MXFP4_DECODE_TILES, FT_LAYOUT_MXFP8_DECODE_TILES):
                pack(guc, H // c, gus, H // 32, 2 * I, H, self.gu_codes[wi], stream=stream)
                pack(dc, I // c, ds, I // 32, H, I, self.d_codes[wi], stream=stream)
            return
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
        elif self.layout == FT_LAYOUT_UMMA_TILES:
            ft_nvfp4_pack_umma(guc, H // 2, gus, H // 16, 2 * I, H, self.gu_codes[wi], stream=stream)
            ft_nvfp4_pack_umma(dc, I // 2, ds, I // 16, H, I, self.d_codes[wi], stream=stream)

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


class MoEWeights:
    """The layer weights handle (ft_moe_weights_create) over canonical NVFP4 experts held by a row-layout
    LayerWeights: each expert's gate, up and down matrices are described in place (gate and up are the even and odd
    rows of the interleaved [2I][H] matrix) and repacked by the library into the requested layouts.
    view(layout) gives the descriptor object the layer calls take."""

    def __init__(self, canonical: LayerWeights, layout_flags: int, stream=None):
        from . import MoEWeightsHandle
        assert canonical.layout == FT_LAYOUT_ROWS
        c = canonical
        H, I = c.H, c.I
        experts = []
        for e in range(c.n):
            guc, gus, dc, ds = (t[e].data_ptr() for t in (c.gu_codes, c.gu_scales, c.d_codes, c.d_scales))
            ts = c.tscale[e].data_ptr()
            experts.append(((guc, H, gus, H // 8, ts), (guc + H // 2, H, gus + H // 16, H // 8, ts + 4),
                            (dc, I // 2, ds, I // 16, ts + 8)))
        self.handle = MoEWeightsHandle(experts, H, I, layout_flags, stream=stream)
        self.E, self.H, self.I, self.device = c.n, H, I, c.device

    def view(self, layout: int) -> "_HandleView":
        return _HandleView(self, layout)


class _DeviceBytes:
    """A library-owned device range presented to torch (zero copy, through the CUDA array interface)."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}


def _rows_view(ptr: int, n: int, row_bytes: int, stride: int, device) -> torch.Tensor:
    flat = torch.as_tensor(_DeviceBytes(ptr, (n - 1) * stride + row_bytes), device=device)
    return flat.as_strided((n, row_bytes), (stride, 1))


class _HandleView:
    """Descriptor of one layout held by a MoEWeights handle, with torch views of its bytes (per expert:
    gu_codes, d_codes, and for the row layout gu_scales, d_scales; tscale [E, 4])."""

    def __init__(self, w: MoEWeights, layout: int):
        self.w, self.layout = w, layout
        self.E, self.H, self.I, self.n, self.device = w.E, w.H, w.I, w.E, w.device
        self.expert_to_slot = None
        d = w.handle.describe(layout)
        E, H, I, dev = w.E, w.H, w.I, w.device
        if layout == FT_LAYOUT_ROWS:
            self.gu_codes = _rows_view(d.gu_codes, E, 2 * I * H // 2, d.gu_codes_stride, dev).view(E, 2 * I, H // 2)
            self.d_codes = _rows_view(d.d_codes, E, H * I // 2, d.d_codes_stride, dev).view(E, H, I // 2)
            self.gu_scales = _rows_view(d.gu_scales, E, 2 * I * H // 16, d.gu_scales_stride, dev).view(E, 2 * I, H // 16)
            self.d_scales = _rows_view(d.d_scales, E, H * I // 16, d.d_scales_stride, dev).view(E, H, I // 16)
        else:
            self.gu_codes = _rows_view(d.gu_codes, E, 2 * I * H * 9 // 16, d.gu_codes_stride, dev)
            self.d_codes = _rows_view(d.d_codes, E, H * I * 9 // 16, d.d_codes_stride, dev)
            self.gu_scales = self.d_scales = None
        self.tscale = _rows_view(d.tscale, E, 16, 16, dev).view(torch.float32)

    def desc(self) -> ft_moe_layer_weights:
        d = self.w.handle.describe(self.layout)
        if self.expert_to_slot is not None:
            d.expert_to_slot = self.expert_to_slot.data_ptr()
        return d


class PrefillLayer:
    """route -> permute -> tensor-core NVFP4 expert FFN with the combine, buffers allocated once."""

    def __init__(self, E: int, H: int, I: int, k: int, T: int, device):
        self.E, self.H, self.I, self.k, self.T = E, H, I, k, T
        i32 = torch.int32
        self.ids = torch.empty((T, k), dtype=i32, device=device)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.offsets = torch.empty(E + 1, dtype=i32, device=device)
        self.perm = torch.empty(T * k, dtype=i32, device=device)
        self.inv = torch.empty(T * k, dtype=i32, device=device)
        self.active = torch.empty(E + 1, dtype=i32, device=device)
        self.ws_perm = torch.empty(max(ft_moe_permute_workspace_size(T, E, k), 256), dtype=torch.uint8, device=device)
        self.ws = torch.empty(ft_moe_prefill_workspace_size(T, k, E, H, I), dtype=torch.uint8, device=device)

    def __call__(self, weights: LayerWeights, logits: torch.Tensor, x: torch.Tensor, out: torch.Tensor,
                 stream=None) -> torch.Tensor:
        ft_moe_route(logits, self.k, self.ids, self.w, stream=stream)
        ft_moe_permute(self.ids, self.E, self.offsets, self.perm, self.inv, self.active, self.ws_perm, stream=stream)
        ft_moe_expert_ffn_nvfp4_prefill(weights, x, self.k, self.offsets, self.perm, self.w, out, self.ws,
                                        stream=stream)
        return out


class StreamedPrefill:
    """Prefill through L layers whose NVFP4 experts live in pinned host memory, double-buffered.

    The experts of layer l+1 are copied host -> device on a side stream into one of two device buffers while layer
    l computes from the other; events order each copy after the layer that last read its buffer, and each layer
    after its copy.  Each expert is one contiguous block in the tensor-core tile layout,
        [gate/up blocks: 2I*H*9/16 bytes][down blocks: H*I*9/16 bytes][tensor scales: 4 floats],
    at a 256-byte stride, in the host pool and in a buffer alike, so a layer moves as one copy.
    """

    def __init__(self, L: int, E: int, H: int, I: int, k: int, T: int, device):
        self.L, self.E, self.H, self.I, self.k, self.T = L, E, H, I, k, T
        self.device = torch.device(device)
        self.gu_bytes = 2 * I * H * 9 // 16
        self.d_bytes = H * I * 9 // 16
        self.expert_bytes = self.gu_bytes + self.d_bytes + 16
        self.slot_stride = (self.expert_bytes + 255) // 256 * 256
        self.layer_bytes = E * self.slot_stride
        self.host = torch.empty(L * self.layer_bytes, dtype=torch.uint8, pin_memory=True)
        self.bufs = [torch.empty(self.layer_bytes, dtype=torch.uint8, device=self.device) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=self.device)
        self.landed = [torch.cuda.Event() for _ in range(2)]  # the layer assigned to buffer b is on the device
        self.freed = [torch.cuda.Event() for _ in range(2)]   # the layer that last read buffer b has finished
        self.layer = PrefillLayer(E, H, I, k, T, self.device)

    def load_layer(self, layer: int, lw: LayerWeights) -> None:
        """Copy the E experts of a device LayerWeights (tensor-core tile layout) into the host pool."""
        assert lw.layout == FT_LAYOUT_UMMA_TILES and lw.n >= self.E
        g, d, eb = self.gu_bytes, self.d_bytes, self.expert_bytes
        stage = torch.zeros((self.E, self.slot_stride), dtype=torch.uint8, device=lw.device)
        stage[:, :g].copy_(lw.gu_codes[:self.E])
        stage[:, g:g + d].copy_(lw.d_codes[:self.E])
        stage[:, g + d:eb].copy_(lw.tscale[:self.E].view(torch.uint8))
        off = layer * self.layer_bytes
        self.host[off:off + self.layer_bytes].view(self.E, self.slot_stride).copy_(stage)  # device -> pinned
        torch.cuda.synchronize(lw.device)

    def buffer_weights(self, b: int) -> "_BufferWeights":
        return _BufferWeights(self, b)

    def _issue_copy(self, layer: int) -> None:
        b = layer % 2
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.freed[b])
            off = layer * self.layer_bytes
            self.bufs[b].copy_(self.host[off:off + self.layer_bytes], non_blocking=True)
            self.landed[b].record(self.copy_stream)

    def __call__(self, logits, xs, outs, stream=None):
        """Layer l reads logits[l] [T, E] fp32 and xs[l] [T, H] bf16 and writes outs[l] [T, H] bf16."""
        stream = torch.cuda.current_stream(self.device) if stream is None else stream
        self._issue_copy(0)
        for l in range(self.L):
            if l + 1 < self.L:
                self._issue_copy(l + 1)  # overlaps this layer's compute
            stream.wait_event(self.landed[l % 2])
            self.layer(self.buffer_weights(l % 2), logits[l], xs[l], outs[l], stream=stream)
            self.freed[l % 2].record(stream)
        return outs


class _BufferWeights:
    """Descriptor of the experts in one StreamedPrefill buffer (tensor-core tile layout, no slot table)."""

    def __init__(self, sp: StreamedPrefill, b: int):
        self.sp, self.b = sp, b
        self.E, self.H, self.I, self.n = sp.E, sp.H, sp.I, sp.E
        self.layout = FT_LAYOUT_UMMA_TILES
        self.device = sp.device

    def desc(self) -> ft_moe_layer_weights:
        sp = self.sp
        d = ft_moe_layer_weights()
        d.E, d.H, d.I, d.n_weights, d.layout = sp.E, sp.H, sp.I, sp.E, FT_LAYOUT_UMMA_TILES
        base = sp.bufs[self.b].data_ptr()
        d.gu_codes, d.gu_codes_stride = base, sp.slot_stride
        d.d_codes, d.d_codes_stride = base + sp.gu_bytes, sp.slot_stride
        d.tscale, d.tscale_stride = base + sp.gu_bytes + sp.d_bytes, sp.slot_stride // 4
        return d


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


class ExpertSlotPool:
    """Expert weights of L layers in pinned host memory, a VRAM pool of S slots per layer, and the LRU cache
    (ft_expert_cache_*) that maps experts to slots.

    Each expert occupies one contiguous block, in the host pool and in its slot alike:
        [gate/up tiles: 2I*H*9/16 bytes][down tiles: H*I*9/16 bytes][tensor scales: 4 floats]
    so that a miss is filled by one cudaMemcpyAsync.  layer_weights(l) describes layer l's slots for the FFN
    kernels (weight index = slot, expert_to_slot = the layer's device table).
    """

    def __init__(self, L: int, E: int, H: int, I: int, S: int, device):
        import ctypes

        from . import ExpertCacheHandle
        self.L, self.E, self.H, self.I, self.S = L, E, H, I, S
        self.device = torch.device(device)
        self.gu_bytes = 2 * I * H * 9 // 16
        self.d_bytes = H * I * 9 // 16
        self.expert_bytes = self.gu_bytes + self.d_bytes + 16
        self.slot_stride = (self.expert_bytes + 255) // 256 * 256
        self.host = torch.empty(L * E * self.slot_stride, dtype=torch.uint8, pin_memory=True)
        self.slots = torch.empty(L * S * self.slot_stride, dtype=torch.uint8, device=self.device)
        self.tables = torch.full((L, E), -1, dtype=torch.int32, device=self.device)
        base = self.host.data_ptr()
        ptrs = [base + i * self.slot_stride for i in range(L * E)]
        self.cache = ExpertCacheHandle(L, E, S, self.expert_bytes, ptrs, self.slots.data_ptr(), self.slot_stride,
                                       self.tables.data_ptr())
        self._ctypes = ctypes

    def host_expert(self, layer: int, e: int) -> torch.Tensor:
        off = (layer * self.E + e) * self.slot_stride
        return self.host[off:off + self.expert_bytes]

    def load_layer(self, layer: int, lw: LayerWeights) -> None:
        """Copy the E experts of a device LayerWeights (decode-tile layout) into the host pool."""
        assert lw.layout == FT_LAYOUT_DECODE_TILES and lw.n >= self.E
        stage = torch.empty((self.E, self.slot_stride), dtype=torch.uint8, device=lw.device)
        stage[:, :self.gu_bytes].copy_(lw.gu_codes[:self.E])
        stage[:, self.gu_bytes:self.gu_bytes + self.d_bytes].copy_(lw.d_codes[:self.E])
        stage[:, self.gu_bytes + self.d_bytes:self.expert_bytes].copy_(lw.tscale[:self.E].view(torch.uint8))
        off = layer * self.E * self.slot_stride
        self.host[off:off + self.E * self.slot_stride].view(self.E, self.slot_stride).copy_(stage)  # device -> pinned
        torch.cuda.synchronize(lw.device)

    def layer_weights(self, layer: int) -> "SlotLayerWeights":
        return SlotLayerWeights(self, layer)

    def resize(self, new_S: int, in_place: bool = False, stream=None) -> None:
        """Elastic resize at a safe point: the cache becomes new_S slots per layer, rebuilt from the experts already
        in VRAM (device-to-device; the least recently used leave when it shrinks).  A new pool is allocated unless
        ``in_place`` (a shrink that compacts the current pool and frees nothing).  The caller orders every fill and
        every kernel that reads the current pool before ``stream`` (default: the current stream)."""
        stream = torch.cuda.current_stream(self.device) if stream is None else stream
        if in_place:
            if new_S > self.S:
                raise ValueError("only a shrink can be done in place")
            new_pool = self.slots
        else:
            new_pool = torch.empty(self.L * new_S * self.slot_stride, dtype=torch.uint8, device=self.device)
        from . import FT_ERR_INVALID_ARG, FtError
        old_pool = self.slots
        try:
            self.cache.resize(new_S, new_pool.data_ptr(), self.slot_stride, stream=stream)
        except FtError as e:
            if e.status == FT_ERR_INVALID_ARG:
                raise  # rejected before any change: the cache still uses the current pool
            self._adopt(new_S, new_pool, old_pool, stream)  # the handle is on the new pool either way
            raise
        self._adopt(new_S, new_pool, old_pool, stream)

    def _adopt(self, new_S, new_pool, old_pool, stream) -> None:
        self.S, self.slots = new_S, new_pool
        if old_pool is not new_pool:
            old_pool.record_stream(stream)  # kept alive until the moves on `stream` have read it


class SlotLayerWeights:
    """Descriptor of one layer's cache slots for the FFN kernels (decode-tile layout)."""

    def __init__(self, pool: ExpertSlotPool, layer: int):
        self.pool, self.layer = pool, layer
        self.E, self.H, self.I = pool.E, pool.H, pool.I
        self.layout = FT_LAYOUT_DECODE_TILES
        self.device = pool.device

    @property
    def n(self) -> int:  # the pool's current slot count (it changes on a resize)
        return self.pool.S

    def desc(self) -> ft_moe_layer_weights:
        p = self.pool
        d = ft_moe_layer_weights()
        d.E, d.H, d.I, d.n_weights, d.layout = p.E, p.H, p.I, p.S, FT_LAYOUT_DECODE_TILES
        base = p.slots.data_ptr() + self.layer * p.S * p.slot_stride
        d.gu_codes, d.gu_codes_stride = base, p.slot_stride
        d.d_codes, d.d_codes_stride = base + p.gu_bytes, p.slot_stride
        d.tscale, d.tscale_stride = base + p.gu_bytes + p.d_bytes, p.slot_stride // 4
        d.expert_to_slot = p.tables[self.layer].data_ptr()
        return d


class CachedDecodeLayer:
    """Decode step of one layer whose experts come from an ExpertSlotPool.

    route (device) -> expert ids to the host -> LRU lookup -> fills of the misses on the copy stream -> publish the
    slot table -> the fused layer kernel (which routes again, identically, and reads weights through the table).

    With prefetch = P > 0 the router also ranks the next P experts of the token, and those are installed in the
    cache for the next token and copied on the copy stream behind this token's fills, overlapping later layers'
    compute (router-driven prefetch; ft_expert_cache_prefetch)."""

    def __init__(self, pool: ExpertSlotPool, layer: int, k: int, T: int, copy_stream=None, timeout_s: float = 2.0,
                 prefetch: int = 0):
        self.pool, self.layer, self.k, self.T = pool, layer, k, T
        self.timeout_s = timeout_s
        self.prefetch = prefetch
        dev = pool.device
        self.weights = pool.layer_weights(layer)
        kr = k + prefetch  # the router ranks k + P experts; the first k are the token's (same order, same ties)
        self.ids = torch.empty((T, kr), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, kr), dtype=torch.float32, device=dev)
        self.ids_host = torch.empty((T, kr), dtype=torch.int32).pin_memory()
        self.fused = FusedDecodeLayer(pool.E, pool.H, pool.I, k, T, dev)
        self.copy_stream = copy_stream if copy_stream is not None else torch.cuda.Stream(device=dev)
        self.filled = torch.cuda.Event()
        self.routed = torch.cuda.Event()
        # host seconds spent, summed over calls: waiting for the routing result, in the cache's host logic
        # (lookup, fill and prefetch enqueues, publish), and enqueueing the rest
        self.host_wait_s = self.host_cache_s = self.host_call_s = 0.0

    def __call__(self, logits: torch.Tensor, x: torch.Tensor, out: torch.Tensor, step: int, stream=None,
                 predicted=None):
        """One token's layer step; returns the (expert, slot) misses filled for it.  `predicted` (host ints,
        optional) replaces the router's next P ranks as the experts installed for the next token."""
        stream = torch.cuda.current_stream(self.pool.device) if stream is None else stream
        t0 = time.perf_counter()
        ft_moe_route(logits, self.k + self.prefetch, self.ids, self.w, stream=stream)
        with torch.cuda.stream(stream):
            self.ids_host.copy_(self.ids, non_blocking=True)
            self.routed.record(stream)
        t1 = time.perf_counter()
        wait_event(self.routed, self.timeout_s, f"layer {self.layer}: routing result")
        t2 = time.perf_counter()
        ranked = self.ids_host.tolist()
        needed = sorted(set(int(e) for row in ranked for e in row[:self.k]))
        _, misses = self.pool.cache.lookup(self.layer, step, needed)
        for e, s in misses:
            self.pool.cache.fill(self.layer, e, s, stream=self.copy_stream)
        self.filled.record(self.copy_stream)
        self.pool.cache.publish(self.layer, stream=stream)
        stream.wait_event(self.filled)
        t3 = time.perf_counter()
        self.fused(self.weights, logits, x, out, routing=False, stream=stream)
        t4 = time.perf_counter()
        if self.prefetch or predicted is not None:
            # the next-ranked experts, for the next token: copied behind this token's fills, which the next step's
            # kernel waits for (same copy stream), while this and later layers compute
            if predicted is None:
                predicted = set(int(e) for row in ranked for e in row[self.k:])
            predicted = sorted(set(int(e) for e in predicted) - set(needed))
            self.prefetched = self.pool.cache.prefetch(self.layer, step, predicted)
            for e, s in self.prefetched:
                self.pool.cache.fill(self.layer, e, s, stream=self.copy_stream)
        t5 = time.perf_counter()
        self.host_wait_s += t2 - t1
        self.host_cache_s += (t3 - t2) + (t5 - t4)
        self.host_call_s += (t1 - t0) + (t4 - t3)
        return misses
