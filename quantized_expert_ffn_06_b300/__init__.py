"""Thin Python binding of libftmoe.so (the C ABI declared in include/ftmoe.h).

Argument marshalling only: every step of the MoE layer runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  If the compiled
library is missing this module raises at import -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libftmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libftmoe.so not found at {LIB_PATH}; build it with "
                      "`python quantized_expert_ffn_06_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

FT_OK, FT_ERR_INVALID_ARG, FT_ERR_CUDA, FT_ERR_UNSUPPORTED, FT_ERR_TIMEOUT, FT_ERR_NO_SLOT, FT_ERR_OOM, \
    FT_ERR_DEVICE = range(8)
FT_LAYOUT_ROWS, FT_LAYOUT_DECODE_TILES, FT_LAYOUT_UMMA_TILES = 0, 1, 2
FT_LAYOUT_MXFP4_ROWS, FT_LAYOUT_MXFP4_DECODE_TILES = 3, 4
FT_LAYOUT_MXFP8_ROWS, FT_LAYOUT_MXFP8_DECODE_TILES = 5, 6
FT_DEVERR_NAN_LOGIT, FT_DEVERR_BAD_SCALE, FT_DEVERR_TIMEOUT, FT_DEVERR_BAD_INDEX, FT_DEVERR_RANGE = 1, 2, 4, 8, 16
FT_WAIT_SITE_NONE, FT_WAIT_SITE_DECODE_H, FT_WAIT_SITE_PREFILL_TOKEN = 0, 1, 2

_vp, _i32, _i64, _u64, _sz, _dbl = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t,
                                    ctypes.c_double)


class FtError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_lib.ft_status_string(status).decode()}: {msg}")
        self.status = status


class ft_moe_layer_weights(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("n_weights", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("gu_codes", _vp), ("gu_codes_stride", _i64),
                ("gu_scales", _vp), ("gu_scales_stride", _i64),
                ("d_codes", _vp), ("d_codes_stride", _i64),
                ("d_scales", _vp), ("d_scales_stride", _i64),
                ("tscale", _vp), ("tscale_stride", _i64),
                ("expert_to_slot", _vp),
                ("gu_sf_tiled", _vp), ("gu_sf_tiled_stride", _i64),
                ("d_sf_tiled", _vp), ("d_sf_tiled_stride", _i64)]


class ft_nvfp4_matrix(ctypes.Structure):
    _fields_ = [("codes", _vp), ("codes_ld", _i64), ("scales", _vp), ("scales_ld", _i64), ("tensor_scale", _vp)]


class ft_nvfp4_expert_desc(ctypes.Structure):
    _fields_ = [("gate", ft_nvfp4_matrix), ("up", ft_nvfp4_matrix), ("down", ft_nvfp4_matrix)]


FT_WEIGHTS_ROWS, FT_WEIGHTS_DECODE_TILES, FT_WEIGHTS_UMMA_TILES = 1, 2, 4


def _sig(name, args, res=ctypes.c_int):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_sig("ft_status_string", [_i32], ctypes.c_char_p)
_sig("ft_last_error", [], ctypes.c_char_p)
_sig("ft_version", [], _i32)
_sig("ft_device_status", [_vp, ctypes.POINTER(ctypes.c_uint32)])
_sig("ft_moe_route", [_vp, _i32, _i32, _i32, _vp, _vp, _vp])
_sig("ft_moe_permute_workspace_size", [_i32, _i32, _i32], _sz)
_sig("ft_moe_permute", [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp])
_sig("ft_moe_decode_workspace_size", [_i32, _i32, _i32, _i32], _sz)
_sig("ft_moe_expert_ffn_nvfp4_decode", [ctypes.POINTER(ft_moe_layer_weights), _vp, _i32, _i32, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _sz, _vp])
_sig("ft_moe_combine", [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp])
_sig("ft_nvfp4_quantize_workspace_size", [_i64, _i64], _sz)
_sig("ft_nvfp4_quantize_weight", [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _sz, _vp])
_sig("ft_nvfp4_quantize_act", [_vp, _i64, _i64, _vp, _vp, _vp])
_sig("ft_gen_normal_f32", [_u64, _u64, _u64, _i64, _dbl, _vp, _vp])
_sig("ft_nvfp4_pack_tiles", [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp])
_sig("ft_moe_layer_decode_workspace_size", [_i32, _i32, _i32, _i32], _sz)
_sig("ft_moe_layer_decode", [ctypes.POINTER(ft_moe_layer_weights), _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _sz,
                             _vp])
_sig("ft_debug_inject_wait_expiry", [_i32, _u64])
_sig("ft_moe_layer_decode_noalloc", [ctypes.POINTER(ft_moe_layer_weights), _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp])
_sig("ft_nvfp4_pack_umma", [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp])
_sig("ft_mxfp4_quantize_weight", [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp])
_sig("ft_mxfp4_pack_tiles", [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp])
_sig("ft_mxfp4_pack_umma", [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp, _i32, _vp])
_sig("ft_mxfp8_quantize_weight", [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp])
_sig("ft_mxfp8_pack_tiles", [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp])
_sig("ft_moe_prefill_workspace_size", [_i32, _i32, _i32, _i32, _i32], _sz)
_sig("ft_moe_expert_ffn_nvfp4_prefill", [ctypes.POINTER(ft_moe_layer_weights), _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _sz, _vp])
_sig("ft_expert_cache_create", [_i32, _i32, _i32, _sz, ctypes.POINTER(ctypes.c_void_p), _vp, _sz, _vp,
                                ctypes.POINTER(ctypes.c_void_p)])
_sig("ft_expert_cache_destroy", [_vp])
_sig("ft_expert_cache_lookup", [_vp, _i32, _i64, ctypes.POINTER(ctypes.c_int32), _i32, ctypes.POINTER(ctypes.c_int32),
                                ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_i32)])
_sig("ft_expert_cache_fill", [_vp, _i32, _i32, _i32, _vp, _vp])
_sig("ft_expert_cache_publish", [_vp, _i32, _vp])
_sig("ft_expert_cache_stats", [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64)])
_sig("ft_expert_cache_inject_fill_failure", [_vp, _i64])
_sig("ft_expert_cache_prefetch", [_vp, _i32, _i64, ctypes.POINTER(ctypes.c_int32), _i32, ctypes.POINTER(ctypes.c_int32),
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_i32)])
_sig("ft_expert_cache_prefetch_stats", [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64)])
_sig("ft_expert_cache_resize", [_vp, _i32, _vp, _sz, _vp])
_sig("ft_expert_cache_resize_plan", [_vp, _i32, ctypes.POINTER(ctypes.c_int32)])

_sig("ft_moe_weights_create", [ctypes.POINTER(ft_nvfp4_expert_desc), _i32, _i32, _i32, _i32, _vp,
                               ctypes.POINTER(ctypes.c_void_p)])
_sig("ft_moe_weights_describe", [_vp, _i32, ctypes.POINTER(ft_moe_layer_weights)])
_sig("ft_moe_weights_destroy", [_vp])

EXPORTED = [n for n in dir(_lib) if n.startswith("ft_")]


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int) -> None:
    if rc != FT_OK:
        raise FtError(rc, _lib.ft_last_error().decode())


def _p(t) -> int | None:
    if t is None or isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _req(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}, got {t.dtype} on {t.device}")


def _ws(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------- status

def ft_version() -> int:
    return _lib.ft_version()


def ft_debug_inject_wait_expiry(site: int, limit_ns: int = 0) -> None:
    """Test hook: make a device wait run out after limit_ns (site FT_WAIT_SITE_*); FT_WAIT_SITE_NONE turns it off."""
    _check(_lib.ft_debug_inject_wait_expiry(int(site), int(limit_ns)))


def ft_device_status(stream=None) -> int:
    """Waits for the stream, returns and clears the device error word (raises on CUDA errors only)."""
    word = ctypes.c_uint32(0)
    rc = _lib.ft_device_status(_s(stream), ctypes.byref(word))
    if rc not in (FT_OK, FT_ERR_DEVICE):
        _check(rc)
    return word.value


# --------------------------------------------------------------------------- router / permute / combine

def ft_moe_route(logits: torch.Tensor, k: int, ids=None, w=None, stream=None):
    _req(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device) if ids is None else ids
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device) if w is None else w
    _check(_lib.ft_moe_route(_p(logits), T, E, k, _p(ids), _p(w), _s(stream)))
    return ids, w


def ft_moe_permute_workspace_size(T: int, E: int, k: int) -> int:
    return _lib.ft_moe_permute_workspace_size(T, E, k)


def ft_moe_permute(ids: torch.Tensor, E: int, offsets=None, perm=None, inv=None, active=None, ws=None, stream=None):
    _req(ids, torch.int32, "ids")
    T, k = ids.shape
    dev = ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    perm = torch.empty(T * k, dtype=torch.int32, device=dev) if perm is None else perm
    inv = torch.empty(T * k, dtype=torch.int32, device=dev) if inv is None else inv
    active = torch.empty(E + 1, dtype=torch.int32, device=dev) if active is None else active
    need = ft_moe_permute_workspace_size(T, E, k)
    ws = _ws(need, dev) if ws is None else ws
    _check(_lib.ft_moe_permute(_p(ids), T, E, k, _p(offsets), _p(perm), _p(inv), _p(active), _p(ws),
                               0 if ws is None else ws.numel() * ws.element_size(), _s(stream)))
    return offsets, perm, inv, active


def ft_moe_combine(y: torch.Tensor, inv: torch.Tensor, w: torch.Tensor, T: int, k: int, out=None, stream=None):
    _req(y, torch.float32, "y")
    H = y.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device) if out is None else out
    _check(_lib.ft_moe_combine(_p(y), _p(inv), _p(w), T, k, H, _p(out), _s(stream)))
    return out


# --------------------------------------------------------------------------- expert FFN

def ft_moe_decode_workspace_size(T: int, k: int, H: int, I: int) -> int:
    return _lib.ft_moe_decode_workspace_size(T, k, H, I)


def ft_moe_expert_ffn_nvfp4_decode(W, x: torch.Tensor, k: int, offsets, perm, active, inv=None, w=None, y=None,
                                   out=None, ws=None, stream=None):
    """W: a LayerWeights (or anything with .desc()).  Returns (y, out)."""
    _req(x, torch.bfloat16, "x")
    T, H = x.shape
    desc = W.desc()
    need = ft_moe_decode_workspace_size(T, k, desc.H, desc.I)
    ws = _ws(need, x.device) if ws is None else ws
    _check(_lib.ft_moe_expert_ffn_nvfp4_decode(ctypes.byref(desc), _p(x), T, k, _p(offsets), _p(perm), _p(active),
                                               _p(inv), _p(w), _p(y), _p(out), _p(ws),
                                               0 if ws is None else ws.numel() * ws.element_size(), _s(stream)))
    return y, out


# --------------------------------------------------------------------------- quantisers / generator

def ft_nvfp4_quantize_weight(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, tensor_scale: torch.Tensor,
                             codes_ld: int | None = None, scales_ld: int | None = None, ws=None, stream=None):
    _req(w, torch.float32, "w")
    N, K = w.shape
    codes_ld = K // 2 if codes_ld is None else codes_ld
    scales_ld = K // 16 if scales_ld is None else scales_ld
    need = _lib.ft_nvfp4_quantize_workspace_size(N, K)
    ws = _ws(need, w.device) if ws is None else ws
    _check(_lib.ft_nvfp4_quantize_weight(_p(w), N, K, _p(codes), codes_ld, _p(scales), scales_ld, _p(tensor_scale),
                                         _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def ft_nvfp4_quantize_act(x: torch.Tensor, codes=None, scales=None, stream=None):
    _req(x, torch.bfloat16, "x")
    T, K = x.shape
    codes = torch.empty((T, K // 2), dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty((T, K // 16), dtype=torch.uint8, device=x.device) if scales is None else scales
    _check(_lib.ft_nvfp4_quantize_act(_p(x), T, K, _p(codes), _p(scales), _s(stream)))
    return codes, scales


def ft_gen_normal_f32(seed: int, stream_id: int, n: int, sigma: float, out: torch.Tensor, first: int = 0,
                      stream=None):
    _req(out, torch.float32, "out")
    _check(_lib.ft_gen_normal_f32(seed, stream_id, first, n, sigma, _p(out), _s(stream)))
    return out


def ft_nvfp4_pack_tiles(codes, codes_ld: int, scales, scales_ld: int, N: int, K: int, tiles, stream=None):
    _check(_lib.ft_nvfp4_pack_tiles(_p(codes), codes_ld, _p(scales), scales_ld, N, K, _p(tiles), _s(stream)))


def ft_mxfp4_quantize_weight(w: torch.Tensor, codes, scales, codes_ld: int | None = None, scales_ld: int | None = None,
                             stream=None):
    """MXFP4 codes [N][K/2] and UE8M0 scales [N][K/32] of an fp32 [N][K] matrix (device)."""
    _req(w, torch.float32, "w")
    N, K = w.shape
    codes_ld = K // 2 if codes_ld is None else codes_ld
    scales_ld = K // 32 if scales_ld is None else scales_ld
    _check(_lib.ft_mxfp4_quantize_weight(_p(w), N, K, _p(codes), codes_ld, _p(scales), scales_ld, _s(stream)))


def ft_mxfp4_pack_tiles(codes, codes_ld: int, scales, scales_ld: int, N: int, K: int, tiles, stream=None):
    _check(_lib.ft_mxfp4_pack_tiles(_p(codes), codes_ld, _p(scales), scales_ld, N, K, _p(tiles), _s(stream)))


def ft_mxfp4_pack_umma(codes, codes_ld: int, scales, scales_ld: int, N: int, K: int, tiles, tscale, ts_count: int = 1,
                       stream=None):
    """MXFP4 matrix [N][K] -> FT_LAYOUT_UMMA_TILES plus its fp32 tensor scale in tscale[0:ts_count] (device)."""
    _check(_lib.ft_mxfp4_pack_umma(_p(codes), codes_ld, _p(scales), scales_ld, N, K, _p(tiles), _p(tscale), ts_count,
                                   _s(stream)))


def ft_mxfp8_quantize_weight(w: torch.Tensor, codes, scales, codes_ld: int | None = None, scales_ld: int | None = None,
                             stream=None):
    """MXFP8 codes [N][K] (E4M3) and UE8M0 scales [N][K/32] of an fp32 [N][K] matrix (device)."""
    _req(w, torch.float32, "w")
    N, K = w.shape
    codes_ld = K if codes_ld is None else codes_ld
    scales_ld = K // 32 if scales_ld is None else scales_ld
    _check(_lib.ft_mxfp8_quantize_weight(_p(w), N, K, _p(codes), codes_ld, _p(scales), scales_ld, _s(stream)))


def ft_mxfp8_pack_tiles(codes, codes_ld: int, scales, scales_ld: int, N: int, K: int, tiles, stream=None):
    _check(_lib.ft_mxfp8_pack_tiles(_p(codes), codes_ld, _p(scales), scales_ld, N, K, _p(tiles), _s(stream)))


def ft_moe_layer_decode_workspace_size(T: int, k: int, H: int, I: int) -> int:
    return _lib.ft_moe_layer_decode_workspace_size(T, k, H, I)


def ft_moe_layer_decode(W, logits: torch.Tensor, x: torch.Tensor, k: int, out: torch.Tensor, ws: torch.Tensor,
                        ids=None, w=None, stream=None):
    """Fused decode layer step (route + group + NVFP4 SwiGLU FFN + combine).  ws must start zero-filled."""
    T = x.shape[0]
    desc = W.desc()
    _check(_lib.ft_moe_layer_decode(ctypes.byref(desc), _p(logits), _p(x), T, k, _p(out), _p(ids), _p(w), _p(ws),
                                    ws.numel() * ws.element_size(), _s(stream)))
    return out


def ft_moe_layer_decode_noalloc(W, logits: torch.Tensor, x: torch.Tensor, k: int, out: torch.Tensor, ids=None, w=None,
                                stream=None):
    """Fused decode layer step with the library's built-in scratch (no workspace, nothing allocated)."""
    T = x.shape[0]
    desc = W.desc()
    _check(_lib.ft_moe_layer_decode_noalloc(ctypes.byref(desc), _p(logits), _p(x), T, k, _p(out), _p(ids), _p(w),
                                            _s(stream)))
    return out


def ft_nvfp4_pack_umma(codes, codes_ld: int, scales, scales_ld: int, N: int, K: int, tiles, stream=None):
    _check(_lib.ft_nvfp4_pack_umma(_p(codes), codes_ld, _p(scales), scales_ld, N, K, _p(tiles), _s(stream)))


def ft_moe_prefill_workspace_size(T: int, k: int, E: int, H: int, I: int) -> int:
    return _lib.ft_moe_prefill_workspace_size(T, k, E, H, I)


def ft_moe_expert_ffn_nvfp4_prefill(W, x: torch.Tensor, k: int, offsets, perm, w, out, ws, stream=None, y=None):
    """Prefill expert FFN on the FP4 tensor cores (weights in FT_LAYOUT_UMMA_TILES): the combine into out (bf16
    [T, H]) and/or the per-row expert outputs into y (fp32 [T*k, H]); either may be None, not both."""
    _req(x, torch.bfloat16, "x")
    T = x.shape[0]
    desc = W.desc()
    _check(_lib.ft_moe_expert_ffn_nvfp4_prefill(ctypes.byref(desc), _p(x), T, k, _p(offsets), _p(perm), _p(w), _p(y),
                                                _p(out), _p(ws), ws.numel() * ws.element_size(), _s(stream)))
    return out


# --------------------------------------------------------------------------- layer weights handle

class MoEWeightsHandle:
    """Owns an ft_moe_weights handle: canonical NVFP4 experts repacked into the requested kernel layouts.

    experts: E entries, each ((gate codes ptr, codes_ld, scales ptr, scales_ld, tensor-scale ptr), up, down) of device
    pointers and row strides in bytes.  layout_flags: a set of FT_WEIGHTS_*.
    """

    def __init__(self, experts, H: int, I: int, layout_flags: int, stream=None):
        E = len(experts)
        arr = (ft_nvfp4_expert_desc * E)()
        for e, mats in enumerate(experts):
            for name, m in zip(("gate", "up", "down"), mats):
                setattr(arr[e], name, ft_nvfp4_matrix(*m))
        h = ctypes.c_void_p()
        _check(_lib.ft_moe_weights_create(arr, E, H, I, layout_flags, _s(stream), ctypes.byref(h)))
        self.h, self.E, self.H, self.I, self.flags = h, E, H, I, layout_flags

    def describe(self, layout: int) -> ft_moe_layer_weights:
        d = ft_moe_layer_weights()
        _check(_lib.ft_moe_weights_describe(self.h, layout, ctypes.byref(d)))
        return d

    def close(self):
        if self.h:
            _lib.ft_moe_weights_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------------------- expert-slot cache

class ExpertCacheHandle:
    """Owns an ft_expert_cache handle (host bookkeeping); the pools stay the caller's."""

    def __init__(self, L: int, E: int, S: int, expert_bytes: int, host_ptrs, slots_ptr: int, slot_stride: int,
                 tables_ptr: int):
        arr = (ctypes.c_void_p * (L * E))(*host_ptrs)
        h = ctypes.c_void_p()
        _check(_lib.ft_expert_cache_create(L, E, S, expert_bytes, arr, slots_ptr, slot_stride, tables_ptr,
                                           ctypes.byref(h)))
        self.h, self.L, self.E, self.S = h, L, E, S

    def close(self):
        if self.h:
            _lib.ft_expert_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def lookup(self, layer: int, step: int, ids):
        """Returns (slots, [(expert, slot) misses]) for one token's expert ids (host ints)."""
        n = len(ids)
        c_ids = (ctypes.c_int32 * max(n, 1))(*ids)
        slots = (ctypes.c_int32 * max(n, 1))()
        me = (ctypes.c_int32 * max(n, 1))()
        ms = (ctypes.c_int32 * max(n, 1))()
        nm = ctypes.c_int(0)
        _check(_lib.ft_expert_cache_lookup(self.h, layer, step, c_ids, n, slots, me, ms, ctypes.byref(nm)))
        return [slots[i] for i in range(n)], [(me[i], ms[i]) for i in range(nm.value)]

    def fill(self, layer: int, expert: int, slot: int, stream=None, event=None):
        _check(_lib.ft_expert_cache_fill(self.h, layer, expert, slot, _s(stream),
                                         None if event is None else event.cuda_event))

    def publish(self, layer: int, stream=None):
        _check(_lib.ft_expert_cache_publish(self.h, layer, _s(stream)))

    def stats(self):
        h, m, b = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.ft_expert_cache_stats(self.h, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b)))
        return h.value, m.value, b.value

    def prefetch(self, layer: int, step: int, ids):
        """Install predicted experts (host ints) ahead of the token that uses them; returns the [(expert, slot)] fills
        the caller must enqueue."""
        n = len(ids)
        c_ids = (ctypes.c_int32 * max(n, 1))(*ids)
        fe = (ctypes.c_int32 * max(n, 1))()
        fs = (ctypes.c_int32 * max(n, 1))()
        nf = ctypes.c_int(0)
        _check(_lib.ft_expert_cache_prefetch(self.h, layer, step, c_ids, n, fe, fs, ctypes.byref(nf)))
        return [(fe[i], fs[i]) for i in range(nf.value)]

    def prefetch_stats(self):
        """(experts installed by prefetches, of which a later lookup used)."""
        p, u = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.ft_expert_cache_prefetch_stats(self.h, ctypes.byref(p), ctypes.byref(u)))
        return p.value, u.value

    def inject_fill_failure(self, fill_index: int):
        _check(_lib.ft_expert_cache_inject_fill_failure(self.h, fill_index))

    def resize_plan(self, new_S: int):
        """[[old slot or -1 for each new slot] for each layer] that resize(new_S) would apply now."""
        moves = (ctypes.c_int32 * (self.L * new_S))()
        _check(_lib.ft_expert_cache_resize_plan(self.h, new_S, moves))
        return [[moves[l * new_S + i] for i in range(new_S)] for l in range(self.L)]

    def resize(self, new_S: int, new_slots_ptr: int, new_slot_stride: int, stream=None):
        """Rebuild the cache as new_S slots per layer in a caller-owned device pool (device-to-device moves and the
        publish of every layer's table, on `stream`)."""
        rc = _lib.ft_expert_cache_resize(self.h, new_S, new_slots_ptr, new_slot_stride, _s(stream))
        if rc != FT_ERR_INVALID_ARG:
            # only a rejected argument leaves the old geometry; any later failure leaves the handle on the new pool
            self.S = new_S
        _check(rc)


from .layer import FusedDecodeLayer, LayerWeights, MoEDecodeLayer  # noqa: E402,F401
