"""Argument checks of the C ABI, with no device: every rejected call returns its status before any CUDA call.

Pointers here are placeholders (aligned or deliberately misaligned addresses) that a rejected call never
dereferences; sizes are chosen so that the check under test is the first one to fail.
"""
import ctypes

import pytest

Q = pytest.importorskip("quantized_expert_ffn_06_b300")
L = Q._lib

P = 0x10000          # a placeholder address, 256-byte aligned
MIS = 0x10001        # the same, misaligned
NULL = None


def weights(E=8, H=256, I=128, layout=Q.FT_LAYOUT_DECODE_TILES, n=None, slot_table=False):
    d = Q.ft_moe_layer_weights()
    d.E, d.H, d.I, d.n_weights, d.layout = E, H, I, E if n is None else n, layout
    d.gu_codes, d.gu_codes_stride = P, 2 * I * H * 9 // 16
    d.d_codes, d.d_codes_stride = P, H * I * 9 // 16
    d.gu_scales, d.d_scales = P, P
    d.gu_scales_stride, d.d_scales_stride = 2 * I * H // 16, H * I // 16
    d.tscale, d.tscale_stride = P, 4
    d.expert_to_slot = P if slot_table else None
    return d


def status(rc, want):
    assert rc == want, (rc, L.ft_last_error())


def test_status_strings_and_version():
    for s in (Q.FT_OK, Q.FT_ERR_INVALID_ARG, Q.FT_ERR_CUDA, Q.FT_ERR_UNSUPPORTED, Q.FT_ERR_NO_SLOT, Q.FT_ERR_OOM):
        assert L.ft_status_string(s)
    assert L.ft_version() > 0


@pytest.mark.parametrize("T,E,k", [(-1, 8, 2), (1, 0, 1), (1, 1025, 8), (1, 8, 0), (1, 8, 9), (1, 64, 33)])
def test_route_rejects_bad_sizes(T, E, k):
    status(L.ft_moe_route(P, T, E, k, P, P, NULL), Q.FT_ERR_INVALID_ARG)
    assert b"ft_moe_route" in L.ft_last_error()


def test_route_null_pointers_and_empty_batch():
    status(L.ft_moe_route(NULL, 4, 8, 2, P, P, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_route(P, 4, 8, 2, NULL, P, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_route(NULL, 0, 8, 2, NULL, NULL, NULL), Q.FT_OK)   # nothing to do, nothing launched


@pytest.mark.parametrize("T,E,k", [(-1, 8, 2), (4, 0, 1), (4, 1025, 2), (4, 8, 0), (4, 8, 9), (1 << 30, 8, 8)])
def test_permute_rejects_bad_sizes(T, E, k):
    status(L.ft_moe_permute(P, T, E, k, P, P, P, NULL, P, 1 << 20, NULL), Q.FT_ERR_INVALID_ARG)


def test_permute_null_pointers():
    status(L.ft_moe_permute(P, 4, 8, 2, NULL, P, P, NULL, P, 1 << 20, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_permute(NULL, 4, 8, 2, P, P, P, NULL, P, 1 << 20, NULL), Q.FT_ERR_INVALID_ARG)
    # a large batch needs its workspace
    status(L.ft_moe_permute(P, 4096, 256, 8, P, P, P, NULL, NULL, 0, NULL), Q.FT_ERR_INVALID_ARG)


@pytest.mark.parametrize("kw", [dict(E=0), dict(E=1025), dict(H=128), dict(I=64), dict(n=4)])
def test_weight_descriptors_are_checked(kw):
    W = weights(**kw)
    ws = L.ft_moe_layer_decode_workspace_size(1, 2, W.H, max(W.I, 128))
    status(L.ft_moe_layer_decode(ctypes.byref(W), P, P, 1, 2, P, NULL, NULL, P, ws, NULL), Q.FT_ERR_INVALID_ARG)


def test_layer_decode_argument_checks():
    W = weights()
    ws = L.ft_moe_layer_decode_workspace_size(4, 2, W.H, W.I)
    args = dict(logits=P, x=P, T=4, k=2, out=P, ids=NULL, w=NULL, ws=P, ws_bytes=ws)

    def call(**over):
        a = dict(args, **over)
        return L.ft_moe_layer_decode(ctypes.byref(a.pop("W", W)), a["logits"], a["x"], a["T"], a["k"], a["out"],
                                     a["ids"], a["w"], a["ws"], a["ws_bytes"], NULL)

    status(L.ft_moe_layer_decode(None, P, P, 4, 2, P, NULL, NULL, P, ws, NULL), Q.FT_ERR_INVALID_ARG)
    status(call(W=weights(layout=Q.FT_LAYOUT_UMMA_TILES)), Q.FT_ERR_INVALID_ARG)
    for bad in (dict(T=-1), dict(T=17), dict(k=0), dict(k=9), dict(logits=NULL), dict(x=NULL), dict(out=NULL),
                dict(ids=P), dict(x=MIS), dict(ws=NULL), dict(ws_bytes=ws - 1), dict(ws=P + 16)):
        status(call(**bad), Q.FT_ERR_INVALID_ARG)
    status(call(T=0), Q.FT_OK)


def test_prefill_argument_checks():
    W = weights(layout=Q.FT_LAYOUT_UMMA_TILES)
    ws = L.ft_moe_prefill_workspace_size(64, 2, W.E, W.H, W.I)

    def call(Wd=W, x=P, T=64, k=2, offsets=P, perm=P, w=P, y=NULL, out=P, wsp=P, ws_bytes=ws):
        return L.ft_moe_expert_ffn_nvfp4_prefill(ctypes.byref(Wd), x, T, k, offsets, perm, w, y, out, wsp, ws_bytes,
                                                 NULL)

    status(call(Wd=weights(layout=Q.FT_LAYOUT_DECODE_TILES)), Q.FT_ERR_INVALID_ARG)
    for bad in (dict(T=-1), dict(k=0), dict(k=9), dict(k=2, T=1 << 30), dict(x=NULL), dict(offsets=NULL),
                dict(x=MIS), dict(out=P + 4), dict(wsp=NULL), dict(ws_bytes=ws - 1), dict(wsp=P + 16),
                dict(out=NULL), dict(y=P + 8), dict(w=NULL)):
        status(call(**bad), Q.FT_ERR_INVALID_ARG)
    status(call(T=0), Q.FT_OK)


def test_combine_argument_checks():
    status(L.ft_moe_combine(P, P, P, 4, 2, 6, P, NULL), Q.FT_ERR_INVALID_ARG)     # H not a multiple of 4
    status(L.ft_moe_combine(P, P, P, 4, 0, 8, P, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_combine(NULL, P, P, 4, 2, 8, P, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_combine(MIS, P, P, 4, 2, 8, P, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_moe_combine(NULL, NULL, NULL, 0, 2, 8, NULL, NULL), Q.FT_OK)


def test_quantiser_argument_checks():
    need = L.ft_nvfp4_quantize_workspace_size(16, 256)
    status(L.ft_nvfp4_quantize_weight(P, 16, 250, P, 125, P, 16, P, P, need, NULL), Q.FT_ERR_INVALID_ARG)  # K % 16
    status(L.ft_nvfp4_quantize_weight(NULL, 16, 256, P, 128, P, 16, P, P, need, NULL), Q.FT_ERR_INVALID_ARG)
    status(L.ft_nvfp4_quantize_weight(P, 16, 256, P, 127, P, 16, P, P, need, NULL), Q.FT_ERR_INVALID_ARG)  # ld < K/2
    status(L.ft_nvfp4_quantize_act(P, 4, 250, P, P, NULL), Q.FT_ERR_INVALID_ARG)


def test_no_alloc_decode_argument_checks_come_before_any_cuda_call():
    """The entry point without a workspace rejects bad arguments before it looks up its scratch (a CUDA call)."""
    W = weights()

    def call(**over):
        a = dict(dict(logits=P, x=P, T=4, k=2, out=P, ids=NULL, w=NULL), **over)
        return L.ft_moe_layer_decode_noalloc(ctypes.byref(a.pop("W", W)), a["logits"], a["x"], a["T"], a["k"], a["out"],
                                             a["ids"], a["w"], NULL)

    status(L.ft_moe_layer_decode_noalloc(None, P, P, 4, 2, P, NULL, NULL, NULL), Q.FT_ERR_INVALID_ARG)
    status(call(W=weights(layout=Q.FT_LAYOUT_UMMA_TILES)), Q.FT_ERR_INVALID_ARG)
    for bad in (dict(T=-1), dict(T=17), dict(k=0), dict(k=9), dict(logits=NULL), dict(x=NULL), dict(out=NULL),
                dict(ids=P), dict(w=P), dict(x=MIS), dict(logits=MIS)):
        status(call(**bad), Q.FT_ERR_INVALID_ARG)
    # T*k*I beyond the built-in scratch
    status(call(W=weights(E=64, I=1024), T=16, k=32), Q.FT_ERR_INVALID_ARG)
    assert b"scratch" in L.ft_last_error()
    status(call(T=0), Q.FT_OK)


def test_mxfp4_argument_checks():
    q = L.ft_mxfp4_quantize_weight
    status(q(P, 16, 250, P, 128, P, 8, NULL), Q.FT_ERR_INVALID_ARG)       # K not a multiple of 32
    status(q(NULL, 16, 256, P, 128, P, 8, NULL), Q.FT_ERR_INVALID_ARG)
    status(q(P, 16, 256, P, 120, P, 8, NULL), Q.FT_ERR_INVALID_ARG)       # codes_ld < K/2
    status(q(P, 16, 256, P, 136, P, 7, NULL), Q.FT_ERR_INVALID_ARG)       # scales_ld < K/32 (and ld not x16)
    status(q(P, 16, 256, MIS, 128, P, 8, NULL), Q.FT_ERR_INVALID_ARG)     # misaligned codes
    pk = L.ft_mxfp4_pack_tiles
    status(pk(P, 128, P, 8, 15, 256, P, NULL), Q.FT_ERR_INVALID_ARG)     # N not a multiple of 16
    status(pk(P, 128, P, 8, 16, 200, P, NULL), Q.FT_ERR_INVALID_ARG)     # K not a multiple of 128
    status(pk(P, 128, P, 4, 16, 256, P, NULL), Q.FT_ERR_INVALID_ARG)     # scales_ld < K/32
    status(pk(NULL, 128, P, 8, 16, 256, P, NULL), Q.FT_ERR_INVALID_ARG)


def test_mxfp4_umma_pack_arguments():
    """The MXFP4 -> tensor-core tile packing rejects bad sizes, counts, pointers and alignment before any CUDA call."""
    pu = L.ft_mxfp4_pack_umma
    status(pu(P, 128, P, 8, 100, 256, P, P, 1, NULL), Q.FT_ERR_INVALID_ARG)   # N not a multiple of 128
    status(pu(P, 128, P, 8, 128, 200, P, P, 1, NULL), Q.FT_ERR_INVALID_ARG)   # K not a multiple of 128
    status(pu(P, 128, P, 8, 128, 256, P, P, 0, NULL), Q.FT_ERR_INVALID_ARG)   # ts_count < 1
    status(pu(P, 128, P, 8, 128, 256, P, P, 5, NULL), Q.FT_ERR_INVALID_ARG)   # ts_count > 4
    status(pu(P, 128, P, 8, 128, 256, P, NULL, 1, NULL), Q.FT_ERR_INVALID_ARG)  # no tensor-scale pointer
    status(pu(P, 96, P, 8, 128, 256, P, P, 1, NULL), Q.FT_ERR_INVALID_ARG)    # codes_ld < K/2
    status(pu(P, 128, P, 4, 128, 256, P, P, 1, NULL), Q.FT_ERR_INVALID_ARG)   # scales_ld < K/32
    status(pu(MIS, 128, P, 8, 128, 256, P, P, 1, NULL), Q.FT_ERR_INVALID_ARG)  # misaligned codes


def test_layer_decode_takes_mxfp4_tiles_without_tensor_scales():
    """MXFP4 tiles are accepted with no tensor-scale pointer (T = 0: checks only, nothing launched); MXFP4 rows are
    not a layout of the fused step, and NVFP4 tiles still need their tensor scales."""
    W = weights(layout=Q.FT_LAYOUT_MXFP4_DECODE_TILES)
    W.tscale, W.tscale_stride = None, 0
    ws = L.ft_moe_layer_decode_workspace_size(4, 2, W.H, W.I)
    status(L.ft_moe_layer_decode(ctypes.byref(W), P, P, 0, 2, P, NULL, NULL, P, ws, NULL), Q.FT_OK)
    status(L.ft_moe_layer_decode(ctypes.byref(W), P, P, 4, 2, NULL, NULL, NULL, P, ws, NULL), Q.FT_ERR_INVALID_ARG)
    R = weights(layout=Q.FT_LAYOUT_MXFP4_ROWS)
    status(L.ft_moe_layer_decode(ctypes.byref(R), P, P, 0, 2, P, NULL, NULL, P, ws, NULL), Q.FT_ERR_INVALID_ARG)
    N = weights()
    N.tscale = None
    status(L.ft_moe_layer_decode(ctypes.byref(N), P, P, 0, 2, P, NULL, NULL, P, ws, NULL), Q.FT_ERR_INVALID_ARG)


def test_mxfp8_argument_checks():
    q = L.ft_mxfp8_quantize_weight
    status(q(P, 16, 250, P, 256, P, 8, NULL), Q.FT_ERR_INVALID_ARG)       # K not a multiple of 32
    status(q(P, 16, 256, P, 240, P, 8, NULL), Q.FT_ERR_INVALID_ARG)       # codes_ld < K
    status(q(P, 16, 256, MIS, 256, P, 8, NULL), Q.FT_ERR_INVALID_ARG)     # misaligned codes
    pk = L.ft_mxfp8_pack_tiles
    status(pk(P, 256, P, 8, 15, 256, P, NULL), Q.FT_ERR_INVALID_ARG)     # N not a multiple of 16
    status(pk(P, 128, P, 8, 16, 256, P, NULL), Q.FT_ERR_INVALID_ARG)     # codes_ld < K
    W = weights(layout=Q.FT_LAYOUT_MXFP8_DECODE_TILES)
    W.tscale, W.tscale_stride = None, 0
    ws = L.ft_moe_layer_decode_workspace_size(4, 2, W.H, W.I)
    status(L.ft_moe_layer_decode(ctypes.byref(W), P, P, 0, 2, P, NULL, NULL, P, ws, NULL), Q.FT_OK)
