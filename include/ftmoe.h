/*
 * ftmoe.h -- C ABI of the sparse Mixture-of-Experts layer step over NVFP4
 * expert weights, for NVIDIA B300 (sm_103a).
 *
 * The step, as the FreeToken pages state the problem:
 *   router softmax + top-k  ->  token-to-expert permutation  ->  expert SwiGLU
 *   FFN over 4-bit block-quantised weights  ->  routing-weighted combine,
 * plus a VRAM expert-slot cache filled from pinned host memory.
 * Sources (cited per function below):
 *   [P4] page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", paragraph
 *        on the MoE core mechanism (MoE的核心机制): router = linear + softmax,
 *        top-K experts, weighted outputs; each expert an independent FFN;
 *        paragraph on bandwidth-aware storage: hot experts stay in VRAM,
 *        asynchronous cudaMemcpyAsync overlaps transfer with compute.
 *   [P5] page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier MoE
 *        拉回本地": section 设计核心 (global LRU expert cache in VRAM, misses
 *        filled from host memory), sections 实测六款消费级硬件 and 局限 (NVFP4
 *        weights read directly).
 *   [P3] page xxmr.cn/news/175150, section 2.2 (tokens are dispatched to the
 *        few selected experts) and section 2.1 (dequantisation at compute time).
 *
 * NVFP4 (bit level): element codes E2M1 (OCP MX v1.0 FP4: values 0, .5, 1,
 * 1.5, 2, 3, 4, 6 and their negatives), one unsigned E4M3 scale per 16
 * consecutive elements along the reduction dimension, one fp32 scale per
 * tensor.  Packed codes: byte j of a row holds element 2j in its low nibble
 * and element 2j+1 in its high nibble.
 *
 * Conventions for every function:
 *  - Returns ft_status; FT_OK is 0.  ft_last_error() gives a thread-local
 *    message for the last failure.  No C++ exception crosses the ABI and no
 *    kernel traps: data errors found on the device (NaN logits, invalid
 *    scales, a bounded wait that ran out) set bits in a per-device error word
 *    read by ft_device_status().
 *  - Pointers marked (device) are device memory owned by the caller; (host)
 *    is host memory owned by the caller.  The library allocates no device
 *    memory on the hot path: scratch comes from a caller workspace whose size
 *    the matching *_workspace_size() function returns.  Workspaces need
 *    256-byte alignment.
 *  - All device work is enqueued asynchronously on the caller's stream; the
 *    functions do not synchronise unless stated.
 *  - Argument errors (sizes <= 0 where a count is required, k > E, E > 1024,
 *    k > 32, null required pointers, misaligned pointers, too-small
 *    workspace) return FT_ERR_INVALID_ARG before anything is enqueued.
 */
#ifndef FTMOE_H_
#define FTMOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FT_API __attribute__((visibility("default")))
#else
#define FT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ft_stream_t; /* a cudaStream_t; NULL is the legacy default stream */
typedef struct CUevent_st* ft_event_t;   /* a cudaEvent_t */

typedef enum ft_status {
    FT_OK = 0,
    FT_ERR_INVALID_ARG = 1,
    FT_ERR_CUDA = 2,
    FT_ERR_UNSUPPORTED = 3,
    FT_ERR_TIMEOUT = 4,
    FT_ERR_NO_SLOT = 5,
    FT_ERR_OOM = 6,
    FT_ERR_DEVICE = 7
} ft_status;

/* Device error-word bits (ft_device_status). */
#define FT_DEVERR_NAN_LOGIT 0x1u     /* a router logit was NaN or +inf */
#define FT_DEVERR_BAD_SCALE 0x2u     /* an E4M3 scale byte was NaN or had its sign bit set */
#define FT_DEVERR_TIMEOUT 0x4u       /* a bounded device wait gave up */
#define FT_DEVERR_BAD_INDEX 0x8u     /* an expert id / slot / offset was out of range */
#define FT_DEVERR_RANGE 0x10u        /* a value had no exact encoding in the target format (ft_mxfp4_pack_umma) */

FT_API const char* ft_status_string(ft_status s);
/* Message for the last failure on this thread ("" if none).  The pointer stays
 * valid until the next ft_* call on the same thread. */
FT_API const char* ft_last_error(void);
/* Library ABI version, (major << 16) | minor. */
FT_API int ft_version(void);

/* Test hook for failure detection (off by default; affects launches made after
 * the call, from any thread).  site FT_WAIT_SITE_DECODE_H makes the down phase
 * of the fused decode step (ft_moe_layer_decode and the tiled
 * ft_moe_expert_ffn_nvfp4_decode) wait for h words of a tag that no CTA
 * writes; site FT_WAIT_SITE_PREFILL_TOKEN makes the MMA issuer of the
 * tensor-core prefill's gate/up GEMM (ft_moe_expert_ffn_nvfp4_prefill, token
 * tiles resident) wait on a barrier that nothing completes before its first
 * token-tile part.  Every wait of the affected kernel is then bounded by
 * limit_ns (0 < limit_ns <= 2 s): the wait runs out, the kernel sets
 * FT_DEVERR_TIMEOUT, finishes without trapping and its output is unspecified.
 * site FT_WAIT_SITE_NONE restores normal waits with the default 2 s bound
 * (limit_ns ignored). */
#define FT_WAIT_SITE_NONE 0
#define FT_WAIT_SITE_DECODE_H 1
#define FT_WAIT_SITE_PREFILL_TOKEN 2
FT_API ft_status ft_debug_inject_wait_expiry(int site, uint64_t limit_ns);

/* Waits for `stream`, then reads and clears the current device's error word.
 * *err_word receives the FT_DEVERR_* bits; returns FT_ERR_DEVICE if any bit was
 * set, FT_ERR_CUDA if the stream reported a CUDA error, FT_OK otherwise. */
FT_API ft_status ft_device_status(ft_stream_t stream, uint32_t* err_word);

/* ------------------------------------------------------------------------ */
/* Weights of one MoE layer                                                   */
/* ------------------------------------------------------------------------ */

/* Layouts of expert weights in device memory (ft_moe_layer_weights.layout). */
#define FT_LAYOUT_ROWS 0         /* row-major codes [N][K/2] + row-major scales [N][K/16] */
#define FT_LAYOUT_DECODE_TILES 1 /* 16-row tiles for the decode kernels, see ft_nvfp4_pack_tiles() */
#define FT_LAYOUT_UMMA_TILES 2   /* 128x128 blocks for the tensor-core prefill, see ft_nvfp4_pack_umma() */
#define FT_LAYOUT_MXFP4_ROWS 3   /* MXFP4: row-major codes [N][K/2] + row-major UE8M0 scales [N][K/32] */
#define FT_LAYOUT_MXFP4_DECODE_TILES 4 /* MXFP4 16-row tiles for the fused decode, see ft_mxfp4_pack_tiles() */
#define FT_LAYOUT_MXFP8_ROWS 5   /* MXFP8: row-major E4M3 codes [N][K] + row-major UE8M0 scales [N][K/32] */
#define FT_LAYOUT_MXFP8_DECODE_TILES 6 /* MXFP8 16-row tiles for the fused decode, see ft_mxfp8_pack_tiles() */

/* Expert weights of one layer in device memory.  For weight index w (the
 * expert id, or its cache slot when expert_to_slot is given):
 *  layout FT_LAYOUT_ROWS
 *   gate/up  codes  gu_codes  + w*gu_codes_stride  : [2I][H/2] bytes; row 2i is
 *                   gate row i, row 2i+1 is up row i (interleaved so that one
 *                   tile holds both halves of each SwiGLU pair)
 *            scales gu_scales + w*gu_scales_stride : [2I][H/16] E4M3 bytes
 *   down     codes  d_codes   + w*d_codes_stride   : [H][I/2]
 *            scales d_scales  + w*d_scales_stride  : [H][I/16]
 *  layout FT_LAYOUT_UMMA_TILES (codes and scales together; scale pointers unused)
 *   gate/up  gu_codes + w*gu_codes_stride : the [2I][H] matrix above packed by
 *            ft_nvfp4_pack_umma() ((2I/128)*(H/128) blocks of 9216 bytes)
 *   down     d_codes  + w*d_codes_stride  : the [H][I] matrix packed likewise
 *  layout FT_LAYOUT_DECODE_TILES (codes and scales together; scale pointers unused)
 *   gate/up  gu_codes + w*gu_codes_stride : the [2I][H] matrix above packed by
 *            ft_nvfp4_pack_tiles() (2I*H*9/16 bytes)
 *   down     d_codes  + w*d_codes_stride  : the [H][I] matrix packed likewise
 *  layout FT_LAYOUT_MXFP4_ROWS: as FT_LAYOUT_ROWS with UE8M0 scales, one per 32
 *            elements: gu_scales [2I][H/32], d_scales [H][I/32]; no tensor scale
 *  layout FT_LAYOUT_MXFP4_DECODE_TILES (codes and scales together): the same
 *            matrices packed by ft_mxfp4_pack_tiles() (2I*H*17/32 and H*I*17/32
 *            bytes); no tensor scale
 *  layout FT_LAYOUT_MXFP8_ROWS / FT_LAYOUT_MXFP8_DECODE_TILES: as the MXFP4 ones
 *            with one E4M3 byte per element (codes [N][K]; tiles of 2I*H*33/32
 *            and H*I*33/32 bytes, see ft_mxfp8_pack_tiles()); no tensor scale
 *  NVFP4 layouts
 *   tensor scales  tscale + w*tscale_stride : float {gate, up, down}
 *   (MX layouts have none: tscale may be NULL and is not read)
 *   gu_sf_tiled / d_sf_tiled (optional, prefill only): scales rearranged for the
 *            block-scaled tensor cores, strides gu_sf_tiled_stride / d_sf_tiled_stride.
 * Strides are in bytes (tscale_stride in floats).  Every base address and
 * stride must be a multiple of 16.  expert_to_slot (device, optional, [E]
 * int32) maps an expert id to its weight index; ids mapping to a negative or
 * out-of-range index set FT_DEVERR_BAD_INDEX and contribute zeros.
 * Sizes: 1 <= E <= 1024 experts; H a multiple of 256; I a multiple of 128. */
typedef struct ft_moe_layer_weights {
    int32_t E, H, I, n_weights; /* n_weights: number of weight indices (E, or cache slots) */
    int32_t layout;             /* FT_LAYOUT_* */
    int32_t reserved0;
    const uint8_t* gu_codes;
    int64_t gu_codes_stride;
    const uint8_t* gu_scales;
    int64_t gu_scales_stride;
    const uint8_t* d_codes;
    int64_t d_codes_stride;
    const uint8_t* d_scales;
    int64_t d_scales_stride;
    const float* tscale;
    int64_t tscale_stride;
    const int32_t* expert_to_slot;
    const uint8_t* gu_sf_tiled;
    int64_t gu_sf_tiled_stride;
    const uint8_t* d_sf_tiled;
    int64_t d_sf_tiled_stride;
} ft_moe_layer_weights;

/* The layer weights handle: canonical NVFP4 expert matrices repacked, once,
 * into the layouts the kernels read.  [P4 MoE core mechanism: each expert an
 * independent FFN; P5 NVFP4 weights]
 * One canonical matrix [N][K] (device memory, caller-owned): codes [N][K/2]
 * with element 2j in the low nibble of byte j, row stride codes_ld bytes
 * (16-byte aligned base, codes_ld a multiple of 16); E4M3 scales [N][K/16],
 * row stride scales_ld bytes, one per 16 consecutive elements of a row; and a
 * pointer to its fp32 tensor scale.  An expert is gate [I][H], up [I][H] and
 * down [H][I]. */
typedef struct ft_nvfp4_matrix {
    const uint8_t* codes;
    int64_t codes_ld;
    const uint8_t* scales;
    int64_t scales_ld;
    const float* tensor_scale;
} ft_nvfp4_matrix;
typedef struct ft_nvfp4_expert_desc {
    ft_nvfp4_matrix gate, up, down;
} ft_nvfp4_expert_desc;
#define FT_WEIGHTS_ROWS (1 << FT_LAYOUT_ROWS)
#define FT_WEIGHTS_DECODE_TILES (1 << FT_LAYOUT_DECODE_TILES)
#define FT_WEIGHTS_UMMA_TILES (1 << FT_LAYOUT_UMMA_TILES)
typedef struct ft_moe_weights ft_moe_weights;
/* experts (host) [E]: the canonical matrices of experts 0..E-1.  layout_flags: a
 * non-empty set of FT_WEIGHTS_*.  The handle allocates device memory for the
 * requested layouts (plus per-expert tensor scales {gate, up, down, 0}), copies
 * and repacks the bytes on `stream` and returns once that work has finished, so
 * the canonical matrices may be freed right after.  Repacking only moves bytes:
 * kernels reading the handle compute on exactly the caller's codes and scales.
 * Sizes: 1 <= E <= 1024, H a multiple of 256, I a multiple of 128.  Errors:
 * FT_ERR_INVALID_ARG (checked before any CUDA call), FT_ERR_OOM (device
 * allocation), FT_ERR_CUDA (a copy failed); *out is NULL on any error. */
FT_API ft_status ft_moe_weights_create(const ft_nvfp4_expert_desc* experts, int E, int H, int I, int layout_flags,
                                       ft_stream_t stream, ft_moe_weights** out);
/* Fills *desc (host) with the descriptor of the handle's copy in `layout`
 * (FT_LAYOUT_*), ready for the FFN and layer calls; FT_ERR_INVALID_ARG if the
 * handle holds no copy in that layout.  The descriptor stays valid until
 * ft_moe_weights_destroy. */
FT_API ft_status ft_moe_weights_describe(const ft_moe_weights* w, int layout, ft_moe_layer_weights* desc);
/* Frees the handle and its device memory (no kernel may still be reading it). */
FT_API ft_status ft_moe_weights_destroy(ft_moe_weights* w);

/* ------------------------------------------------------------------------ */
/* Router                                                                     */
/* ------------------------------------------------------------------------ */

/* [P4 MoE core mechanism] Softmax over E router logits and top-k selection.
 *   logits (device) fp32 [T][E], row-major.
 *   ids    (device) int32 [T][k]: expert ids by decreasing logit; equal logits
 *          go to the lower expert index.  Selection compares the fp32 logits.
 *   w      (device) fp32 [T][k]: exp(l_j - max) / sum over the k selected,
 *          i.e. the softmax restricted to the selected experts and
 *          renormalised to sum to 1.  A row whose logits are all -inf gets 1/k.
 * NaN or +inf logits set FT_DEVERR_NAN_LOGIT (outputs of that row are then
 * unspecified).  1 <= k <= min(E, 32), E <= 1024, T >= 0. */
FT_API ft_status ft_moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, ft_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Permutation                                                                */
/* ------------------------------------------------------------------------ */

FT_API size_t ft_moe_permute_workspace_size(int T, int E, int k);

/* [P3 §2.2, P4] Groups the T*k (token, slot) pairs by expert: a stable
 * counting sort of f = t*k + j by ids[f].
 *   offsets (device) int32 [E+1]: exclusive prefix sum of the per-expert
 *           counts; expert e owns permuted rows [offsets[e], offsets[e+1]).
 *   perm    (device) int32 [T*k]: perm[p] = f of the p-th permuted row; rows of
 *           one expert are in increasing f.
 *   inv     (device) int32 [T*k]: inv[f] = p.
 *   active  (device, optional) int32 [E+1]: active[0] = number of experts with
 *           at least one row, active[1..] their ids ascending.
 * Result is bit-identical to the sequential definition for any launch.
 * ids out of [0, E) set FT_DEVERR_BAD_INDEX. */
FT_API ft_status ft_moe_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* perm, int32_t* inv,
                         int32_t* active, void* ws, size_t ws_bytes, ft_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert FFN                                                                 */
/* ------------------------------------------------------------------------ */

FT_API size_t ft_moe_decode_workspace_size(int T, int k, int H, int I);

/* [P4 MoE core mechanism; P3 §2.1; P5 NVFP4] Decode expert FFN, bf16
 * activations, NVFP4 weights dequantised in registers, fp32 accumulation:
 * for each permuted row p of expert e (token t = perm[p] / k):
 *   g = Wg x_t, u = Wu x_t, h = bf16(silu(g) * u), y_p = Wd h.
 *   x       (device) bf16 [T][H].
 *   offsets, perm, active: from ft_moe_permute.
 *   y       (device, optional) fp32 [T*k][H]: per-row expert outputs.
 *   out     (device, optional) bf16 [T][H]: if given (with inv and w), the
 *           combine is applied: out[t] = bf16(sum_j w[t][j] * y[inv[t*k+j]]).
 * At least one of y, out.  Intended for small T (up to a few dozen tokens);
 * works for any T. */
FT_API ft_status ft_moe_expert_ffn_nvfp4_decode(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k,
                                         const int32_t* offsets, const int32_t* perm, const int32_t* active,
                                         const int32_t* inv, const float* w, float* y, uint16_t* out, void* ws,
                                         size_t ws_bytes, ft_stream_t stream);

/* Fused decode layer step for up to 16 tokens, weights in FT_LAYOUT_DECODE_TILES
 * (NVFP4), FT_LAYOUT_MXFP4_DECODE_TILES (MXFP4) or FT_LAYOUT_MXFP8_DECODE_TILES
 * (MXFP8, the same scale handling; exact unless a block is more than 2^15
 * below the largest of its row's K-block):
 * router top-k (same selection and weights as ft_moe_route), grouping by
 * expert (same order as ft_moe_permute), the SwiGLU expert FFN on the 4-bit
 * weights and the weighted combine, in one launch of one CTA per SM.
 * [P4 MoE core mechanism; P3 §2.1; P5 NVFP4, and MXFP4 in its limits]
 * MXFP4: per 128-element K-block, each 16-row tile row takes the largest of
 * its four block exponents r; the codes are scaled by 2^(x - r) in f16 before
 * the tensor-core product and the fp32 partial by 2^r after it -- exact unless
 * a block is more than 2^22 below the largest of its row's K-block, whose bits
 * below f16's subnormal range are then lost.
 *   logits (device) fp32 [T][E]; x (device) bf16 [T][H], 16-byte aligned.
 *   out    (device) bf16 [T][H]: out[t] = bf16(sum_j w[t][j] * y_{t,j}), the
 *          sum over a token's experts taken in slot order j, fp32.
 *   ids, w (device, optional, both or neither) [T][k]: the routing result.
 *   ws: ft_moe_layer_decode_workspace_size(T, k, H, I) bytes, 256-byte
 *       aligned, ZERO-FILLED before its first use.  Its first 8 bytes hold a
 *       64-bit call counter (each call adds one per CTA) from which the tag of
 *       the h values the gate/up phase hands to the down phase is derived (a
 *       32-bit tag that skips 0 and repeats only after 2^32 - 1 calls); calls
 *       sharing a workspace must not overlap on the device.  A call whose wait
 *       ran out (FT_DEVERR_TIMEOUT) leaves the workspace consistent.
 * 0 <= T <= 16, 1 <= k <= min(E, 32).  The activations are staged in shared
 * memory as f16: T'*(H+32) + T'*k*(I+32) halves must fit 120 KB for a launch
 * of T' tokens.  A larger batch runs as consecutive launches over the largest
 * token chunks that fit (tokens are independent here, so the result is the
 * same); FT_ERR_UNSUPPORTED only if a single token does not fit (then use the
 * separate calls with FT_LAYOUT_ROWS).
 * The launch allows programmatic dependent launch: the kernel reads no input
 * before the preceding kernel in the stream has completed.  Its grid is one CTA
 * per SM and the phases hand over through global memory, so every CTA must be
 * able to run at once: a kernel on another stream holding SMs for longer than
 * the wait bound (2 s) makes the call report FT_DEVERR_TIMEOUT. */
FT_API size_t ft_moe_layer_decode_workspace_size(int T, int k, int H, int I);
FT_API ft_status ft_moe_layer_decode(const ft_moe_layer_weights* W, const float* logits, const uint16_t* x, int T,
                                     int k, uint16_t* out, int32_t* ids, float* w, void* ws, size_t ws_bytes,
                                     ft_stream_t stream);

/* The fused decode layer step above, for callers that cannot allocate device
 * memory.  (No counterpart in the pages: this is a deployment convenience.)
 * Typical such callers are:
 *  - a plugin that its host hands only input and output buffers, with no way
 *    to ask for a workspace;
 *  - an application whose own pool allocator owns all device memory and
 *    forbids other components from calling cudaMalloc;
 *  - a latency-critical decode loop that must not take the allocator's locks
 *    and implicit synchronisation.
 * Arguments as ft_moe_layer_decode, without ws: the scratch (the call counter
 * and the h hand-off words, 256 + 4*T*k*I bytes) lives in a device array
 * inside the library of FT_NOALLOC_DECODE_MAX_SCRATCH bytes.  Every GPU that
 * loads the library holds it until the process exits.
 *  - T*k*I > 262144 returns FT_ERR_INVALID_ARG before anything is enqueued.
 *  - The function allocates nothing: no cudaMalloc, no cudaFree, no
 *    allocating library call.  Each call first clears the part of the array it
 *    uses with cudaMemsetAsync on `stream`, so it never depends on what
 *    earlier calls left there.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current.  Make that first call
 *    before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other threads, or two in flight on different streams) race and
 *    give wrong results.  Serialise them. */
#define FT_NOALLOC_DECODE_MAX_SCRATCH ((1u << 20) + 256u)
FT_API ft_status ft_moe_layer_decode_noalloc(const ft_moe_layer_weights* W, const float* logits, const uint16_t* x,
                                             int T, int k, uint16_t* out, int32_t* ids, float* w, ft_stream_t stream);

FT_API size_t ft_moe_prefill_workspace_size(int T, int k, int E, int H, int I);

/* [P4 MoE core mechanism; P5 NVFP4; P3 §2.1] Prefill expert FFN and combine on
 * the block-scaled FP4 tensor cores (tcgen05.mma kind::mxf4nvf4, TMEM
 * accumulators).  The FP4 MMA needs FP4 on both sides, so activations are
 * NVFP4 too ("A4"): x rows and h rows are quantised with unit tensor scale,
 * per 16 elements along the reduction dimension:
 *   g = Wg q(x_t), u = Wu q(x_t), h = bf16(silu(g) * u), y_p = Wd q(h),
 *   out[t] = bf16( sum_j w[t][j] * y_{inv[t*k+j]} ), fp32 (order of the
 *   additions not fixed: fp32 atomics).
 *   W (device) weights in FT_LAYOUT_UMMA_TILES; H a multiple of 128, I a
 *          multiple of 128.  With a slot table (expert_to_slot), an expert
 *          with rows whose slot is outside [0, n_weights) sets
 *          FT_DEVERR_BAD_INDEX and its rows contribute nothing.
 *   x (device) bf16 [T][H], 16-byte aligned; offsets, perm (device) from
 *   ft_moe_permute; w (device) fp32 [T][k] routing weights (needed with out).
 *   y (device, optional) fp32 [T*k][H], 16-byte aligned: y_p of every permuted
 *          row p (tensor scale applied, no routing weight).
 *   out (device, optional) bf16 [T][H], 8-byte aligned: the combine.  At least
 *          one of y, out.  A misaligned x, y or out is FT_ERR_INVALID_ARG.
 *   ws: ft_moe_prefill_workspace_size(T, k, E, H, I) bytes, 256-byte aligned
 *       (per-expert tile offsets, quantised x and h tiles, an fp32 output
 *       accumulator); no initial content needed.
 * Each expert's rows are padded to whole 128-row tiles; the padding rows of a
 * tile hold whatever the workspace held and never reach the outputs.
 * offsets that do not partition [0, T*k) in order (offsets[0] = 0, non-
 * decreasing, offsets[E] = T*k) set FT_DEVERR_BAD_INDEX; no expert row is then
 * computed and out is all zeros. */
FT_API ft_status ft_moe_expert_ffn_nvfp4_prefill(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k,
                                                 const int32_t* offsets, const int32_t* perm, const float* w, float* y,
                                                 uint16_t* out, void* ws, size_t ws_bytes, ft_stream_t stream);

/* [P4 MoE core mechanism] Routing-weighted combine:
 * out[t][n] = bf16( sum_{j<k} w[t][j] * y[inv[t*k+j]][n] ), fp32, j order.
 *   y (device) fp32 [T*k][H]; inv, w as above; out (device) bf16 [T][H].
 * An inv entry outside [0, T*k) sets FT_DEVERR_BAD_INDEX and adds nothing. */
FT_API ft_status ft_moe_combine(const float* y, const int32_t* inv, const float* w, int T, int k, int H, uint16_t* out,
                         ft_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert-slot cache                                                          */
/* ------------------------------------------------------------------------ */

/* [P5 设计核心, second principle; P4 bandwidth-aware storage] A VRAM cache of
 * experts per layer with LRU replacement, filled from pinned host memory by
 * cudaMemcpyAsync on a side stream.  Adjacent tokens route to overlapping
 * experts, so most routed accesses hit and only misses cross PCIe.
 * Policy (the pages say only "global LRU"): one cache of S slots per layer,
 * initially empty; a token's experts are visited in ascending id; a hit
 * refreshes the expert's stamp to `step`; a miss takes the lowest free slot,
 * else evicts the slot with the oldest stamp among experts the token does not
 * select (lower slot on a tie).
 * Memory is the caller's:
 *   host_experts (host) [L*E] pointers, expert e of layer l at [l*E + e]:
 *       expert_bytes each, in pinned host memory, laid out exactly as a slot.
 *   slots (device) the slot pool: slot s of layer l at slots + (l*S + s)*slot_stride
 *       (slot_stride >= expert_bytes, slot_stride and slots 256-byte aligned).
 *   tables (device) int32 [L][E]: expert -> slot or -1, written by _publish; give
 *       tables + l*E as expert_to_slot of layer l's ft_moe_layer_weights.
 * The handle is host memory, freed by ft_expert_cache_destroy.  The first
 * _publish makes a small pinned staging area; create and lookup touch no device.
 * Calls on one handle are serialised by an internal lock. */
typedef struct ft_expert_cache ft_expert_cache;
FT_API ft_status ft_expert_cache_create(int L, int E, int S, size_t expert_bytes, const void* const* host_experts,
                                        void* slots, size_t slot_stride, int32_t* tables, ft_expert_cache** out);
FT_API ft_status ft_expert_cache_destroy(ft_expert_cache* cache);
/* One token's expert ids (host, n <= S, distinct, in [0, E)).  slots_out[i]
 * (host) receives the slot of ids[i]; the misses, which the caller must fill
 * before the layer reads them, are miss_experts[0..*n_miss) / miss_slots
 * (host, room for n), ascending expert id.  Pure host bookkeeping. */
FT_API ft_status ft_expert_cache_lookup(ft_expert_cache* cache, int layer, int64_t step, const int32_t* ids, int n,
                                        int32_t* slots_out, int32_t* miss_experts, int32_t* miss_slots, int* n_miss);
/* Enqueues the copy of expert `expert` of `layer` from its pinned host source
 * into `slot` on copy_stream, then records `done` (optional) there.  A copy
 * that cannot be enqueued returns FT_ERR_CUDA (nothing recorded). */
FT_API ft_status ft_expert_cache_fill(ft_expert_cache* cache, int layer, int expert, int slot, ft_stream_t copy_stream,
                                      ft_event_t done);
/* Enqueues on `stream` the copy of layer `layer`'s expert -> slot table into
 * tables + layer*E (from a pinned ring of 4 staging copies per layer; a ring
 * entry still in flight is waited for on the host). */
FT_API ft_status ft_expert_cache_publish(ft_expert_cache* cache, int layer, ft_stream_t stream);
/* [P4 bandwidth-aware storage: experts predicted from the gate outputs are
 * fetched ahead, asynchronously, so the transfer overlaps the computation]
 * Installs the predicted experts ids (host, n <= E; repeats ignored) of layer
 * `layer` ahead of the token that will use them.  Policy (the pages give
 * none): ids are visited in ascending order; one already resident is left as
 * it is (a prediction is not a use); otherwise it takes the lowest free slot,
 * else the slot with the oldest stamp older than `step` (lower slot on a tie)
 * whose expert is not among `ids`, so neither a predicted expert nor one
 * stamped `step` -- the current token's, which a kernel may still be reading --
 * is displaced; when no slot qualifies the id is skipped.  An installed
 * expert gets stamp step - 1.  fill_experts / fill_slots (host, room for n)
 * receive the copies the caller must enqueue (ft_expert_cache_fill) before a
 * layer reads them, ascending expert id; *n_fill their count.  The caller
 * orders those copies after every kernel that may still read a displaced slot
 * (experts stamped below `step`: earlier tokens' layer kernels), e.g. by
 * enqueueing them on a copy stream only once this layer's previous kernel has
 * completed.  Pure host bookkeeping. */
FT_API ft_status ft_expert_cache_prefetch(ft_expert_cache* cache, int layer, int64_t step, const int32_t* ids, int n,
                                          int32_t* fill_experts, int32_t* fill_slots, int* n_fill);
/* Experts installed by prefetches since creation, and how many of those a later
 * lookup used before they left the cache. */
FT_API ft_status ft_expert_cache_prefetch_stats(ft_expert_cache* cache, int64_t* prefetched, int64_t* used);
/* Counters since creation: hit and miss accesses, bytes enqueued by fills. */
FT_API ft_status ft_expert_cache_stats(ft_expert_cache* cache, int64_t* hits, int64_t* misses, int64_t* bytes_filled);
/* [P5 设计核心, third mechanism] Elastic resize at a safe point: the cache
 * becomes new_S slots per layer in the pool new_slots (device, caller-owned,
 * slot s of layer l at new_slots + (l*new_S + s)*new_slot_stride; alignment as
 * in _create), rebuilt from the experts already in VRAM with no host reload.
 * Policy (the pages give none): per layer, all resident experts are kept if
 * they fit, else the new_S most recently used (lower old slot on equal
 * stamps); kept experts take new slots 0.. in ascending old-slot order and keep
 * their stamps; the others leave the cache.  Counters are unchanged.
 * The moves run on `stream` (a copy kernel between disjoint pools, ordered
 * cudaMemcpyAsync in place), followed by the publish of every layer's table
 * on `stream`.  Safe point: every fill into the
 * old pool and every kernel reading it must be ordered before `stream`; the
 * old pool must stay allocated until `stream` passes this call.  new_slots may
 * overlap the old pool only as a shrink in place (same base and stride,
 * new_S <= S); any other overlap is FT_ERR_INVALID_ARG.  FT_ERR_INVALID_ARG
 * is returned before any change; every other error leaves the handle on the
 * new pool: if a move cannot be enqueued (FT_ERR_CUDA) the cache is empty and
 * nothing is published; if a table publish fails the moves stand.  Either way
 * publish each layer before its next use.
 * A lookup after a shrink needs n <= new_S. */
FT_API ft_status ft_expert_cache_resize(ft_expert_cache* cache, int new_S, void* new_slots, size_t new_slot_stride,
                                        ft_stream_t stream);
/* The plan ft_expert_cache_resize(new_S) would apply now, without applying it
 * (pure host): moves (host) int32 [L][new_S], the old slot whose expert goes to
 * each new slot, -1 for a free one. */
FT_API ft_status ft_expert_cache_resize_plan(ft_expert_cache* cache, int new_S, int32_t* moves);
/* Test hook: the slot copy with 0-based index `fill_index` (counting every
 * fill call and every copy a resize enqueues on this handle: one per moved
 * slot in place, one per launch of up to 256 moves between disjoint pools)
 * returns FT_ERR_CUDA without enqueuing it; -1 turns the hook off. */
FT_API ft_status ft_expert_cache_inject_fill_failure(ft_expert_cache* cache, int64_t fill_index);

/* ------------------------------------------------------------------------ */
/* Quantisation and synthetic weights                                         */
/* ------------------------------------------------------------------------ */

FT_API size_t ft_nvfp4_quantize_workspace_size(int64_t N, int64_t K);

/* NVFP4 weight quantiser, fp32 arithmetic with IEEE division:
 *   s_t = amax / 2688 (1 if that is 0); per 16-block: sb = E4M3_rn_sat(amax_b /
 *   6 / s_t), eff = e4m3(sb) * s_t, code = E2M1_rn_sat(w / eff) (0 when eff is
 *   0; a negative value that rounds to 0 is code 0).
 *   w (device) fp32 [N][K]; codes (device) rows of K/2 bytes at byte stride
 *   codes_ld; scales (device) rows of K/16 bytes at stride scales_ld;
 *   tensor_scale (device) one float.  K a multiple of 32. */
FT_API ft_status ft_nvfp4_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                   uint8_t* scales, int64_t scales_ld, float* tensor_scale, void* ws,
                                   size_t ws_bytes, ft_stream_t stream);

/* NVFP4 activation quantiser with unit tensor scale (bf16 input): per
 * 16-block sb = E4M3_rn_sat(amax_b / 6), code = E2M1_rn_sat(x / e4m3(sb)).
 *   x (device) bf16 [T][K]; codes (device) [T][K/2]; scales (device) [T][K/16]
 *   row-major.  K a multiple of 32. */
FT_API ft_status ft_nvfp4_quantize_act(const uint16_t* x, int64_t T, int64_t K, uint8_t* codes, uint8_t* scales,
                                ft_stream_t stream);

/* Packs a row-major NVFP4 matrix [N][K] (codes [N][K/2] at byte stride
 * codes_ld, scales [N][K/16] at stride scales_ld) into FT_LAYOUT_DECODE_TILES:
 * N/16 tiles of 16*K*9/16 bytes.  Within a tile, per 128-element K-block kb
 * (K/128 of them): 1024 code bytes, byte i of piece q (bytes 16q..16q+15 of the
 * row's 64 bytes in that block) of row 8h+g at kb*1024 + h*512 + (g*4+q)*16 + i;
 * then, after all code blocks, 128 scale bytes per K-block: scale 2q+b of the
 * block's eight for row 8h+g at (K/128)*1024 + kb*128 + (g*4+q)*4 + 2h + b.
 * Warp lane L = 4g+q thus reads the 16 code bytes at L*16 and 512 + L*16 (rows
 * g and g+8) and the scale word at L*4: consecutive lanes, consecutive
 * addresses, no bank conflicts.  N a multiple of 16, K a multiple of 128.
 * All pointers (device). */
FT_API ft_status ft_nvfp4_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                                     int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream);

/* Packs a row-major NVFP4 matrix [N][K] (codes [N][K/2] at byte stride
 * codes_ld, scales [N][K/16] at stride scales_ld) into FT_LAYOUT_UMMA_TILES:
 * (N/128)*(K/128) blocks of 9216 bytes, block (rt, ks) of rows 128*rt.. and
 * K 128*ks.. at (rt*(K/128) + ks)*9216.  Within a block, code byte b (0..63) of
 * row r at (b/16)*2048 + (r/8)*128 + (r%8)*16 + b%16 (the tensor core's
 * K-major no-swizzle layout: 8-row x 16-byte core matrices) and scale j (0..7)
 * of row r at 8192 + (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4 (the scale-factor
 * layout moved to TMEM by tcgen05.cp .32x128b.warpx4).  N and K multiples of
 * 128.  All pointers (device). */
FT_API ft_status ft_nvfp4_pack_umma(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                                    int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream);

/* MXFP4 weight quantiser [P5 limits: MXFP4 among the weight formats; the OCP
 * Microscaling v1.0 format]: fp32 w [N][K] (device, row-major, 16-byte
 * aligned) -> E2M1 codes [N][K/2] (element 2j in the low nibble of byte j; row
 * stride codes_ld, a multiple of 16, >= K/2) and UE8M0 scales [N][K/32] (row
 * stride scales_ld >= K/32).  Per 32-element block: X = floor(log2(amax)) - 2
 * clamped to [-127, 127] (-127 for an all-zero block), scale byte X + 127,
 * code = E2M1 round-to-nearest-even of v / 2^X saturating at 6, -0 stored as
 * +0.  NaN or inf inputs set FT_DEVERR_BAD_SCALE.  K a multiple of 32.  No
 * workspace; asynchronous on `stream`. */
FT_API ft_status ft_mxfp4_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                          uint8_t* scales, int64_t scales_ld, ft_stream_t stream);

/* Packs a row-major MXFP4 matrix [N][K] (codes [N][K/2] at byte stride
 * codes_ld, scales [N][K/32] at stride scales_ld) into
 * FT_LAYOUT_MXFP4_DECODE_TILES: N/16 tiles of 16*K*17/32 bytes.  Within a
 * tile, per 128-element K-block kb: the 1024 code bytes exactly as
 * ft_nvfp4_pack_tiles() places them; then, after all code blocks, 64 scale
 * bytes per K-block: the scale of block 4kb+q of row 8h+g at
 * (K/128)*1024 + kb*64 + (g*4+q)*2 + h.  Warp lane L = 4g+q thus holds the
 * codes of exactly one block of rows g and g+8 and reads their two scale bytes
 * at L*2.  N a multiple of 16, K a multiple of 128.  All pointers (device). */
FT_API ft_status ft_mxfp4_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                                     int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream);

/* MXFP4 weights for the tensor-core prefill [P5 limits: MXFP4 among the
 * weight formats]: packs a row-major MXFP4 matrix [N][K] (codes [N][K/2] at
 * byte stride codes_ld, UE8M0 scales [N][K/32] at stride scales_ld) into
 * FT_LAYOUT_UMMA_TILES, the layout of ft_nvfp4_pack_umma(), and writes the
 * matrix's fp32 tensor scale to tscale[0 .. ts_count-1] (device).  The E2M1
 * codes are copied unchanged; the scale 2^(s-127) of each 32-element block
 * becomes the E4M3 scale 2^(s-s0) of both of its 16-element halves, with
 * s0 = (largest s over blocks holding a non-zero code) - 8 and tensor scale
 * 2^(s0-127).  Powers of two from 2^-9 to 2^8 are exact E4M3 values, so every
 * product code x scale x tensor scale equals the MX one exactly when the
 * matrix's non-zero blocks span at most 17 octaves (s >= largest s - 17).  A
 * block beyond that sets FT_DEVERR_RANGE (its scale is written as 0); a scale
 * byte of 255 (NaN) sets FT_DEVERR_BAD_SCALE, is written as 0 and does not
 * count in s0.  Blocks whose codes are all
 * zero get scale 0.  With no non-zero block the tensor scale is 1.  Three
 * launches on `stream`; tscale[0] serves as their scratch word until the
 * last.  N and K multiples of 128, 1 <= ts_count <= 4; codes and tiles
 * 16-byte aligned, codes_ld a multiple of 16, tscale 4-byte aligned. */
FT_API ft_status ft_mxfp4_pack_umma(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                                    int64_t N, int64_t K, uint8_t* tiles, float* tscale, int ts_count,
                                    ft_stream_t stream);

/* MXFP8 weight quantiser [P5 limits: FP8 among the weight formats; the OCP
 * Microscaling v1.0 MXFP8 format]: as ft_mxfp4_quantize_weight with E4M3
 * elements: X = floor(log2(amax)) - 8 clamped to [-127, 127], code = E4M3
 * round-to-nearest-even of v / 2^X saturating at 448 (sign in bit 7, -0 stored
 * as +0), one byte per element: codes [N][K] at row stride codes_ld (a
 * multiple of 16, >= K). */
FT_API ft_status ft_mxfp8_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                          uint8_t* scales, int64_t scales_ld, ft_stream_t stream);

/* Packs a row-major MXFP8 matrix [N][K] (codes [N][K], scales [N][K/32]) into
 * FT_LAYOUT_MXFP8_DECODE_TILES: N/16 tiles of 16*K*33/32 bytes.  Within a tile,
 * per 128-element K-block kb: 2048 code bytes, the 32 bytes of elements
 * 32q .. 32q+31 of row 8h+g at kb*2048 + h*1024 + (g*4+q)*32; after all code
 * blocks, 64 scale bytes per K-block placed as in ft_mxfp4_pack_tiles()
 * ((K/128)*2048 + kb*64 + (g*4+q)*2 + h).  N a multiple of 16, K of 128.
 * All pointers (device). */
FT_API ft_status ft_mxfp8_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                                     int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream);

/* Synthetic weights: out[j] = (float)(sigma * Z_{first+j}) where Z is the
 * Box-Muller normal of Philox4x32-10 block (first+j)/2 with counter
 * (q_lo, q_hi, stream_lo, stream_hi) and key (seed_lo, seed_hi), evaluated in
 * fp64 (cosine branch for even index, sine branch for odd).  out (device). */
FT_API ft_status ft_gen_normal_f32(uint64_t seed, uint64_t stream_id, uint64_t first, int64_t n, double sigma, float* out,
                            ft_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FTMOE_H_ */
