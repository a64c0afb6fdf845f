// decode.cu -- expert SwiGLU FFN for small token counts (decode): NVFP4
// weights streamed with 128-bit loads, dequantised in registers, fp32
// accumulation, warp-shuffle reductions.
//
// Each expert is an independent FFN with its own weights (page
// "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", MoE core mechanism);
// weights are restored to higher precision at compute time (page
// xxmr.cn/news/175150 §2.1), here in registers: an E2M1 pair converts exactly
// to f16x2 and the product with its E4M3 block scale is exact in f16 (at most
// 6 significant bits, magnitudes within [2^-10, 2688]); the fp32 tensor scale
// is applied to the fp32 dot product.
#include "common.cuh"

#include <algorithm>

namespace ft {

constexpr int kGuWarps = 8;   // gate/up: one (gate, up) row pair per warp
constexpr int kDnWarps = 8;   // down: rows per warp depend on I
constexpr int kTokChunk = 4;  // tokens staged in shared memory per pass

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Dot of 8 dequantised weights (4 code bytes of word `cw`, scaled by f16x2
// `sc`) with 8 f16 activations `xv` (as 4 f16x2 words), accumulated in fp32.
__device__ __forceinline__ float dot8_f16(uint32_t cw, uint32_t sc, const uint4& xv, float acc) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t wv = hmul2(e2m1x2_to_f16x2((cw >> (8 * b)) & 0xFFu), sc);
        acc = fma_f16_f32((uint16_t)(wv & 0xFFFFu), (uint16_t)(xw[b] & 0xFFFFu), acc);
        acc = fma_f16_f32((uint16_t)(wv >> 16), (uint16_t)(xw[b] >> 16), acc);
    }
    return acc;
}

// Position of activation element `el` in the staged, lane-interleaved layout:
// lane l of 1024-element chunk c reads quarter q (8 elements) at
// ((c*4 + q)*32 + l)*8, so a warp's 16-byte shared loads are conflict-free.
__device__ __forceinline__ int xperm_index(int el) {
    const int c = el >> 10, w = el & 1023;
    const int l = w >> 5, q = (w >> 3) & 3, r = el & 7;
    return (((c * 4 + q) * 32 + l) << 3) + r;
}

__global__ void __launch_bounds__(kGuWarps * 32) k_decode_gateup(ft_moe_layer_weights W,
                                                                 const uint16_t* __restrict__ x, int k,
                                                                 const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ perm,
                                                                 const int32_t* __restrict__ active,
                                                                 uint16_t* __restrict__ hbuf) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int H = W.H, I = W.I;
    const int groups = I / kGuWarps;
    const int a = blockIdx.x / groups, g = blockIdx.x % groups;
    if (a >= active[0]) return;
    const int e = active[1 + a];
    const int p0 = offsets[e], p1 = offsets[e + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = g * kGuWarps + warp;
    const int wi = weight_index(W, e);
    if (wi < 0) {
        if (lane == 0)
            for (int p = p0; p < p1; ++p) hbuf[(int64_t)p * I + i] = 0;
        return;
    }
    const int nchunk = (H + 1023) / 1024;
    const int xsz = nchunk * 1024;
    __half* xs = reinterpret_cast<__half*>(smem);
    const uint8_t* gc = W.gu_codes + (int64_t)wi * W.gu_codes_stride + (int64_t)(2 * i) * (H / 2);
    const uint8_t* gs = W.gu_scales + (int64_t)wi * W.gu_scales_stride + (int64_t)(2 * i) * (H / 16);
    const float tsg = W.tscale[(int64_t)wi * W.tscale_stride + 0];
    const float tsu = W.tscale[(int64_t)wi * W.tscale_stride + 1];

    for (int pc = p0; pc < p1; pc += kTokChunk) {
        const int nt = min(kTokChunk, p1 - pc);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTokChunk * xsz; idx += blockDim.x) {
            const int j = idx / xsz, el = idx - j * xsz;
            float v = 0.0f;
            if (j < nt && el < H) {
                const int t = perm[pc + j] / k;
                v = bf16_to_f32(x[(int64_t)t * H + el]);
            }
            xs[j * xsz + xperm_index(el)] = __float2half_rn(v);
        }
        __syncthreads();
        float ag[kTokChunk], au[kTokChunk];
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j) ag[j] = au[j] = 0.0f;
        for (int c = 0; c < nchunk; ++c) {
            const int o = c * 512 + lane * 16;
            if (o < H / 2) {
                const uint4 cg = ld_stream(gc + o);
                const uint4 cu = ld_stream(gc + H / 2 + o);
                const uint32_t sg = *reinterpret_cast<const uint16_t*>(gs + o / 8);
                const uint32_t su = *reinterpret_cast<const uint16_t*>(gs + H / 16 + o / 8);
                const uint32_t sgl = e4m3_to_f16x2_bcast(sg & 0xFFu), sgh = e4m3_to_f16x2_bcast(sg >> 8);
                const uint32_t sul = e4m3_to_f16x2_bcast(su & 0xFFu), suh = e4m3_to_f16x2_bcast(su >> 8);
                const uint32_t wg[4] = {cg.x, cg.y, cg.z, cg.w};
                const uint32_t wu[4] = {cu.x, cu.y, cu.z, cu.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int j = 0; j < kTokChunk; ++j) {
                        if (j < nt) {
                            const uint4 xv =
                                *reinterpret_cast<const uint4*>(xs + j * xsz + (((c * 4 + q) * 32 + lane) << 3));
                            ag[j] = dot8_f16(wg[q], q < 2 ? sgl : sgh, xv, ag[j]);
                            au[j] = dot8_f16(wu[q], q < 2 ? sul : suh, xv, au[j]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j) {
            if (j < nt) {
                const float gsum = warp_sum(ag[j]) * tsg;
                const float usum = warp_sum(au[j]) * tsu;
                if (lane == 0) hbuf[(int64_t)(pc + j) * I + i] = bf16_bits(silu_f32(gsum) * usum);
            }
        }
    }
}

// Down projection: a warp covers `rpw` rows, `lpr` lanes per row (I/2 bytes
// per row, 16 bytes per lane per step).  h rows staged as fp32 in a
// lane-interleaved layout.
__global__ void __launch_bounds__(kDnWarps * 32) k_decode_down(ft_moe_layer_weights W, int k,
                                                               const int32_t* __restrict__ offsets,
                                                               const int32_t* __restrict__ active,
                                                               const uint16_t* __restrict__ hbuf,
                                                               float* __restrict__ y) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int H = W.H, I = W.I;
    const int lpr = min(32, I / 32);
    const int rpw = 32 / lpr;
    const int rows_cta = kDnWarps * rpw;
    const int groups = (H + rows_cta - 1) / rows_cta;
    const int a = blockIdx.x / groups, g = blockIdx.x % groups;
    if (a >= active[0]) return;
    const int e = active[1 + a];
    const int p0 = offsets[e], p1 = offsets[e + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / lpr, sl = lane % lpr;
    const int n = g * rows_cta + warp * rpw + sub;
    const bool row_ok = n < H;
    const int wi = weight_index(W, e);
    if (wi < 0) {
        if (row_ok && sl == 0)
            for (int p = p0; p < p1; ++p) y[(int64_t)p * H + n] = 0.0f;
        return;
    }
    const int step = 16 * lpr;                 // bytes of a row per warp step
    const int nch = (I / 2 + step - 1) / step;  // steps per row
    const int ipad = nch * step * 2;            // staged elements per token
    float* hs = reinterpret_cast<float*>(smem);
    const uint8_t* dc = W.d_codes + (int64_t)wi * W.d_codes_stride + (int64_t)n * (I / 2);
    const uint8_t* ds = W.d_scales + (int64_t)wi * W.d_scales_stride + (int64_t)n * (I / 16);
    const float tsd = W.tscale[(int64_t)wi * W.tscale_stride + 2];

    for (int pc = p0; pc < p1; pc += kTokChunk) {
        const int nt = min(kTokChunk, p1 - pc);
        __syncthreads();
        // element el of a row: step c = el / (32*lpr), lane l, quarter q of 4 floats
        for (int idx = threadIdx.x; idx < kTokChunk * ipad; idx += blockDim.x) {
            const int j = idx / ipad, el = idx - j * ipad;
            float v = 0.0f;
            if (j < nt && el < I) v = bf16_to_f32(hbuf[(int64_t)(pc + j) * I + el]);
            const int c = el / (32 * lpr), w = el - c * 32 * lpr;
            const int l = w >> 5, q = (w >> 2) & 7, r = el & 3;
            hs[j * ipad + ((c * 8 + q) * lpr + l) * 4 + r] = v;
        }
        __syncthreads();
        float acc[kTokChunk];
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j) acc[j] = 0.0f;
        if (row_ok) {
            for (int c = 0; c < nch; ++c) {
                const int o = c * step + sl * 16;
                if (o < I / 2) {
                    const uint4 cw = ld_stream(dc + o);
                    const uint32_t s2 = *reinterpret_cast<const uint16_t*>(ds + o / 8);
                    const uint32_t sl0 = e4m3_to_f16x2_bcast(s2 & 0xFFu), sl1 = e4m3_to_f16x2_bcast(s2 >> 8);
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float wf[8];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const uint32_t wv = hmul2(e2m1x2_to_f16x2((words[q] >> (8 * b)) & 0xFFu), q < 2 ? sl0 : sl1);
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
                            wf[2 * b] = f.x;
                            wf[2 * b + 1] = f.y;
                        }
#pragma unroll
                        for (int j = 0; j < kTokChunk; ++j) {
                            if (j < nt) {
                                const float* hb = hs + j * ipad + ((c * 8 + 2 * q) * lpr + sl) * 4;
                                const float4 h0 = *reinterpret_cast<const float4*>(hb);
                                const float4 h1 = *reinterpret_cast<const float4*>(hb + lpr * 4);
                                float s = acc[j];
                                s = fmaf(wf[0], h0.x, s);
                                s = fmaf(wf[1], h0.y, s);
                                s = fmaf(wf[2], h0.z, s);
                                s = fmaf(wf[3], h0.w, s);
                                s = fmaf(wf[4], h1.x, s);
                                s = fmaf(wf[5], h1.y, s);
                                s = fmaf(wf[6], h1.z, s);
                                s = fmaf(wf[7], h1.w, s);
                                acc[j] = s;
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j) {
            float s = acc[j];
            for (int o2 = lpr / 2; o2 > 0; o2 >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o2);
            if (j < nt && row_ok && sl == 0) y[(int64_t)(pc + j) * H + n] = s * tsd;
        }
    }
}

ft_status decode_tiles_grouped(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k, const int32_t* offsets,
                               const int32_t* perm, const float* w, float* y, uint16_t* out, void* ws, size_t ws_bytes,
                               ft_stream_t stream);

ft_status validate_weights(const ft_moe_layer_weights* W, const char* fn) {
    if (!W) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weights descriptor is null");
    if (W->E <= 0 || W->E > 1024 || W->H <= 0 || W->H % 256 || W->I <= 0 || W->I % 128 || W->n_weights <= 0)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= E <= 1024, H a multiple of 256, I a multiple of 128");
    const bool rows = W->layout == FT_LAYOUT_ROWS || W->layout == FT_LAYOUT_MXFP4_ROWS || W->layout == FT_LAYOUT_MXFP8_ROWS;
    const bool mx = W->layout >= FT_LAYOUT_MXFP4_ROWS && W->layout <= FT_LAYOUT_MXFP8_DECODE_TILES;  // no tensor scale
    if (!W->gu_codes || !W->d_codes || (!mx && !W->tscale) || (rows && (!W->gu_scales || !W->d_scales)))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null weight pointer");
    if (!W->expert_to_slot && W->n_weights < W->E)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": n_weights < E without a slot table");
    const void* ptrs[4] = {W->gu_codes, W->gu_scales, W->d_codes, W->d_scales};
    for (const void* p : ptrs)
        if (p && !aligned(p, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weight pointers need 16-byte alignment");
    if (W->gu_codes_stride % 16 || W->gu_scales_stride % 16 || W->d_codes_stride % 16 || W->d_scales_stride % 16)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weight strides need to be multiples of 16 bytes");
    if (!mx && W->tscale_stride < 3) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": tscale_stride < 3");
    return FT_OK;
}

}  // namespace ft

using namespace ft;

namespace {
size_t align256(size_t b) { return (b + 255) / 256 * 256; }
}  // namespace

extern "C" {

size_t ft_moe_decode_workspace_size(int T, int k, int H, int I) {
    if (T <= 0 || k <= 0 || H <= 0 || I <= 0) return 0;
    const size_t rows = (size_t)T * k;
    // [0, 256): call counter of the tiled kernel; then its h words (4 bytes per value), or
    // h (bf16) and y (fp32) of the row kernels
    const size_t row_path = align256(rows * I * sizeof(uint16_t)) + align256(rows * H * sizeof(float));
    return 256 + std::max(row_path, align256(rows * I * 4));
}

ft_status ft_moe_expert_ffn_nvfp4_decode(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k,
                                         const int32_t* offsets, const int32_t* perm, const int32_t* active,
                                         const int32_t* inv, const float* w, float* y, uint16_t* out, void* ws,
                                         size_t ws_bytes, ft_stream_t stream) {
    const char* fn = "ft_moe_expert_ffn_nvfp4_decode";
    ft_status st = validate_weights(W, fn);
    if (st != FT_OK) return st;
    if (T < 0 || k <= 0 || k > W->E || k > 32) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need T >= 0, 1 <= k <= min(E, 32)");
    if (T == 0) return FT_OK;
    if (!x || !offsets || !perm || !active) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (!y && !out) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need y or out");
    if (out && (!inv || !w)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": out needs inv and w");
    const size_t need = ft_moe_decode_workspace_size(T, k, W->H, W->I);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": workspace missing, too small or not 256-byte aligned");
    if (y && !aligned(y, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": y needs 16-byte alignment");
    if (W->layout == FT_LAYOUT_DECODE_TILES)
        return decode_tiles_grouped(W, x, T, k, offsets, perm, w, y, out, ws, ws_bytes, stream);
    if (W->layout != FT_LAYOUT_ROWS) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": unknown weight layout");
    const int H = W->H, I = W->I;
    const int rows = T * k;
    uint16_t* hbuf = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + 256);
    float* ybuf = y ? y : reinterpret_cast<float*>(static_cast<char*>(ws) + 256 + align256((size_t)rows * I * 2));
    const int max_active = std::min(W->E, rows);
    cudaStream_t s = cu(stream);

    const int nchunk = (H + 1023) / 1024;
    const size_t smem_gu = (size_t)kTokChunk * nchunk * 1024 * sizeof(__half);
    if (smem_gu > 48 * 1024) cudaFuncSetAttribute(k_decode_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
    const int grid_gu = max_active * (I / kGuWarps);
    k_decode_gateup<<<grid_gu, kGuWarps * 32, smem_gu, s>>>(*W, x, k, offsets, perm, active, hbuf);

    const int lpr = std::min(32, I / 32), rpw = 32 / lpr, rows_cta = kDnWarps * rpw;
    const int step = 16 * lpr, nch = (I / 2 + step - 1) / step;
    const size_t smem_dn = (size_t)kTokChunk * nch * step * 2 * sizeof(float);
    if (smem_dn > 48 * 1024) cudaFuncSetAttribute(k_decode_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
    const int grid_dn = max_active * ((H + rows_cta - 1) / rows_cta);
    k_decode_down<<<grid_dn, kDnWarps * 32, smem_dn, s>>>(*W, k, offsets, active, hbuf, ybuf);
    st = check_launch(fn);
    if (st != FT_OK) return st;
    if (out) return ft_moe_combine(ybuf, inv, w, T, k, H, out, stream);
    return FT_OK;
}

}  // extern "C"
