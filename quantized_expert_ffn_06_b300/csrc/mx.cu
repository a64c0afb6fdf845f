// mx.cu -- MX expert weights (MXFP4 and MXFP8): the block quantisers and the
// packing into the decode kernel's 16-row tiles.
//
// The page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier MoE 拉回本地"
// (section 局限) lists MXFP4 beside NVFP4 and FP8 as the weight formats the
// engine depends on, without a bit layout.  The format here is the OCP
// Microscaling (MX) v1.0 one: 32 consecutive elements of a row share a UE8M0
// scale byte s standing for 2^(s - 127); elements are E2M1.  Quantising a
// block: X = floor(log2(amax)) - 2 (2 = exponent of E2M1's largest normal),
// clamped to [-127, 127] (-127 for an all-zero block); code = E2M1_rn_sat(v /
// 2^X) with -0 stored as +0; s = X + 127.  No tensor scale.  MXFP8 is the same
// with E4M3 elements (emax 8, largest finite 448), one byte each.
#include "common.cuh"

namespace ft {

// floor(log2(a)) of a finite a > 0, subnormals included.
__device__ __forceinline__ int floor_log2_f32(float a) {
    const uint32_t b = __float_as_uint(a);
    const int eb = (int)(b >> 23);
    if (eb > 0) return eb - 127;
    return (31 - __clz((int)(b & 0x7FFFFFu))) - 149;  // subnormal: m * 2^-149
}

// One thread per 32-element block of a [N][K] fp32 matrix.
__global__ void __launch_bounds__(256) k_mx_quant_weight(const float* __restrict__ w, int64_t N, int64_t K,
                                                         uint8_t* __restrict__ codes, int64_t codes_ld,
                                                         uint8_t* __restrict__ scales, int64_t scales_ld) {
    const int64_t nb = K / 32;
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= N * nb) return;
    const int64_t n = blk / nb, b = blk % nb;
    float v[32];
    const float4* src = reinterpret_cast<const float4*>(w + n * K + b * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    float amax = 0.0f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float a = fabsf(v[i]);
        bad |= !(a <= 3.4028235e38f);
        amax = fmaxf(amax, a);
    }
    if (bad) raise_dev_error(FT_DEVERR_BAD_SCALE);
    int X = (amax > 0.0f) ? floor_log2_f32(amax) - 2 : -127;
    X = max(-127, min(127, X));
    // 2^-X as an fp32 (X >= -127 and floor(log2(amax)) <= 127 keep -X within [-125, 127]: a normal)
    const float inv = __int_as_float((127 - X) << 23);
    uint32_t byte[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) byte[i] = f32x2_to_e2m1x2_rn_sat(v[2 * i] * inv, v[2 * i + 1] * inv);
    uint4 c;
    c.x = byte[0] | (byte[1] << 8) | (byte[2] << 16) | (byte[3] << 24);
    c.y = byte[4] | (byte[5] << 8) | (byte[6] << 16) | (byte[7] << 24);
    c.z = byte[8] | (byte[9] << 8) | (byte[10] << 16) | (byte[11] << 24);
    c.w = byte[12] | (byte[13] << 8) | (byte[14] << 16) | (byte[15] << 24);
    *reinterpret_cast<uint4*>(codes + n * codes_ld + b * 16) = c;
    scales[n * scales_ld + b] = (uint8_t)(X + 127);
}

// One thread per 32-element block of a [N][K] fp32 matrix, E4M3 elements.
__global__ void __launch_bounds__(256) k_mx8_quant_weight(const float* __restrict__ w, int64_t N, int64_t K,
                                                          uint8_t* __restrict__ codes, int64_t codes_ld,
                                                          uint8_t* __restrict__ scales, int64_t scales_ld) {
    const int64_t nb = K / 32;
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= N * nb) return;
    const int64_t n = blk / nb, b = blk % nb;
    float v[32];
    const float4* src = reinterpret_cast<const float4*>(w + n * K + b * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    float amax = 0.0f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float a = fabsf(v[i]);
        bad |= !(a <= 3.4028235e38f);
        amax = fmaxf(amax, a);
    }
    if (bad) raise_dev_error(FT_DEVERR_BAD_SCALE);
    int X = (amax > 0.0f) ? floor_log2_f32(amax) - 8 : -127;
    X = max(-127, min(127, X));
    const float inv = __int_as_float((127 - X) << 23);  // 2^-X, a normal (-X within [-119, 127])
    uint32_t word[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t wd = 0;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            uint16_t pr;  // {element 4i+j in the low byte, 4i+j+1 in the high byte}
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(v[4 * i + j + 1] * inv), "f"(v[4 * i + j] * inv));
            uint32_t lo = pr & 0xFFu, hi = pr >> 8;
            if ((lo & 0x7Fu) == 0) lo = 0;  // -0 stored as +0
            if ((hi & 0x7Fu) == 0) hi = 0;
            wd |= (lo | (hi << 8)) << (8 * j);
        }
        word[i] = wd;
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + n * codes_ld + b * 32);
    dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
    dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
    scales[n * scales_ld + b] = (uint8_t)(X + 127);
}

// [N][K] row-major MXFP8 codes/scales -> 16-row tiles (layout in ft_mxfp8_pack_tiles).
__global__ void __launch_bounds__(256) k_mx8_pack_tiles(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                        const uint8_t* __restrict__ scales, int64_t scales_ld,
                                                        int64_t N, int64_t K, uint8_t* __restrict__ tiles) {
    const int64_t KB = K / 128;
    const int64_t tile_bytes = KB * 2112;
    const int64_t per_tile = KB * 128 + KB * 32;  // 16-byte code pieces + 2-byte scale pairs
    const int64_t total = (N / 16) * per_tile;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / per_tile;
        int64_t r = i % per_tile;
        uint8_t* dst = tiles + tile * tile_bytes;
        if (r < KB * 128) {  // code piece (kb, h, g, q, p): bytes 32q + 16p .. +15 of row 8h+g's 128 in block kb
            const int64_t kb = r / 128;
            const int rem = (int)(r % 128);
            const int h = rem / 64, g = (rem / 8) & 7, q = (rem / 2) & 3, pc = rem & 1;
            const int64_t row = tile * 16 + 8 * h + g;
            const uint4 v = *reinterpret_cast<const uint4*>(codes + row * codes_ld + kb * 128 + 32 * q + 16 * pc);
            *reinterpret_cast<uint4*>(dst + kb * 2048 + h * 1024 + (g * 4 + q) * 32 + 16 * pc) = v;
        } else {  // scale pair (kb, g, q): block 4kb + q of rows g and g+8
            r -= KB * 128;
            const int64_t kb = r / 32;
            const int rem = (int)(r % 32);
            const int g = rem / 4, q = rem & 3;
            const uint8_t s0 = scales[(tile * 16 + g) * scales_ld + kb * 4 + q];
            const uint8_t s1 = scales[(tile * 16 + 8 + g) * scales_ld + kb * 4 + q];
            *reinterpret_cast<uint16_t*>(dst + KB * 2048 + kb * 64 + (g * 4 + q) * 2) = (uint16_t)(s0 | ((uint32_t)s1 << 8));
        }
    }
}

// [N][K] row-major MXFP4 codes/scales -> 16-row tiles (layout in ft_mxfp4_pack_tiles).
__global__ void __launch_bounds__(256) k_mx_pack_tiles(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                       const uint8_t* __restrict__ scales, int64_t scales_ld,
                                                       int64_t N, int64_t K, uint8_t* __restrict__ tiles) {
    const int64_t KB = K / 128;
    const int64_t tile_bytes = KB * 1088;
    const int64_t per_tile = KB * 64 + KB * 32;  // 16-byte code pieces + 2-byte scale pairs
    const int64_t total = (N / 16) * per_tile;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / per_tile;
        int64_t r = i % per_tile;
        uint8_t* dst = tiles + tile * tile_bytes;
        if (r < KB * 64) {  // code piece (kb, h, g, q): bytes 16q..16q+15 of row 8h+g's 64 bytes in block kb
            const int64_t kb = r / 64;
            const int rem = (int)(r % 64);
            const int h = rem / 32, g = (rem / 4) & 7, q = rem & 3;
            const int64_t row = tile * 16 + 8 * h + g;
            const uint4 v = *reinterpret_cast<const uint4*>(codes + row * codes_ld + kb * 64 + 16 * q);
            *reinterpret_cast<uint4*>(dst + kb * 1024 + h * 512 + (g * 4 + q) * 16) = v;
        } else {  // scale pair (kb, g, q): block 4kb + q of rows g and g+8
            r -= KB * 64;
            const int64_t kb = r / 32;
            const int rem = (int)(r % 32);
            const int g = rem / 4, q = rem & 3;
            const uint8_t s0 = scales[(tile * 16 + g) * scales_ld + kb * 4 + q];
            const uint8_t s1 = scales[(tile * 16 + 8 + g) * scales_ld + kb * 4 + q];
            *reinterpret_cast<uint16_t*>(dst + KB * 1024 + kb * 64 + (g * 4 + q) * 2) =
                (uint16_t)(s0 | ((uint32_t)s1 << 8));
        }
    }
}

}  // namespace ft

using namespace ft;

extern "C" {

ft_status ft_mxfp4_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                   uint8_t* scales, int64_t scales_ld, ft_stream_t stream) {
    const char* fn = "ft_mxfp4_quantize_weight";
    if (N <= 0 || K <= 0 || K % 32)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need N > 0 and K a positive multiple of 32");
    if (!w || !codes || !scales) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (codes_ld < K / 2 || scales_ld < K / 32 || codes_ld % 16)
        return fail(FT_ERR_INVALID_ARG,
                    std::string(fn) + ": leading dimensions too small or codes_ld not a multiple of 16");
    if (!aligned(w, 16) || !aligned(codes, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": misaligned w or codes");
    const int64_t nblk = N * (K / 32);
    k_mx_quant_weight<<<(unsigned)((nblk + 255) / 256), 256, 0, cu(stream)>>>(w, N, K, codes, codes_ld, scales,
                                                                               scales_ld);
    return check_launch(fn);
}

ft_status ft_mxfp4_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                              int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream) {
    const char* fn = "ft_mxfp4_pack_tiles";
    if (N <= 0 || K <= 0 || N % 16 || K % 128)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need N a multiple of 16 and K a multiple of 128");
    if (!codes || !scales || !tiles) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (!aligned(codes, 16) || codes_ld % 16 || !aligned(tiles, 16) || scales_ld < K / 32 || codes_ld < K / 2)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": codes/tiles need 16-byte alignment and row strides");
    const int64_t total = (N / 16) * (K / 128) * 96;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 32);
    k_mx_pack_tiles<<<(unsigned)blocks, 256, 0, cu(stream)>>>(codes, codes_ld, scales, scales_ld, N, K, tiles);
    return check_launch(fn);
}

ft_status ft_mxfp8_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                   uint8_t* scales, int64_t scales_ld, ft_stream_t stream) {
    const char* fn = "ft_mxfp8_quantize_weight";
    if (N <= 0 || K <= 0 || K % 32)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need N > 0 and K a positive multiple of 32");
    if (!w || !codes || !scales) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (codes_ld < K || scales_ld < K / 32 || codes_ld % 16)
        return fail(FT_ERR_INVALID_ARG,
                    std::string(fn) + ": leading dimensions too small or codes_ld not a multiple of 16");
    if (!aligned(w, 16) || !aligned(codes, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": misaligned w or codes");
    const int64_t nblk = N * (K / 32);
    k_mx8_quant_weight<<<(unsigned)((nblk + 255) / 256), 256, 0, cu(stream)>>>(w, N, K, codes, codes_ld, scales,
                                                                                scales_ld);
    return check_launch(fn);
}

ft_status ft_mxfp8_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                              int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream) {
    const char* fn = "ft_mxfp8_pack_tiles";
    if (N <= 0 || K <= 0 || N % 16 || K % 128)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need N a multiple of 16 and K a multiple of 128");
    if (!codes || !scales || !tiles) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (!aligned(codes, 16) || codes_ld % 16 || !aligned(tiles, 16) || scales_ld < K / 32 || codes_ld < K)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": codes/tiles need 16-byte alignment and row strides");
    const int64_t total = (N / 16) * (K / 128) * 160;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 32);
    k_mx8_pack_tiles<<<(unsigned)blocks, 256, 0, cu(stream)>>>(codes, codes_ld, scales, scales_ld, N, K, tiles);
    return check_launch(fn);
}

}  // extern "C"
