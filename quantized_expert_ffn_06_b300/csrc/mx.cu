// mx.cu -- MX expert weights (MXFP4 and MXFP8): the block quantisers, the
// packing into the decode kernel's 16-row tiles, and the exact re-encoding of
// MXFP4 into the FP4 tensor-core tiles of the prefill.
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

// ---------------------------------------------------------------------------- MXFP4 -> FP4 tensor-core tiles

// The UMMA tile layout (the one ft_nvfp4_pack_umma writes): [R][K] in blocks of 128 rows x 128 K, 9216 bytes,
// block (rt, ks) at (rt*(K/128) + ks)*9216; code byte b (0..63) of row r at (b/16)*2048 + (r/8)*128 + (r%8)*16 +
// b%16, E4M3 scale j (0..7, one per 16 elements) of row r at 8192 + (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4.
__device__ __forceinline__ int mxu_code_off(int r, int b) { return (b >> 4) * 2048 + (r >> 3) * 128 + (r & 7) * 16 + (b & 15); }
__device__ __forceinline__ int mxu_scale_off(int r, int j) { return 8192 + (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3); }

// A 32-element block holds a non-zero code when some nibble has a non-zero magnitude (E2M1 +-0 are 0x0 / 0x8).
__device__ __forceinline__ bool mx4_block_nonzero(uint4 c) { return ((c.x | c.y | c.z | c.w) & 0x77777777u) != 0u; }

// Pass 1, one thread per block: the largest scale byte over blocks with a non-zero code, into *smax (int, -1
// initially).  A NaN scale byte (255) does not count: pass 2 reports it and the other blocks keep their span.
__global__ void __launch_bounds__(256) k_mx_umma_smax(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                      const uint8_t* __restrict__ scales, int64_t scales_ld,
                                                      int64_t N, int64_t K, int* __restrict__ smax) {
    const int64_t nb = K / 32, i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int v = -1;
    if (i < N * nb) {
        const int64_t r = i / nb, b = i - r * nb;
        const uint4 c = *reinterpret_cast<const uint4*>(codes + r * codes_ld + b * 16);
        const int sb = scales[r * scales_ld + b];
        if (sb != 255 && mx4_block_nonzero(c)) v = sb;
    }
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0 && v >= 0) atomicMax(smax, v);
}

// E4M3 byte of 2^d, -9 <= d <= 8: normals (d >= -6) have exponent field d + 7 and no mantissa; 2^-7 .. 2^-9 are
// the subnormals m * 2^-9 with m = 4, 2, 1.
__device__ __forceinline__ uint32_t e4m3_pow2(int d) { return d >= -6 ? (uint32_t)(d + 7) << 3 : 1u << (d + 9); }

// Pass 2, as the NVFP4 packing: per row and 128-K block, four 16-byte code pieces and one group of 8 scales.
__global__ void __launch_bounds__(256) k_mx_pack_umma(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                      const uint8_t* __restrict__ scales, int64_t scales_ld,
                                                      int64_t N, int64_t K, const int* __restrict__ smax,
                                                      uint8_t* __restrict__ out) {
    const int64_t KSN = K / 128, per_row = 5, total = N * KSN * per_row;
    const int s0 = __ldg(smax) - 8;
    bool range = false, nan = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / (KSN * per_row), rem = i - row * (KSN * per_row), ks = rem / per_row;
        const int piece = (int)(rem - ks * per_row), r = (int)(row % 128);
        uint8_t* blk = out + ((row / 128) * KSN + ks) * 9216;
        const uint8_t* crow = codes + row * codes_ld + ks * 64;
        if (piece < 4) {
            *reinterpret_cast<uint4*>(blk + mxu_code_off(r, piece * 16)) =
                *reinterpret_cast<const uint4*>(crow + piece * 16);
        } else {
            for (int q = 0; q < 4; ++q) {  // the four MX blocks of this 128-K block
                const uint32_t sb = scales[row * scales_ld + ks * 4 + q];
                const bool nz = mx4_block_nonzero(*reinterpret_cast<const uint4*>(crow + q * 16));
                uint32_t e = 0;
                if (sb == 255u) {
                    nan = true;
                } else if (nz) {
                    const int d = (int)sb - s0;
                    if (d < -9) range = true;
                    else e = e4m3_pow2(d);
                }
                blk[mxu_scale_off(r, 2 * q)] = (uint8_t)e;
                blk[mxu_scale_off(r, 2 * q + 1)] = (uint8_t)e;
            }
        }
    }
    if (range) raise_dev_error(FT_DEVERR_RANGE);
    if (nan) raise_dev_error(FT_DEVERR_BAD_SCALE);
}

// Pass 3: the tensor scale 2^(s0 - 127) (1 when no block is non-zero) replaces the scratch word.
__global__ void k_mx_umma_tscale(float* tscale, int n) {
    const int sm = *reinterpret_cast<const int*>(tscale);
    const float t = sm < 0 ? 1.0f : ldexpf(1.0f, sm - 8 - 127);
    for (int i = 0; i < n; ++i) tscale[i] = t;
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

ft_status ft_mxfp4_pack_umma(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                             int64_t N, int64_t K, uint8_t* tiles, float* tscale, int ts_count, ft_stream_t stream) {
    const char* fn = "ft_mxfp4_pack_umma";
    if (N <= 0 || K <= 0 || N % 128 || K % 128)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need N and K multiples of 128");
    if (ts_count < 1 || ts_count > 4) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= ts_count <= 4");
    if (!codes || !scales || !tiles || !tscale) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (!aligned(codes, 16) || codes_ld % 16 || !aligned(tiles, 16) || !aligned(tscale, 4) || codes_ld < K / 2 ||
        scales_ld < K / 32)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": codes/tiles need 16-byte alignment and row strides");
    cudaStream_t s = cu(stream);
    int* smax = reinterpret_cast<int*>(tscale);
    if (cudaMemsetAsync(smax, 0xFF, sizeof(int), s) != cudaSuccess)
        return fail(FT_ERR_CUDA, std::string(fn) + ": memset failed");
    const int64_t nblk = N * (K / 32);
    k_mx_umma_smax<<<(unsigned)((nblk + 255) / 256), 256, 0, s>>>(codes, codes_ld, scales, scales_ld, N, K, smax);
    const int64_t total = N * (K / 128) * 5;
    k_mx_pack_umma<<<(unsigned)std::min<int64_t>((total + 255) / 256, 148 * 64), 256, 0, s>>>(
        codes, codes_ld, scales, scales_ld, N, K, smax, tiles);
    k_mx_umma_tscale<<<1, 1, 0, s>>>(tscale, ts_count);
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
