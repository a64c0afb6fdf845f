// quant.cu -- NVFP4 quantisers (weights and activations) and the synthetic
// weight generator.
//
// NVFP4 as the page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier
// MoE 拉回本地" uses it (sections on the evaluation and the limits): E2M1
// codes, an unsigned E4M3 scale per 16 elements, an fp32 scale per tensor.
// Quantiser definition (fp32, IEEE division): s_t = amax/2688 (1 if zero);
// per 16-block sb = E4M3_rn_sat(amax_b/6/s_t), eff = e4m3(sb)*s_t,
// code = E2M1_rn_sat(w/eff), with -0 codes stored as +0.  Activations use the
// same steps with s_t = 1.
#include "common.cuh"

namespace ft {

// amax over a tensor; non-negative floats order like their bit patterns.
__global__ void __launch_bounds__(256) k_amax(const float* __restrict__ w, int64_t n, unsigned int* amax_bits) {
    float m = 0.0f;
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float a = fabsf(w[i]);
        if (!(a <= 3.4028235e38f)) bad = true;  // NaN or inf
        else m = fmaxf(m, a);
    }
    if (bad) raise_dev_error(FT_DEVERR_BAD_SCALE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
        atomicMax(amax_bits, __float_as_uint(m));
    }
}

__global__ void k_tensor_scale(const unsigned int* amax_bits, float* ts) {
    float st = __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
    if (st == 0.0f) st = 1.0f;
    *ts = st;
}

// One thread per 16-element block of a [N][K] fp32 matrix.
__global__ void __launch_bounds__(256) k_quant_weight(const float* __restrict__ w, int64_t N, int64_t K,
                                                      const float* __restrict__ ts, uint8_t* __restrict__ codes,
                                                      int64_t codes_ld, uint8_t* __restrict__ scales,
                                                      int64_t scales_ld) {
    const int64_t nb = K / 16;
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= N * nb) return;
    const int64_t n = blk / nb, b = blk % nb;
    const float st = *ts;
    float v[16];
    const float4* src = reinterpret_cast<const float4*>(w + n * K + b * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    uint2 c;
    uint32_t sb;
    quant_block16(v, st, c, sb);
    *reinterpret_cast<uint2*>(codes + n * codes_ld + b * 8) = c;
    scales[n * scales_ld + b] = (uint8_t)sb;
}

// One thread per 16-element block of a [T][K] bf16 matrix, unit tensor scale.
__global__ void __launch_bounds__(256) k_quant_act(const uint16_t* __restrict__ x, int64_t T, int64_t K,
                                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    const int64_t nb = K / 16;
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= T * nb) return;
    const int64_t t = blk / nb, b = blk % nb;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K + b * 16);
    float v[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 u = src[q];
        const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * q + 2 * i] = __uint_as_float(words[i] << 16);
            v[8 * q + 2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
        }
    }
    uint2 c;
    uint32_t sb;
    quant_block16_bf16(v, c, sb);  // bf16 inputs, unit tensor scale
    *reinterpret_cast<uint2*>(codes + t * (K / 2) + b * 8) = c;
    scales[t * nb + b] = (uint8_t)sb;
}

// ----------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11) + Box-Muller in fp64
// ----------------------------------------------------------------------------
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0;
        const uint32_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

__device__ __forceinline__ double u53(uint32_t a, uint32_t b) {
    const uint64_t m = ((uint64_t)(a >> 5) << 26) | (uint64_t)(b >> 6);
    return (double)m * 0x1.0p-53;
}

__global__ void __launch_bounds__(256) k_gen_normal(uint64_t seed, uint64_t sid, uint64_t first, int64_t n,
                                                    double sigma, float* __restrict__ out) {
    const uint64_t q0 = first >> 1;
    const uint64_t nq = ((first + (uint64_t)n - 1) >> 1) - q0 + 1;
    for (uint64_t qi = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; qi < nq;
         qi += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t q = q0 + qi;
        uint32_t c[4] = {(uint32_t)q, (uint32_t)(q >> 32), (uint32_t)sid, (uint32_t)(sid >> 32)};
        philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
        const double u1 = u53(c[0], c[1]) + 0x1.0p-53;
        const double u2 = u53(c[2], c[3]);
        const double rad = sqrt(-2.0 * log(u1));
        const double th = 6.283185307179586 * u2;
        double sn, cs;
        sincos(th, &sn, &cs);
        const uint64_t i0 = 2 * q, i1 = 2 * q + 1;
        if (i0 >= first && i0 < first + (uint64_t)n) out[i0 - first] = __double2float_rn(sigma * (rad * cs));
        if (i1 >= first && i1 < first + (uint64_t)n) out[i1 - first] = __double2float_rn(sigma * (rad * sn));
    }
}

}  // namespace ft

using namespace ft;

extern "C" {

size_t ft_nvfp4_quantize_workspace_size(int64_t N, int64_t K) {
    (void)N;
    (void)K;
    return 256;
}

ft_status ft_nvfp4_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, int64_t codes_ld,
                                   uint8_t* scales, int64_t scales_ld, float* tensor_scale, void* ws,
                                   size_t ws_bytes, ft_stream_t stream) {
    if (N <= 0 || K <= 0 || K % 32)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_weight: need N > 0 and K a positive multiple of 32");
    if (!w || !codes || !scales || !tensor_scale) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_weight: null pointer");
    if (codes_ld < K / 2 || scales_ld < K / 16 || codes_ld % 8)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_weight: leading dimensions too small or codes_ld not a multiple of 8");
    if (!aligned(w, 16) || !aligned(codes, 8)) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_weight: misaligned w or codes");
    if (!ws || ws_bytes < ft_nvfp4_quantize_workspace_size(N, K) || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_weight: workspace missing or too small");
    cudaStream_t s = cu(stream);
    unsigned int* amax = static_cast<unsigned int*>(ws);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, std::string("ft_nvfp4_quantize_weight: ") + cudaGetErrorString(e));
    const int64_t n = N * K;
    const int64_t blocks_amax = std::min<int64_t>((n + 255) / 256, 148 * 16);
    k_amax<<<(unsigned)blocks_amax, 256, 0, s>>>(w, n, amax);
    k_tensor_scale<<<1, 1, 0, s>>>(amax, tensor_scale);
    const int64_t nblk = N * (K / 16);
    k_quant_weight<<<(unsigned)((nblk + 255) / 256), 256, 0, s>>>(w, N, K, tensor_scale, codes, codes_ld, scales,
                                                                   scales_ld);
    return check_launch("ft_nvfp4_quantize_weight");
}

ft_status ft_nvfp4_quantize_act(const uint16_t* x, int64_t T, int64_t K, uint8_t* codes, uint8_t* scales,
                                ft_stream_t stream) {
    if (T < 0 || K <= 0 || K % 32)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_act: need T >= 0 and K a positive multiple of 32");
    if (T == 0) return FT_OK;
    if (!x || !codes || !scales) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_act: null pointer");
    if (!aligned(x, 16) || !aligned(codes, 8)) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_quantize_act: misaligned x or codes");
    const int64_t nblk = T * (K / 16);
    k_quant_act<<<(unsigned)((nblk + 255) / 256), 256, 0, cu(stream)>>>(x, T, K, codes, scales);
    return check_launch("ft_nvfp4_quantize_act");
}

ft_status ft_gen_normal_f32(uint64_t seed, uint64_t stream_id, uint64_t first, int64_t n, double sigma, float* out,
                            ft_stream_t stream) {
    if (n < 0) return fail(FT_ERR_INVALID_ARG, "ft_gen_normal_f32: n < 0");
    if (n == 0) return FT_OK;
    if (!out) return fail(FT_ERR_INVALID_ARG, "ft_gen_normal_f32: out is null");
    const int64_t pairs = n / 2 + 2;
    const int64_t blocks = std::min<int64_t>((pairs + 255) / 256, 148 * 32);
    k_gen_normal<<<(unsigned)blocks, 256, 0, cu(stream)>>>(seed, stream_id, first, n, sigma, out);
    return check_launch("ft_gen_normal_f32");
}

}  // extern "C"
