// common.cuh -- shared plumbing of the sm_103a MoE kernels: status handling,
// the per-device error word, and small PTX helpers for the NVFP4 formats.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <string>

#include "../../include/ftmoe.h"

namespace ft {

// ----------------------------------------------------------------------------
// host-side status plumbing
// ----------------------------------------------------------------------------
void set_error(const std::string& msg);
ft_status fail(ft_status s, const std::string& msg);
ft_status check_launch(const char* what);
inline cudaStream_t cu(ft_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ----------------------------------------------------------------------------
// device error word (one per device; read and cleared by ft_device_status)
// ----------------------------------------------------------------------------
extern __device__ unsigned int g_err_word;

__device__ __forceinline__ void raise_dev_error(unsigned int bits) { atomicOr(&g_err_word, bits); }

// ----------------------------------------------------------------------------
// NVFP4 helpers
// ----------------------------------------------------------------------------

// Two E2M1 codes (low nibble = first element) -> f16x2 (first element in the
// low half).  Exact: every E2M1 value is an f16 value.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(out) : "r"(byte));
    return out;
}

// E4M3 scale byte -> f16x2 with the value in both halves (exact: E4M3 values
// are f16 normals).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t b) {
    uint32_t out;
    const uint32_t pair = (b & 0xFFu) | ((b & 0xFFu) << 8);
    asm("{\n\t.reg .b16 p;\n\tcvt.u16.u32 p, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, p;\n\t}" : "=r"(out) : "r"(pair));
    return out;
}

// Unsigned E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t h2 = e4m3_to_f16x2_bcast(b);
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// fp32 -> E4M3 byte, round to nearest even, saturating to 448 (input >= 0).
__device__ __forceinline__ uint32_t f32_to_e4m3_rn_sat(float r) {
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(r));
    return out & 0xFFu;  // second source lands in the low byte
}

// two fp32 -> packed E2M1 byte (lo -> low nibble), round to nearest even,
// saturating to +-6; a code of -0 is replaced by +0.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2_rn_sat(float lo, float hi) {
    uint16_t out;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(out) : "f"(hi), "f"(lo));
    uint32_t v = out & 0xFFu;
    if ((v & 0x0Fu) == 0x08u) v &= 0xF0u;
    if ((v & 0xF0u) == 0x80u) v &= 0x0Fu;
    return v;
}

// Block quantiser (fp32, IEEE division): 16 values -> 8 code bytes + 1 E4M3
// scale byte, with tensor scale st: sb = E4M3_rn_sat(amax/6/st),
// eff = e4m3(sb)*st, code = E2M1_rn_sat(v/eff) (0 when eff is 0).
__device__ __forceinline__ void quant_block16(const float (&v)[16], float st, uint2& codes, uint32_t& sb) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 6.0f);
    const float r = __fdiv_rn(d, st);
    sb = f32_to_e4m3_rn_sat(r);
    const float eff = __fmul_rn(e4m3_to_f32(sb), st);
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        b[i] = (eff == 0.0f) ? 0u : f32x2_to_e2m1x2_rn_sat(__fdiv_rn(v[2 * i], eff), __fdiv_rn(v[2 * i + 1], eff));
    codes.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    codes.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
}

// The same block quantiser for bf16-valued inputs with unit tensor scale (activations, and h after its bf16
// rounding), with one reciprocal per block instead of a division per element.  With v of at most 8 significant
// bits and eff an E4M3 value (at most 4), v / eff is either exactly a midpoint of the E2M1 grid (0.25, 0.75, 1.25,
// 1.75, 2.5, 3.5, 5) or at least 2^-17 away from every midpoint.  q = v * (1/eff) rounded, followed by one residual
// correction q + (v - q * eff) / eff evaluated with fused multiply-adds (the reciprocal-refinement step of
// Markstein's division), lands within a few fp32 units of v / eff, so on the same side of every midpoint, and at
// an exact midpoint on the midpoint itself.  The E2M1 conversion then rounds it exactly as it rounds the
// correctly rounded quotient.  Finite inputs only.
__device__ __forceinline__ void quant_block16_bf16(const float (&v)[16], uint2& codes, uint32_t& sb) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    sb = f32_to_e4m3_rn_sat(__fdiv_rn(amax, 6.0f));
    const float eff = e4m3_to_f32(sb);
    uint32_t b[8];
    if (eff == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = 0u;
    } else {
        const float inv = __frcp_rn(eff);
        float q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float q0 = __fmul_rn(v[i], inv);
            q[i] = __fmaf_rn(__fmaf_rn(-q0, eff, v[i]), inv, q0);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = f32x2_to_e2m1x2_rn_sat(q[2 * i], q[2 * i + 1]);
    }
    codes.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    codes.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
}

// acc += a(f16) * b(f16), fp32 accumulate.
__device__ __forceinline__ float fma_f16_f32(uint16_t a, uint16_t b, float acc) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(acc));
    return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ uint16_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Order-preserving key of an fp32 logit: larger value -> larger key; -0 and +0
// map to the same key; NaN to 1 (below every number); 0 is never produced.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (v != v) ? 1u : key;
}

// Top-k selection of one token's E logits by one warp (E <= 256, k <= 32).
// Lane l holds experts l, l+32, ..., l+224 (consecutive lanes, consecutive
// addresses) and sorts its keys once, descending, by a stable odd-even
// transposition network (equal keys keep ascending expert order).  Round j
// takes the warp-wide maximum of the lanes' head keys and, among the lanes
// holding it, the lowest expert id (two redux.sync); that lane pops its head.
// `row` may point to shared or global memory.  Lane j < k gets expert j.
__device__ __forceinline__ int select_topk8(const float* row, int E, int k, bool& bad) {
    const int lane = threadIdx.x & 31;
    uint32_t key[8], ex[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        const bool in = e < E;
        const float v = in ? row[e] : 0.0f;
        key[i] = in ? logit_key(v) : 0u;
        ex[i] = (uint32_t)e;
        bad |= in && ((v != v) || (v == INFINITY));
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
        for (int i = r & 1; i + 1 < 8; i += 2) {
            const bool sw = key[i + 1] > key[i];
            const uint32_t ka = key[i], kb = key[i + 1], ea = ex[i], eb = ex[i + 1];
            key[i] = sw ? kb : ka;
            key[i + 1] = sw ? ka : kb;
            ex[i] = sw ? eb : ea;
            ex[i + 1] = sw ? ea : eb;
        }
    }
    int my_e = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        const uint32_t gk = __reduce_max_sync(0xffffffffu, key[0]);
        const uint32_t we = __reduce_min_sync(0xffffffffu, key[0] == gk ? ex[0] : 0xFFFFFFFFu);
        if (lane == j) my_e = (int)we;
        const bool win = ex[0] == we;  // expert ids are distinct: exactly one lane pops
#pragma unroll
        for (int i = 0; i < 7; ++i) {
            key[i] = win ? key[i + 1] : key[i];
            ex[i] = win ? ex[i + 1] : ex[i];
        }
        key[7] = win ? 0u : key[7];
    }
    return my_e;
}

// Wait-expiry test hook (ft_debug_inject_wait_expiry): the bound on any single wait and the site made to expire,
// read by the host code of each kernel at launch.
unsigned long long wait_hook_ns();
int wait_hook_site();

// weight index of an expert (identity, or through a slot table)
__device__ __forceinline__ int weight_index(const ft_moe_layer_weights& W, int e) {
    if (W.expert_to_slot == nullptr) return e;
    const int s = W.expert_to_slot[e];
    if (s < 0 || s >= W.n_weights) {
        raise_dev_error(FT_DEVERR_BAD_INDEX);
        return -1;
    }
    return s;
}

}  // namespace ft
