/*
 * ftoracle.c -- plain, slow, fp64 CPU oracle of the sparse-MoE layer step over
 * NVFP4 expert weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this library; the CUDA path never does,
 * and it shares no code, header or table with it.
 *
 * What it follows:
 *  - Router: "a linear layer plus softmax gives each expert a probability, the
 *    top-K experts are taken and their outputs weighted" -- page "FreeToken：
 *    753B大模型塞进单卡的本地部署硬件账该怎么算", paragraph on the MoE core
 *    mechanism (MoE的核心机制).  Logits are the input here; selection runs on
 *    the fp32 logits with equal values going to the lower expert index, and the
 *    k selected probabilities are renormalised to sum to one.
 *  - Experts: each expert is an independent FFN with its own weights (same
 *    paragraph); the FFN is SwiGLU: y = Wd (silu(Wg x) * (Wu x)).
 *  - Weights: NVFP4 as used by the page "8GB 笔记本 39.3 tok/s、单卡跑 753B：
 *    FreeToken 把 frontier MoE 拉回本地" (sections 为什么 frontier 模型…,
 *    实测六款消费级硬件, 局限).  Bit-level format: E2M1 element codes (OCP
 *    Microscaling Formats v1.0, FP4 E2M1: bias 1, no inf/NaN, max 6), one E4M3
 *    scale per 16 consecutive elements along the reduction dimension (OCP 8-bit
 *    floating point, E4M3: bias 7, max 448, S.1111.111 is NaN), and one fp32
 *    scale per tensor.  Dequantised value = e2m1 * e4m3 * tensor_scale, exact
 *    in fp64.
 *  - Activations are bf16; h = silu(g)*u is rounded to bf16 before the down
 *    projection; the combined output is rounded to bf16.  Everything else is
 *    fp64.
 *
 * The quantisers (weights and, for the block-scaled tensor-core path,
 * activations) are definitions of data, so they are written in fp32 exactly
 * as specified below; every other step is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORA_API __attribute__((visibility("default")))

enum { ORA_OK = 0, ORA_ERR_ARG = 1 };

/* ------------------------------------------------------------------------- */
/* number formats                                                             */
/* ------------------------------------------------------------------------- */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * exponent 0 is subnormal: value m * 0.5; otherwise 2^(e-1) * (1 + m/2). */
ORA_API double ora_e2m1_value(uint8_t code) {
    const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * exponent 0 is subnormal: m * 2^-9; S.1111.111 is NaN (returns NAN). */
ORA_API double ora_e4m3_value(uint8_t b) {
    if ((b & 0x7F) == 0x7F) return NAN;
    const int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    const double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest E2M1 code to v (fp32), ties to the even code, |v| > 6 saturates to
 * 6, and a value that rounds to zero is encoded as +0 (code 0). */
ORA_API uint8_t ora_e2m1_encode(float v) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    const double a = fabs((double)v);
    int c = 7;
    if (a < 6.0) {
        int i = 0;
        while (!(a < grid[i + 1])) ++i; /* grid[i] <= a < grid[i+1] */
        const double mid = 0.5 * (grid[i] + grid[i + 1]);
        if (a < mid)
            c = i;
        else if (a > mid)
            c = i + 1;
        else
            c = (i % 2 == 0) ? i : i + 1; /* tie: the even code */
    }
    if (c == 0) return 0;
    return (uint8_t)(((v < 0.0f) ? 8 : 0) | c);
}

/* Nearest non-negative E4M3 code to r >= 0 (fp32), ties to the even code,
 * saturating to 448 (0x7E). */
ORA_API uint8_t ora_e4m3_encode(float r) {
    const double a = (double)r;
    if (!(a < 448.0)) return 0x7E;
    int lo = 0; /* largest code whose value is <= a */
    for (int c = 1; c <= 0x7E; ++c)
        if (ora_e4m3_value((uint8_t)c) <= a) lo = c;
    if (ora_e4m3_value((uint8_t)lo) == a) return (uint8_t)lo;
    const double vlo = ora_e4m3_value((uint8_t)lo), vhi = ora_e4m3_value((uint8_t)(lo + 1));
    const double mid = 0.5 * (vlo + vhi);
    if (a < mid) return (uint8_t)lo;
    if (a > mid) return (uint8_t)(lo + 1);
    return (uint8_t)((lo % 2 == 0) ? lo : lo + 1);
}

/* Round an fp64 value to the nearest bf16 value (8 significant bits, fp32
 * exponent range, ties to even), returned as fp64. */
ORA_API double ora_bf16_round(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    (void)frexp(v, &e);                 /* |v| in [2^(e-1), 2^e) */
    const int q = (e >= -125) ? e - 8 : -133; /* exponent of one unit in the last place */
    const double r = ldexp(rint(ldexp(v, -q)), q);
    if (fabs(r) >= 0x1.0p128) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

/* ------------------------------------------------------------------------- */
/* quantisation (fp32 arithmetic, as defined)                                 */
/* ------------------------------------------------------------------------- */

/* One 16-element block with scale divisor s (the tensor scale; 1 for
 * activations): sb = E4M3(amax/6/s); eff = e4m3(sb)*s; code = E2M1(w/eff). */
static void quant_block16(const float* w, float s, uint8_t* codes16, uint8_t* sb_out) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        const float a = fabsf(w[i]);
        if (a > amax) amax = a;
    }
    const float d = amax / 6.0f;
    const float r = d / s;
    const uint8_t sb = ora_e4m3_encode(r);
    *sb_out = sb;
    const float eff = (float)ora_e4m3_value(sb) * s;
    for (int i = 0; i < 16; ++i) codes16[i] = (eff == 0.0f) ? 0 : ora_e2m1_encode(w[i] / eff);
}

static void pack_row(const uint8_t* codes, int64_t K, uint8_t* packed) {
    for (int64_t j = 0; j < K / 2; ++j) packed[j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
}

/* Weight tensor [N, K] -> packed codes [N, K/2] (low nibble = even element),
 * scales [N, K/16], tensor scale.  s_t = amax/(6*448) in fp32, or 1 when the
 * tensor is zero or that quotient underflows to zero. */
ORA_API int ora_quantize_weight(const float* w, int64_t N, int64_t K, uint8_t* codes, uint8_t* scales,
                                float* tensor_scale) {
    if (N <= 0 || K <= 0 || K % 16 != 0) return ORA_ERR_ARG;
    float amax = 0.0f;
    int bad = 0;
#pragma omp parallel for reduction(max : amax) reduction(| : bad)
    for (int64_t i = 0; i < N * K; ++i) {
        if (!isfinite(w[i])) bad = 1;
        const float a = fabsf(w[i]);
        if (a > amax) amax = a;
    }
    if (bad) return ORA_ERR_ARG;
    float st = amax / 2688.0f;
    if (st == 0.0f) st = 1.0f;
    *tensor_scale = st;
    /* rows are independent: the row loop may run on several threads */
#pragma omp parallel
    {
        uint8_t* tmp = (uint8_t*)malloc((size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t b = 0; b < K / 16; ++b)
                quant_block16(w + n * K + b * 16, st, tmp + b * 16, scales + n * (K / 16) + b);
            pack_row(tmp, K, codes + n * (K / 2));
        }
        free(tmp);
    }
    return ORA_OK;
}

/* Activation rows [T, K] (fp32 values, here always bf16-exact) -> NVFP4 with
 * unit tensor scale: sb = E4M3(amax/6), code = E2M1(x/e4m3(sb)). */
ORA_API int ora_quantize_act(const float* x, int64_t T, int64_t K, uint8_t* codes, uint8_t* scales) {
    if (T <= 0 || K <= 0 || K % 16 != 0) return ORA_ERR_ARG;
    uint8_t* tmp = (uint8_t*)malloc((size_t)K);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t b = 0; b < K / 16; ++b) quant_block16(x + t * K + b * 16, 1.0f, tmp + b * 16, scales + t * (K / 16) + b);
        pack_row(tmp, K, codes + t * (K / 2));
    }
    free(tmp);
    return ORA_OK;
}

/* Dequantise [N, K] packed NVFP4 to fp64: e2m1(code) * e4m3(scale) * s_t. */
ORA_API int ora_dequantize(const uint8_t* codes, const uint8_t* scales, double tensor_scale, int64_t N, int64_t K,
                           double* out) {
    if (N <= 0 || K <= 0 || K % 16 != 0) return ORA_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const uint8_t byte = codes[n * (K / 2) + k / 2];
            const uint8_t c = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            const double s = ora_e4m3_value(scales[n * (K / 16) + k / 16]);
            if (isnan(s) || s < 0) bad = 1;
            out[n * K + k] = ora_e2m1_value(c) * s * tensor_scale;
        }
    return bad ? ORA_ERR_ARG : ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* router                                                                     */
/* ------------------------------------------------------------------------- */

/* ids[t, j]: the j-th largest logit of row t (ties -> lower expert index);
 * w[t, j] = exp(l_j - m) / sum_{i in top-k} exp(l_i - m), m the row maximum,
 * i.e. softmax over all experts followed by renormalisation over the k
 * selected.  A row whose maximum is -inf gets weights 1/k.  NaN and +inf
 * logits are invalid. */
ORA_API int ora_route(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
    if (T < 0 || E <= 0 || k <= 0 || k > E) return ORA_ERR_ARG;
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        for (int e = 0; e < E; ++e)
            if (isnan(l[e]) || l[e] == INFINITY) {
                free(taken);
                return ORA_ERR_ARG;
            }
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: equal keeps the lower index */
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        const double m = (double)l[ids[(int64_t)t * k]];
        if (m == -INFINITY) {
            for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = 1.0 / k;
            continue;
        }
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp((double)l[ids[(int64_t)t * k + j]] - m);
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = exp((double)l[ids[(int64_t)t * k + j]] - m) / den;
    }
    free(taken);
    return ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* permutation                                                                */
/* ------------------------------------------------------------------------- */

/* Stable counting sort of the T*k slots f = t*k + j by expert ids[f]:
 * offsets[e] = number of slots with a smaller expert id (offsets[E] = T*k),
 * perm[p] = f for the p-th slot in (expert, f) order, inv[f] = p. */
ORA_API int ora_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* perm, int32_t* inv) {
    if (T < 0 || E <= 0 || k <= 0) return ORA_ERR_ARG;
    const int64_t n = (int64_t)T * k;
    for (int64_t f = 0; f < n; ++f)
        if (ids[f] < 0 || ids[f] >= E) return ORA_ERR_ARG;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t f = 0; f < n; ++f) offsets[ids[f] + 1] += 1;
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t f = 0; f < n; ++f) {
        const int e = ids[f];
        const int32_t p = offsets[e] + fill[e]++;
        perm[p] = (int32_t)f;
        inv[f] = p;
    }
    free(fill);
    return ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* expert FFN                                                                 */
/* ------------------------------------------------------------------------- */

static double silu(double z) { return z / (1.0 + exp(-z)); }

static double dot(const double* a, const double* b, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

static void deq_vec(const uint8_t* codes, const uint8_t* scales, int64_t K, double* out) {
    for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = codes[k / 2];
        const uint8_t c = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        out[k] = ora_e2m1_value(c) * ora_e4m3_value(scales[k / 16]);
    }
}

/* One expert over R rows of activations.
 *
 * Wg, Wu are the dequantised [I, H] gate/up matrices and Wd the [H, I] down
 * matrix (fp64, from ora_dequantize).  x: [R, H] fp64 (bf16-exact values).
 * mode 0 (bf16 activations): g = Wg x, u = Wu x, h = bf16(silu(g) u), y = Wd h.
 * mode 1 (NVFP4 activations, for the block-scaled tensor-core path): x is
 * first quantised per 16 along H with unit tensor scale, and h (after its
 * bf16 rounding) per 16 along I; the products use the dequantised values.
 * h_out [R, I] (optional) receives h after rounding, y: [R, H]. */
ORA_API int ora_expert_ffn(const double* Wg, const double* Wu, const double* Wd, int64_t H, int64_t I,
                           const double* x, int64_t R, int mode, double* h_out, double* y) {
    if (H <= 0 || I <= 0 || R < 0 || H % 16 || I % 16 || (mode != 0 && mode != 1)) return ORA_ERR_ARG;
    int err = 0;
#pragma omp parallel
    {
        double* xa = (double*)malloc(sizeof(double) * (size_t)H);
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        float* f = (float*)malloc(sizeof(float) * (size_t)(H > I ? H : I));
        uint8_t* qc = (uint8_t*)malloc((size_t)(H > I ? H : I) / 2);
        uint8_t* qs = (uint8_t*)malloc((size_t)(H > I ? H : I) / 16);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            const double* xr = x + r * H;
            if (mode == 1) {
                for (int64_t i = 0; i < H; ++i) f[i] = (float)xr[i];
                if (ora_quantize_act(f, 1, H, qc, qs) != ORA_OK) err = 1;
                deq_vec(qc, qs, H, xa);
            } else {
                memcpy(xa, xr, sizeof(double) * (size_t)H);
            }
            for (int64_t i = 0; i < I; ++i) {
                const double g = dot(Wg + i * H, xa, H);
                const double u = dot(Wu + i * H, xa, H);
                h[i] = ora_bf16_round(silu(g) * u);
            }
            if (h_out) memcpy(h_out + r * I, h, sizeof(double) * (size_t)I);
            if (mode == 1) {
                for (int64_t i = 0; i < I; ++i) f[i] = (float)h[i];
                if (ora_quantize_act(f, 1, I, qc, qs) != ORA_OK) err = 1;
                deq_vec(qc, qs, I, h);
            }
            for (int64_t n = 0; n < H; ++n) y[r * H + n] = dot(Wd + n * I, h, I);
        }
        free(xa);
        free(h);
        free(f);
        free(qc);
        free(qs);
    }
    return err ? ORA_ERR_ARG : ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* combine                                                                    */
/* ------------------------------------------------------------------------- */

/* out[t, n] = bf16( sum_{j=0..k-1} w[t, j] * y[inv[t*k + j], n] ), summed in
 * fp64 in j order.  out_pre (optional) receives the sum before rounding. */
ORA_API int ora_combine(const double* y, const int32_t* inv, const double* w, int T, int k, int64_t H, double* out,
                        double* out_pre) {
    if (T < 0 || k <= 0 || H <= 0) return ORA_ERR_ARG;
    for (int t = 0; t < T; ++t)
        for (int64_t n = 0; n < H; ++n) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += w[(int64_t)t * k + j] * y[(int64_t)inv[(int64_t)t * k + j] * H + n];
            if (out_pre) out_pre[(int64_t)t * H + n] = s;
            out[(int64_t)t * H + n] = ora_bf16_round(s);
        }
    return ORA_OK;
}

ORA_API void ora_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

ORA_API int ora_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
