// decode_fused.cu -- one persistent launch per MoE layer for small token
// counts (decode): router top-k, expert grouping, NVFP4 gate/up projection with
// SwiGLU, down projection and routing-weighted combine.
//
// The step follows the page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算"
// (MoE core mechanism: linear + softmax router, top-K experts, weighted sum of
// independent expert FFNs).  Decode is bound by streaming the selected
// experts' weights from HBM, so the kernel is organised around that stream:
//
//  * Weights sit in HBM in 16-row tiles (ft_nvfp4_pack_tiles): a tile of a
//    [N][K] matrix holds, per 128-element K-block, 1 KB of codes arranged so
//    that the 32 lanes of a warp read 16 conflict-free bytes each, then 128 B
//    of E4M3 scales (4 per lane).  One tile is one contiguous bulk copy.
//  * One producer warp streams tiles with cp.async.bulk into a ring of shared
//    memory stages guarded by mbarriers; 16 consumer warps decode E2M1 pairs to
//    f16 in registers (exact), multiply by the block scale in f16 (exact: at
//    most 6 significant bits, magnitudes in [2^-10, 2688]) and feed mma.sync
//    m16n8k16 with fp32 accumulation.  The tensor cores only take over the
//    multiply-adds of this HBM-bound GEMV; tokens are the mma's N.
//  * Prologue: every CTA routes redundantly (top-k by rank, so all threads
//    work at once), groups the (token, slot) pairs by expert and stages the
//    activations as f16, all before the first weight byte is needed.
//  * Phase 1 (gate/up) splits the selected experts' gate/up tiles evenly over
//    the CTAs; each CTA writes h = bf16(silu(g) * u) for its pairs.  A bounded
//    grid barrier follows.  Phase 2 (down + combine) gives each CTA a range of
//    output rows for all selected experts, so the weighted sum over experts is
//    accumulated in a fixed order in shared memory.  Phase-2 tiles are
//    prefetched into the ring while phase 1 runs; several experts' tiles share
//    one ring slot.
//  * Grid = one CTA per SM, all co-resident, which the barrier relies on.
//    Every wait is bounded by a %globaltimer budget; on expiry the kernel
//    sets FT_DEVERR_TIMEOUT and finishes without trapping.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace ft {

namespace dk {
constexpr int NCW = 16;                  // consumer warps
constexpr int THREADS = 32 * (NCW + 1);  // + one producer warp
constexpr int MAXT = 16;                 // tokens per launch
constexpr int MAXK = 32;                 // experts per token
constexpr int MAXF = MAXT * MAXK;        // (token, slot) pairs
constexpr int TG = 8;                    // tokens per mma pass (mma N)
constexpr int MAXNS = 8;                 // ring stages
constexpr int MAXU = MAXF;               // selected experts per launch
constexpr int MAX_OUT_TILES = 4;         // 16-row output tiles per CTA in phase 2
constexpr unsigned long long WAIT_NS = 2000000000ull;  // bound on any single wait
}  // namespace dk

struct DecodeArgs {
    ft_moe_layer_weights W;
    const float* logits;      // route mode: [T][E]
    const int32_t* offsets;   // grouped mode: [E+1]
    const int32_t* perm;      // grouped mode: [T*k]
    const float* w_in;        // grouped mode: [T][k]
    const uint16_t* x;        // [T][H] bf16
    uint16_t* out;            // [T][H] bf16, optional
    float* y;                 // [T*k][H] fp32 per permuted row, optional (grouped mode)
    int32_t* ids_out;         // route mode, optional
    float* w_out;             // route mode, optional
    uint16_t* hbuf;           // [T*k][I] bf16
    unsigned int* bar;        // grid barrier counter (monotonic, starts at 0)
    int T, k;
    int stage_bytes, nstages;
    int xs_stride;            // halves per staged row (general path; both phases)
    int xs_bytes;             // bytes of the staging area
    int tge;                  // token columns per mma pass (<= 8)
    int fast;                 // all x rows and all h rows fit in the staging area
};

struct DecodeSmem {
    unsigned long long full[dk::MAXNS];
    unsigned long long empty[dk::MAXNS];
    int ids[dk::MAXF];         // route mode: expert of slot f = t*k + j
    float wts[dk::MAXF];       // routing weight of slot f
    float selv[dk::MAXF];      // route mode: selected logit of slot f
    int plist[dk::MAXF];       // slots grouped by expert ascending, increasing f within an expert
    int pexp[dk::MAXF];        // expert of plist position p
    int rexp[dk::MAXF];        // power-of-two pre-scale of staged h row p (fast path)
    int ulist[dk::MAXU];       // selected experts, ascending
    int ubeg[dk::MAXU + 1];    // plist range of each selected expert
    int uwi[dk::MAXU];         // weight index of each selected expert (-1: invalid slot)
    float uts[dk::MAXU][3];    // tensor scales (gate, up, down) of each selected expert
    int U;
    int flag;
    int xexp[dk::MAXT];        // power-of-two pre-scale of staged x rows
    float oacc[dk::MAX_OUT_TILES][16][dk::MAXT];
};

// ---------------------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and the device error bit) on expiry.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, uint32_t parity) {
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(b, parity)) {
        if (globaltimer() - t0 > dk::WAIT_NS) {
            raise_dev_error(FT_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(b))
                 : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(dk::NCW * 32) : "memory"); }

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t byte_of(const uint4& v, int b) {
    const uint32_t w = (b < 4) ? v.x : (b < 8) ? v.y : (b < 12) ? v.z : v.w;
    return (w >> (8 * (b & 3))) & 0xFFu;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return (i == 0) ? v.x : (i == 1) ? v.y : (i == 2) ? v.z : v.w;
}

// ---------------------------------------------------------------------------- tile math

// Partial products of one 16-row tile over K-blocks kb0, kb0+step, ... (K = 128*KB)
// against staged f16 activation rows into the mma accumulator d (rows g, g+8;
// token columns 2q, 2q+1).  `xrow` is this lane's activation row (column g).
//
// Lane (g, q) owns the 16 code bytes q of rows g and g+8 of each K-block, i.e.
// 32 consecutive elements per row.  mma s (of 8 per K-block) takes elements
// 4s..4s+3 of them: the pair 4s, 4s+1 as the fragment's k = 2q, 2q+1 and the
// pair 4s+2, 4s+3 as k = 2q+8, 2q+9.  The activations are read at the same
// element positions, so the dot product is unchanged by this K order.
__device__ __forceinline__ void tile_partial(const uint8_t* tile, int KB, int kb0, int step, const __half* xrow,
                                             float (&d)[4]) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const uint8_t* scl = tile + KB * 1024;
    const __half* xr0 = xrow + 32 * q;
    for (int kb = kb0; kb < KB; kb += step) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(tile + kb * 1024 + (q * 8 + g) * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(tile + kb * 1024 + 512 + (q * 8 + g) * 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(scl + kb * 128 + (q * 8 + g) * 4);
        const uint32_t sg0 = e4m3_to_f16x2_bcast(sc & 0xFFu), sg1 = e4m3_to_f16x2_bcast((sc >> 8) & 0xFFu);
        const uint32_t sh0 = e4m3_to_f16x2_bcast((sc >> 16) & 0xFFu), sh1 = e4m3_to_f16x2_bcast(sc >> 24);
        const __half* xr = xr0 + kb * 128;
        uint4 xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = *reinterpret_cast<const uint4*>(xr + 8 * i);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t sa = (s < 4) ? sg0 : sg1, sb = (s < 4) ? sh0 : sh1;
            const uint32_t a0 = hmul2(e2m1x2_to_f16x2(byte_of(c0, 2 * s)), sa);
            const uint32_t a2 = hmul2(e2m1x2_to_f16x2(byte_of(c0, 2 * s + 1)), sa);
            const uint32_t a1 = hmul2(e2m1x2_to_f16x2(byte_of(c1, 2 * s)), sb);
            const uint32_t a3 = hmul2(e2m1x2_to_f16x2(byte_of(c1, 2 * s + 1)), sb);
            const uint32_t b0 = word_of(xv[s >> 1], (2 * s) & 3);
            const uint32_t b1 = word_of(xv[s >> 1], (2 * s + 1) & 3);
            mma16816(d, a0, a1, a2, a3, b0, b1);
        }
    }
}

// red layout: [NCW][16 rows][tge token columns]
__device__ __forceinline__ void store_partial(float* red, int tge, int warp, const float (&d)[4], int ntok) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    float* r = red + warp * 16 * tge;
    if (2 * q < ntok) {
        r[g * tge + 2 * q] = d[0];
        r[(g + 8) * tge + 2 * q] = d[2];
    }
    if (2 * q + 1 < ntok) {
        r[g * tge + 2 * q + 1] = d[1];
        r[(g + 8) * tge + 2 * q + 1] = d[3];
    }
}

// Stage `n` rows of `K` bf16 values as f16 into xs (row stride `stride`
// halves), row r from src + row_off(r), by `nthr` threads with index `ti`;
// `sync` is the barrier of those threads.  Rows whose values would not fit
// f16 are pre-scaled by a power of two recorded in exps[r] (0 normally).
template <typename RowOff, typename Sync>
__device__ void stage_rows(int* exps, int* flag, __half* xs, int stride, const uint16_t* src, int n, int K,
                           RowOff row_off, int ti, int nthr, Sync sync) {
    const int per_row = K / 8;
    for (int r = ti; r < n; r += nthr) exps[r] = 0;
    if (ti == 0) *flag = 0;
    sync();
    bool big = false;
    for (int idx = ti; idx < n * per_row; idx += nthr) {
        const int r = idx / per_row, c = idx - r * per_row;
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src + row_off(r) + (int64_t)c * 8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = bf16_to_f32((uint16_t)(w[i] & 0xFFFFu)), hi = bf16_to_f32((uint16_t)(w[i] >> 16));
            big |= !(fabsf(lo) < 60000.0f) || !(fabsf(hi) < 60000.0f);
            const __half2 h = __floats2half2_rn(lo, hi);
            o[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(xs + r * stride + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (big) *flag = 1;
    sync();
    if (*flag) {  // rare: rescale rows by a power of two so that they fit f16
        const int w = ti >> 5, lane = ti & 31, nw = nthr >> 5;
        for (int r = w; r < n; r += nw) {
            float m = 0.0f;
            for (int i = lane; i < K; i += 32) m = fmaxf(m, fabsf(bf16_to_f32(__ldcg(src + row_off(r) + i))));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) exps[r] = (m >= 16384.0f) ? ilogbf(m) - 14 : 0;
        }
        sync();
        for (int idx = ti; idx < n * K; idx += nthr) {
            const int r = idx / K, c = idx - r * K;
            xs[r * stride + c] = __float2half_rn(ldexpf(bf16_to_f32(__ldcg(src + row_off(r) + c)), -exps[r]));
        }
        sync();
    }
}

// ---------------------------------------------------------------------------- work split

struct Split {
    int64_t p1_beg, p1_end;  // phase-1 tiles (over all selected experts' gate/up tiles)
    int o_beg, o_end;        // phase-2 output tiles (16 rows of H)
};

__device__ __forceinline__ Split split_work(int U, int I, int H, int G, int c) {
    Split s;
    const int64_t n1 = (int64_t)U * (2 * I / 16);
    s.p1_beg = n1 * c / G;
    s.p1_end = n1 * (c + 1) / G;
    const int n2 = H / 16;
    s.o_beg = (int)((int64_t)n2 * c / G);
    s.o_end = (int)((int64_t)n2 * (c + 1) / G);
    return s;
}

// ---------------------------------------------------------------------------- kernel

__global__ void __launch_bounds__(dk::THREADS, 1) k_moe_decode(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(dsm);
    uint8_t* ring = dsm + ((sizeof(DecodeSmem) + 127) / 128) * 128;
    __half* xs = reinterpret_cast<__half*>(ring + (size_t)a.nstages * a.stage_bytes);
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + a.xs_bytes);

    const ft_moe_layer_weights& W = a.W;
    const int H = W.H, I = W.I, E = W.E, T = a.T, k = a.k;
    const int nf = T * k;
    const int tge = a.tge;          // token columns per pass (<= 8)
    const bool fast = a.fast != 0;  // all x rows and all h rows fit in xs
    // staged-row strides in halves: the fast path holds T rows of H, then nf rows of I; the
    // general path holds tge rows of either, at the wider stride
    const int xstride = fast ? H + 8 : a.xs_stride;
    const int hstride = fast ? I + 8 : a.xs_stride;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    auto all_sync = [] { __syncthreads(); };

    // ---------------- prologue (all warps): barriers, x, routing, grouping
    if (tid < dk::MAXNS) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < dk::MAX_OUT_TILES * 16 * dk::MAXT; i += dk::THREADS) (&sm.oacc[0][0][0])[i] = 0.0f;
    float* scratch = reinterpret_cast<float*>(ring);  // the ring is free until the producer starts
    if (a.logits) {
        for (int i = tid; i < T * E; i += dk::THREADS) scratch[i] = a.logits[i];
        for (int f = tid; f < nf; f += dk::THREADS) sm.ids[f] = f % k;  // stays in range if logits are NaN
    } else {
        for (int i = tid; i <= E; i += dk::THREADS) reinterpret_cast<int*>(scratch)[i] = a.offsets[i];
        for (int f = tid; f < nf; f += dk::THREADS) {
            int pf = a.perm[f];
            if (pf < 0 || pf >= nf) {
                raise_dev_error(FT_DEVERR_BAD_INDEX);
                pf = 0;
            }
            sm.plist[f] = pf;
            sm.wts[f] = a.w_in[f];
        }
    }
    if (fast)  // all T activation rows, once (its barriers also publish the loads above)
        stage_rows(sm.xexp, &sm.flag, xs, xstride, a.x, T, H, [&](int r) { return (int64_t)r * H; }, tid,
                   dk::THREADS, all_sync);
    else
        __syncthreads();

    if (a.logits) {
        // top-k by rank: candidate e of token t has rank #{e2 : l2 > l or (l2 == l and e2 < e)};
        // equal logits go to the lower expert id, as in ft_moe_route
        bool bad = false;
        for (int cand = tid; cand < T * E; cand += dk::THREADS) {
            const int t = cand / E, e = cand - t * E;
            const float* row = scratch + t * E;
            const float v = row[e];
            bad |= (v != v) || (v == INFINITY);
            int r = 0;
            for (int e2 = 0; e2 < E; ++e2) {
                const float v2 = row[e2];
                r += (v2 > v) || (v2 == v && e2 < e);
            }
            if (r < k) {
                sm.ids[t * k + r] = e;
                sm.selv[t * k + r] = v;
            }
        }
        if (bad) raise_dev_error(FT_DEVERR_NAN_LOGIT);
        __syncthreads();
        if (warp < T) {  // weights as the router computes them: exp(l_j - l_0) / sum, same butterfly sum
            const float vj = (lane < k) ? sm.selv[warp * k + lane] : -INFINITY;
            const float m = __shfl_sync(0xffffffffu, vj, 0);
            float wj;
            if (m == -INFINITY || m != m) {
                wj = 1.0f / (float)k;
            } else {
                const float ej = (lane < k) ? expf(vj - m) : 0.0f;
                const float sum = warp_sum(ej);
                wj = ej / sum;
            }
            if (lane < k) {
                sm.wts[warp * k + lane] = wj;
                if (c == 0 && a.ids_out) {
                    a.ids_out[warp * k + lane] = sm.ids[warp * k + lane];
                    a.w_out[warp * k + lane] = wj;
                }
            }
        }
        // grouping: plist position of slot f = #{f2 : e2 < e} + #{f2 < f : e2 == e}
        for (int f = tid; f < nf; f += dk::THREADS) {
            const int e = sm.ids[f];
            int pos = 0;
            for (int f2 = 0; f2 < nf; ++f2) {
                const int e2 = sm.ids[f2];
                pos += (e2 < e) || (e2 == e && f2 < f);
            }
            sm.plist[pos] = f;
            sm.pexp[pos] = e;
        }
    } else {
        const int* offs = reinterpret_cast<const int*>(scratch);
        for (int p = tid; p < nf; p += dk::THREADS) {  // expert owning position p: last e with offs[e] <= p
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (offs[mid] <= p) lo = mid;
                else hi = mid - 1;
            }
            if (offs[lo] > p || offs[lo + 1] <= p || offs[E] != nf) raise_dev_error(FT_DEVERR_BAD_INDEX);
            sm.pexp[p] = lo;
        }
    }
    __syncthreads();
    // selected experts = segment starts of pexp
    for (int p = tid; p < nf; p += dk::THREADS) {
        if (p == 0 || sm.pexp[p] != sm.pexp[p - 1]) {
            int u = 0;
            for (int p2 = 1; p2 <= p; ++p2) u += (sm.pexp[p2] != sm.pexp[p2 - 1]);
            sm.ulist[u] = sm.pexp[p];
            sm.ubeg[u] = p;
        }
    }
    if (tid == 0) {
        int u = (nf > 0) ? 1 : 0;
        for (int p2 = 1; p2 < nf; ++p2) u += (sm.pexp[p2] != sm.pexp[p2 - 1]);
        sm.U = u;
        sm.ubeg[u] = nf;
    }
    __syncthreads();
    const int U = sm.U;
    for (int u = tid; u < U; u += dk::THREADS) {
        const int wi = weight_index(W, sm.ulist[u]);
        sm.uwi[u] = wi;
        for (int j = 0; j < 3; ++j) sm.uts[u][j] = (wi >= 0) ? W.tscale[(int64_t)wi * W.tscale_stride + j] : 0.0f;
    }
    __syncthreads();

    const Split sp = split_work(U, I, H, G, c);
    const int tiles_gu = 2 * I / 16;
    const int KB1 = H / 128, KB2 = I / 128;
    const int bytes1 = 9 * H, bytes2 = 9 * I;  // one 16-row tile of [.][H] or [.][I]
    const int J = fast ? max(1, min(a.stage_bytes / bytes2, dk::NCW)) : 1;  // experts per phase-2 slot
    const int n_p1 = (int)(sp.p1_end - sp.p1_beg);
    const int n_ot = sp.o_end - sp.o_beg;
    const int n_jg = (U + J - 1) / J;  // expert groups per output tile
    const int n_chunks = n_p1 + n_ot * n_jg;

    if (warp == dk::NCW) {
        // ---------------- producer: stream tiles into the ring
        if (lane == 0) {
            for (int n = 0; n < n_chunks; ++n) {
                const int s = n % a.nstages, use = n / a.nstages;
                if (use > 0 && !mbar_wait(&sm.empty[s], (use - 1) & 1)) break;
                uint8_t* dst = ring + (size_t)s * a.stage_bytes;
                if (n < n_p1) {
                    const int64_t t = sp.p1_beg + n;
                    const int u = (int)(t / tiles_gu), lt = (int)(t % tiles_gu);
                    const int wi = sm.uwi[u];
                    if (wi < 0) {
                        mbar_arrive(&sm.full[s]);
                    } else {
                        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)bytes1);
                        bulk_g2s(dst, W.gu_codes + (int64_t)wi * W.gu_codes_stride + (int64_t)lt * bytes1,
                                 (uint32_t)bytes1, &sm.full[s]);
                    }
                } else {
                    const int m = n - n_p1;
                    const int jg = m / n_ot, ot = sp.o_beg + m % n_ot;
                    const int u0 = jg * J, nj = min(J, U - u0);
                    uint32_t tx = 0;
                    for (int jj = 0; jj < nj; ++jj) tx += (sm.uwi[u0 + jj] >= 0) ? (uint32_t)bytes2 : 0u;
                    mbar_arrive_expect_tx(&sm.full[s], tx);
                    for (int jj = 0; jj < nj; ++jj) {
                        const int wi = sm.uwi[u0 + jj];
                        if (wi >= 0)
                            bulk_g2s(dst + jj * bytes2,
                                     W.d_codes + (int64_t)wi * W.d_codes_stride + (int64_t)ot * bytes2,
                                     (uint32_t)bytes2, &sm.full[s]);
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers (warps 0 .. NCW-1)
    auto csync = [] { consumer_sync(); };
    const int g8 = lane >> 2;  // this lane's mma column
    int buf = 0;
    int staged_u = -1, staged_g = -1;
    for (int n = 0; n < n_p1; ++n) {
        const int s = n % a.nstages, use = n / a.nstages;
        const int64_t t = sp.p1_beg + n;
        const int u = (int)(t / tiles_gu), lt = (int)(t % tiles_gu);
        const int wi = sm.uwi[u];
        const int pb = sm.ubeg[u], tu = sm.ubeg[u + 1] - pb;
        mbar_wait(&sm.full[s], use & 1);
        const uint8_t* tile = ring + (size_t)s * a.stage_bytes;
        const int ngroups = (tu + tge - 1) / tge;
        for (int gi = 0; gi < ngroups; ++gi) {
            const int g0 = gi * tge, nt = min(tge, tu - g0);
            if (!fast && (staged_u != u || staged_g != gi)) {
                csync();  // earlier readers of xs / xexp are done
                stage_rows(sm.xexp, &sm.flag, xs, xstride, a.x, nt, H,
                           [&](int r) { return (int64_t)(sm.plist[pb + g0 + r] / k) * H; }, tid, dk::NCW * 32, csync);
                staged_u = u;
                staged_g = gi;
            }
            const int col = min(g8, nt - 1);
            const int xr = fast ? sm.plist[pb + g0 + col] / k : col;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            if (wi >= 0) tile_partial(tile, KB1, warp, dk::NCW, xs + xr * xstride, d);
            float* rb = red + buf * dk::NCW * 16 * tge;
            store_partial(rb, tge, warp, d, nt);
            consumer_sync();
            if (gi == ngroups - 1 && tid == 0) mbar_arrive(&sm.empty[s]);
            if (tid < 8 * nt) {
                const int p = tid / nt, tt = tid - p * nt;
                const int nw = min(dk::NCW, KB1);
                float gs = 0.f, us = 0.f;
                for (int w = 0; w < nw; ++w) {
                    gs += rb[(w * 16 + 2 * p) * tge + tt];
                    us += rb[(w * 16 + 2 * p + 1) * tge + tt];
                }
                const int f = sm.plist[pb + g0 + tt];
                float hv = 0.0f;
                if (wi >= 0) {
                    const float sc = ldexpf(1.0f, sm.xexp[fast ? f / k : tt]);
                    hv = silu_f32(gs * sm.uts[u][0] * sc) * (us * sm.uts[u][1] * sc);
                }
                a.hbuf[(int64_t)f * I + lt * 8 + p] = bf16_bits(hv);
            }
            buf ^= 1;
        }
    }

    // ---------------- grid barrier: every CTA's h is written
    __threadfence();
    consumer_sync();
    if (tid == 0) {
        const unsigned int old = atomicAdd(a.bar, 1u);
        const unsigned int target = (old / (unsigned)G + 1u) * (unsigned)G;
        const unsigned long long t0 = globaltimer();
        while (true) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.bar) : "memory");
            if ((int)(v - target) >= 0) break;
            if (globaltimer() - t0 > dk::WAIT_NS) {
                raise_dev_error(FT_DEVERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
    }
    consumer_sync();

    // ---------------- phase 2: down projection and combine over this CTA's output rows
    if (fast && n_ot > 0)  // all h rows in plist order, once
        stage_rows(sm.rexp, &sm.flag, xs, hstride, a.hbuf, nf, I,
                   [&](int r) { return (int64_t)sm.plist[r] * I; }, tid, dk::NCW * 32, csync);
    staged_u = -1;
    staged_g = -1;
    const int wpe = dk::NCW / J;  // warps per expert of a slot
    for (int m = 0; m < n_ot * n_jg; ++m) {
        const int n = n_p1 + m;
        const int s = n % a.nstages, use = n / a.nstages;
        const int jg = m / n_ot, otl = m % n_ot, ot = sp.o_beg + otl;
        const int u0 = jg * J, nj = min(J, U - u0);
        mbar_wait(&sm.full[s], use & 1);
        const uint8_t* slot = ring + (size_t)s * a.stage_bytes;
        if (fast) {
            // warp w works on expert jj = w / wpe of the slot, K-blocks w % wpe, w % wpe + wpe, ...
            const int jj = warp / wpe;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            int nt = 1;
            if (jj < nj) {
                const int u = u0 + jj;
                const int pb = sm.ubeg[u], tu = sm.ubeg[u + 1] - pb;
                nt = tu;
                const int xr = pb + min(g8, tu - 1);
                if (sm.uwi[u] >= 0) tile_partial(slot + jj * bytes2, KB2, warp % wpe, wpe, xs + xr * hstride, d);
            }
            float* rb = red + buf * dk::NCW * 16 * tge;
            store_partial(rb, tge, warp, d, min(nt, tge));
            consumer_sync();
            if (tid == 0) mbar_arrive(&sm.empty[s]);
            if (tid < 16 * T) {  // (row r, token tok): add this slot's experts in ascending order
                const int r = tid / T, tok = tid - r * T;
                const int nw = min(wpe, KB2);
                float acc = sm.oacc[otl][r][tok];
                for (int j2 = 0; j2 < nj; ++j2) {
                    const int u = u0 + j2;
                    const int pb = sm.ubeg[u], tu = sm.ubeg[u + 1] - pb;
                    for (int tt = 0; tt < tu; ++tt) {
                        const int f = sm.plist[pb + tt];
                        if (f / k != tok) continue;
                        float ys = 0.f;
                        for (int w = 0; w < nw; ++w) ys += rb[((j2 * wpe + w) * 16 + r) * tge + tt];
                        ys = (sm.uwi[u] >= 0) ? ys * sm.uts[u][2] * ldexpf(1.0f, sm.rexp[pb + tt]) : 0.0f;
                        acc += sm.wts[f] * ys;
                        if (a.y) a.y[(int64_t)(pb + tt) * H + ot * 16 + r] = ys;
                    }
                }
                sm.oacc[otl][r][tok] = acc;
            }
            buf ^= 1;
        } else {
            // one expert per slot; its tokens in groups of tge, restaged when they change
            const int u = u0;
            const int wi = sm.uwi[u];
            const int pb = sm.ubeg[u], tu = sm.ubeg[u + 1] - pb;
            const int ngroups = (tu + tge - 1) / tge;
            for (int gi = 0; gi < ngroups; ++gi) {
                const int g0 = gi * tge, nt = min(tge, tu - g0);
                if (staged_u != u || staged_g != gi) {
                    csync();
                    stage_rows(sm.xexp, &sm.flag, xs, hstride, a.hbuf, nt, I,
                               [&](int r) { return (int64_t)sm.plist[pb + g0 + r] * I; }, tid, dk::NCW * 32, csync);
                    staged_u = u;
                    staged_g = gi;
                }
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                if (wi >= 0) tile_partial(slot, KB2, warp, dk::NCW, xs + min(g8, nt - 1) * hstride, d);
                float* rb = red + buf * dk::NCW * 16 * tge;
                store_partial(rb, tge, warp, d, nt);
                consumer_sync();
                if (gi == ngroups - 1 && tid == 0) mbar_arrive(&sm.empty[s]);
                if (tid < 16 * nt) {
                    const int r = tid / nt, tt = tid - r * nt;
                    const int nw = min(dk::NCW, KB2);
                    float ys = 0.f;
                    for (int w = 0; w < nw; ++w) ys += rb[(w * 16 + r) * tge + tt];
                    const int f = sm.plist[pb + g0 + tt];
                    ys = (wi >= 0) ? ys * sm.uts[u][2] * ldexpf(1.0f, sm.xexp[tt]) : 0.0f;
                    sm.oacc[otl][r][f / k] += sm.wts[f] * ys;
                    if (a.y) a.y[(int64_t)(pb + g0 + tt) * H + ot * 16 + r] = ys;
                }
                buf ^= 1;
            }
        }
    }
    consumer_sync();
    if (a.out) {
        for (int i = tid; i < n_ot * 16 * T; i += dk::NCW * 32) {
            const int tok = i / (n_ot * 16), rr = i - tok * n_ot * 16;
            const int otl = rr / 16, r = rr % 16;
            a.out[(int64_t)tok * H + (sp.o_beg + otl) * 16 + r] = bf16_bits(sm.oacc[otl][r][tok]);
        }
    }
}

// ---------------------------------------------------------------------------- tile packing

// [N][K] row-major codes/scales -> 16-row tiles (layout in ft_nvfp4_pack_tiles).
__global__ void __launch_bounds__(256) k_pack_tiles(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                    const uint8_t* __restrict__ scales, int64_t scales_ld,
                                                    int64_t N, int64_t K, uint8_t* __restrict__ tiles) {
    const int64_t KB = K / 128;
    const int64_t tile_bytes = KB * 1152;
    const int64_t per_tile = KB * 64 + KB * 32;  // 16-byte code pieces + 4-byte scale words
    const int64_t total = (N / 16) * per_tile;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / per_tile;
        int64_t r = i % per_tile;
        uint8_t* dst = tiles + tile * tile_bytes;
        if (r < KB * 64) {  // code piece: (kb, h, q, g)
            const int64_t kb = r / 64;
            const int rem = (int)(r % 64);
            const int h = rem / 32, q = (rem / 8) & 3, g = rem & 7;
            const int64_t row = tile * 16 + 8 * h + g;
            const uint4 v = *reinterpret_cast<const uint4*>(codes + row * codes_ld + kb * 64 + 16 * q);
            *reinterpret_cast<uint4*>(dst + kb * 1024 + h * 512 + (q * 8 + g) * 16) = v;
        } else {  // scale word: (kb, q, g)
            r -= KB * 64;
            const int64_t kb = r / 32;
            const int rem = (int)(r % 32);
            const int q = rem / 8, g = rem & 7;
            const uint8_t* s0 = scales + (tile * 16 + g) * scales_ld + kb * 8 + 2 * q;
            const uint8_t* s1 = scales + (tile * 16 + 8 + g) * scales_ld + kb * 8 + 2 * q;
            const uint32_t w = (uint32_t)s0[0] | ((uint32_t)s0[1] << 8) | ((uint32_t)s1[0] << 16) | ((uint32_t)s1[1] << 24);
            *reinterpret_cast<uint32_t*>(dst + KB * 1024 + kb * 128 + (q * 8 + g) * 4) = w;
        }
    }
}

// ---------------------------------------------------------------------------- host side

static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct DecodeLaunch {
    int nstages, stage_bytes, xs_stride, xs_bytes, tge, fast;
    size_t smem;
};

// Shared memory: static part, ring of stages (one 16-row tile of the wider
// matrix each), staging area for f16 activation / h rows, partial tiles.
static bool plan_decode(int T, int k, int H, int I, DecodeLaunch& p) {
    const size_t budget = 227 * 1024;
    const size_t fixed = align_up(sizeof(DecodeSmem), 128);
    p.stage_bytes = (int)align_up((size_t)9 * std::max(H, I), 128);
    p.xs_stride = std::max(H, I) + 8;
    auto try_plan = [&](bool fast, int tge) {
        const size_t red = align_up((size_t)2 * dk::NCW * 16 * tge * sizeof(float), 128);
        const size_t xs = fast ? align_up((size_t)std::max(T * (H + 8), T * k * (I + 8)) * 2, 128)
                               : align_up((size_t)tge * p.xs_stride * 2, 128);
        if (fixed + xs + red + 2 * (size_t)p.stage_bytes > budget) return false;
        p.fast = fast ? 1 : 0;
        p.tge = tge;
        p.xs_bytes = (int)xs;
        p.nstages = (int)std::min<size_t>(dk::MAXNS, (budget - fixed - xs - red) / p.stage_bytes);
        p.smem = fixed + (size_t)p.nstages * p.stage_bytes + xs + red;
        return true;
    };
    // fast path: every x row and every h row staged at once (T <= 8, one mma pass per expert)
    if (T <= dk::TG && try_plan(true, T)) return true;
    for (int tge = std::min(T, dk::TG); tge >= 1; tge /= 2)
        if (try_plan(false, tge)) return true;
    return false;
}

static ft_status launch_decode(const DecodeArgs& args0, ft_stream_t stream, const char* fn) {
    DecodeLaunch p;
    const ft_moe_layer_weights& W = args0.W;
    if (!plan_decode(args0.T, args0.k, W.H, W.I, p))
        return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": layer too large for the decode kernel's shared memory");
    const int G = sm_count();
    if (W.H / 16 > dk::MAX_OUT_TILES * G)
        return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": H too large for one output tile range per SM");
    const size_t ring = (size_t)p.nstages * p.stage_bytes;
    if ((size_t)args0.T * W.E * 4 > ring || (size_t)(W.E + 1) * 4 > ring)
        return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": router logits do not fit the prologue scratch");
    DecodeArgs a = args0;
    a.nstages = p.nstages;
    a.stage_bytes = p.stage_bytes;
    a.xs_stride = p.xs_stride;
    a.xs_bytes = p.xs_bytes;
    a.tge = p.tge;
    a.fast = p.fast;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(k_moe_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    k_moe_decode<<<G, dk::THREADS, p.smem, cu(stream)>>>(a);
    return check_launch(fn);
}

ft_status validate_weights(const ft_moe_layer_weights* W, const char* fn);

// Workspace: [0, 256) grid-barrier counter (zero before first use), then h.
static size_t fused_workspace_size(int T, int k, int I) { return 256 + align_up((size_t)T * k * I * 2, 256); }

// grouped-mode launch used by ft_moe_expert_ffn_nvfp4_decode for tiled weights
ft_status decode_tiles_grouped(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k, const int32_t* offsets,
                               const int32_t* perm, const float* w, float* y, uint16_t* out, void* ws, size_t ws_bytes,
                               ft_stream_t stream) {
    const char* fn = "ft_moe_expert_ffn_nvfp4_decode";
    if (T > dk::MAXT || k > dk::MAXK)
        return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": tiled decode supports T <= 16 and k <= 32");
    if (!aligned(x, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": x needs 16-byte alignment");
    const size_t need = fused_workspace_size(T, k, W->I);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": workspace missing, too small or not 256-byte aligned");
    DecodeArgs a{};
    a.W = *W;
    a.offsets = offsets;
    a.perm = perm;
    a.w_in = w;
    a.x = x;
    a.out = out;
    a.y = y;
    a.bar = static_cast<unsigned int*>(ws);
    a.hbuf = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + 256);
    a.T = T;
    a.k = k;
    return launch_decode(a, stream, fn);
}

}  // namespace ft

using namespace ft;

extern "C" {

ft_status ft_nvfp4_pack_tiles(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                              int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream) {
    if (N <= 0 || K <= 0 || N % 16 || K % 128)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_tiles: need N a multiple of 16 and K a multiple of 128");
    if (!codes || !scales || !tiles) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_tiles: null pointer");
    if (!aligned(codes, 16) || codes_ld % 16 || !aligned(tiles, 16) || scales_ld < K / 16 || codes_ld < K / 2)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_tiles: codes/tiles need 16-byte alignment and row strides");
    const int64_t total = (N / 16) * (K / 128) * 96;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 64);
    k_pack_tiles<<<(unsigned)blocks, 256, 0, cu(stream)>>>(codes, codes_ld, scales, scales_ld, N, K, tiles);
    return check_launch("ft_nvfp4_pack_tiles");
}

size_t ft_moe_layer_decode_workspace_size(int T, int k, int H, int I) {
    (void)H;
    if (T <= 0 || k <= 0 || I <= 0) return 0;
    return fused_workspace_size(T, k, I);
}

ft_status ft_moe_layer_decode(const ft_moe_layer_weights* W, const float* logits, const uint16_t* x, int T, int k,
                              uint16_t* out, int32_t* ids, float* w, void* ws, size_t ws_bytes, ft_stream_t stream) {
    const char* fn = "ft_moe_layer_decode";
    ft_status st = validate_weights(W, fn);
    if (st != FT_OK) return st;
    if (W->layout != FT_LAYOUT_DECODE_TILES)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weights must use FT_LAYOUT_DECODE_TILES");
    if (T < 0 || T > dk::MAXT || k <= 0 || k > W->E || k > dk::MAXK)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 0 <= T <= 16 and 1 <= k <= min(E, 32)");
    if (T == 0) return FT_OK;
    if (!logits || !x || !out) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if ((ids == nullptr) != (w == nullptr))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": give both ids and w or neither");
    if (!aligned(x, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": x needs 16-byte alignment");
    const size_t need = fused_workspace_size(T, k, W->I);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": workspace missing, too small or not 256-byte aligned");
    DecodeArgs a{};
    a.W = *W;
    a.logits = logits;
    a.x = x;
    a.out = out;
    a.ids_out = ids;
    a.w_out = w;
    a.bar = static_cast<unsigned int*>(ws);
    a.hbuf = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + 256);
    a.T = T;
    a.k = k;
    return launch_decode(a, stream, fn);
}

}  // extern "C"
