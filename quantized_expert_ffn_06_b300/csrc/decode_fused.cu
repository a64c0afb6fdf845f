// decode_fused.cu -- one persistent launch per MoE layer for small token
// counts (decode): router top-k, expert grouping, NVFP4 gate/up projection with
// SwiGLU, down projection and routing-weighted combine.
//
// The step follows the page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算"
// (MoE core mechanism: linear + softmax router, top-K experts, weighted sum of
// independent expert FFNs).  Decode is bound by streaming the selected experts'
// weights from HBM, and at batch 1 a layer moves only ~14 MB (a few
// microseconds), so the kernel is built around the latency of that stream:
//
//  * Weights sit in HBM in 16-row tiles (ft_nvfp4_pack_tiles): per 128-element
//    K-block 1 KB of codes in which lane L of a warp owns the 16-byte pieces at
//    L*16 and 512 + L*16 (its mma A fragment for rows L/4 and L/4 + 8), then
//    128 B of E4M3 scales, one 4-byte word per lane.  One tile is one bulk copy
//    and every shared-memory read of it is conflict-free.
//  * Prologue: x and the router logits land in shared memory by one bulk copy
//    each.  Each token's top-k is found by one warp: every lane sorts its
//    (up to eight) keys once, then k rounds of a warp-wide integer max over the
//    lanes' heads (order-preserving keys, ties to the lower expert id).  All
//    threads stage the activations as f16, and up to 32 (token, slot) pairs are
//    grouped by expert inside one warp.  Every CTA does this redundantly, so
//    the weight stream starts without any inter-CTA traffic.
//  * One producer warp issues every tile the CTA needs with cp.async.bulk into
//    a ring of shared-memory stages guarded by mbarriers; the down-projection
//    tiles are prefetched while the gate/up tiles are consumed.  Its other
//    lanes fetch the experts' tensor scales into shared memory, and it
//    triggers the dependent launch, off the consumers' path.
//  * Sixteen consumer warps form four groups.  A group owns whole tiles: its
//    four warps split a tile's K-blocks, decode each E2M1 pair exactly to f16
//    (cvt.rn.f16x2.e2m1x2), multiply by the E4M3 block scale in f16 (exact: at
//    most 6 significant bits, magnitudes in [2^-10, 2688]) and feed mma.sync
//    m16n8k16 with fp32 accumulation (tokens are the mma's N).  The tensor cores
//    only take over the multiply-adds of this HBM-bound GEMV.  The group then
//    reduces its four partial tiles and writes h = bf16(silu(g) * u).
//  * The gate/up phase writes h as 64-bit words {bf16, bf16, call epoch}; the
//    down phase of every CTA waits (bounded) for exactly the words it reads, so
//    no grid-wide barrier separates the phases.
//    In the down phase each CTA owns a range of 16-row output tiles for all
//    selected experts; a warp computes one expert's down tile (for rows of 8+
//    K-blocks, one or two experts per chunk and their K-blocks split across
//    the group's warps), and the weighted sum over a token's k experts is
//    taken in slot order j from shared memory.
//  * The control code runs once per launch, so its size and latency are on the
//    critical path: divisions by launch-time constants are host-computed
//    multiply-high divisors, slow paths are out of line, one-shot loops stay
//    rolled.
//  * A batch whose f16 staging does not fit one launch runs as launches over
//    token chunks (ft_moe_layer_decode).
//  * Grid = one CTA per SM, all co-resident, which those waits rely on.  Every
//    wait is bounded by a %globaltimer budget; on expiry the kernel sets
//    FT_DEVERR_TIMEOUT, stops waiting and finishes without trapping.
//  * The launch allows programmatic dependent launch: the kernel waits for its
//    predecessor's results (griddepcontrol.wait) before reading any input, and
//    lets its successor be scheduled once all of its own CTAs have started.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace ft {

namespace dk {
constexpr int NCW = 16;                  // consumer warps
constexpr int NG = 4;                    // consumer groups
constexpr int WPG = NCW / NG;            // warps per group
constexpr int THREADS = 32 * (NCW + 1);  // + one producer warp
constexpr int MAXT = 16;                 // tokens per launch
constexpr int MAXK = 32;                 // experts per token
constexpr int MAXNS = 16;                // ring stages
constexpr int XPAD = 32;                 // halves of padding per staged f16 row (bank spread between rows)
constexpr size_t SMEM_BUDGET = 227 * 1024;
constexpr size_t XS_BUDGET = 120 * 1024;  // staged activations: x and h, separate buffers
constexpr unsigned long long WAIT_NS = 2000000000ull;  // bound on any single wait
}  // namespace dk

// Division by a divisor fixed at launch: q = x / d as one multiply-high with
// m = ceil(2^32 / d), exact whenever x * d < 2^32 (every use below stays far
// inside that).  Runtime integer division is a long instruction sequence, and
// this kernel's control code runs once per launch, so its size is its latency.
struct FastDiv {
    uint32_t d, m;  // m == 0 encodes d == 1
};

static FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.m = (d <= 1) ? 0u : (uint32_t)((0x100000000ull + d - 1) / d);
    return f;
}

__device__ __forceinline__ int fdiv(int x, const FastDiv& f) {
    return f.m ? (int)__umulhi((uint32_t)x, f.m) : x;
}

// Shared-memory plan, computed on the host (byte offsets into dynamic shared memory).
struct DecodePlan {
    int nstages, stage_bytes;  // ring
    int J;                     // down tiles (experts) per phase-2 stage
    int tcol;                  // token columns of a partial tile (T)
    int max_ot;                // phase-2 output tiles per CTA, at most
    int xs_stride, hs_stride;  // halves per staged x / h row
    int off_bars, off_ids, off_wts, off_plist, off_pexp, off_hexp, off_ulist, off_ubeg, off_uwi, off_misc;
    int off_xs, off_hs, off_red, off_ybuf, off_ring, off_ptok, off_ts;
    int smem;
    FastDiv dv_ns;    // ring stages
    FastDiv dv_tgu;   // gate/up tiles per expert (2I/16)
    FastDiv dv_k;     // slots per token
    FastDiv dv_xrow;  // 16-byte pieces per x row (H/8)
    FastDiv dv_hrow;  // h words per row (I/2)
    FastDiv dv_g;     // CTAs in the grid
    FastDiv dv_t;     // tokens
    FastDiv dv_j;     // down tiles per stage (J)
    int logits_bulk;  // the logits are copied into the ring by one bulk copy
    float inv_k;      // 1/k, rounded to nearest (the weight of every slot of a -inf row)
};

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
    void* hbuf;               // [T*k][I/2] h words {bf16, bf16, epoch}, by permuted row
    unsigned int* bar;        // call counter (monotonic, starts at 0): G per call
    int T, k;
    DecodePlan P;
};

// misc ints in shared memory
// (xexp: MAXT entries, tags: MAXNS; FLAG / HFLAG: x / h rows needed rescaling)
enum { M_U = 0, M_FLAG = 1, M_ABORT = 2, M_EPOCH = 3, M_XEXP = 4, M_TAGS = 4 + 16, M_TS = 4 + 16 + 16, M_HFLAG = M_TS + 1 };

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

// Gives up a bounded wait: the first expiry in a CTA sets FT_DEVERR_TIMEOUT and
// the CTA's abort flag; returns whether the wait may go on.
__device__ __forceinline__ bool wait_budget_left(unsigned long long t0, volatile int* abort_flag) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 > dk::WAIT_NS) {
        *abort_flag = 1;
        raise_dev_error(FT_DEVERR_TIMEOUT);
        return false;
    }
    return true;
}

// Bounded wait on an mbarrier phase (slow path, out of line).  On expiry, or
// if the CTA already gave up, returns false.
__device__ __noinline__ bool mbar_wait_slow(unsigned long long* b, uint32_t parity, volatile int* abort_flag) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(b, parity))
        if (!wait_budget_left(t0, abort_flag)) return false;
    return true;
}

__device__ __forceinline__ bool mbar_wait(unsigned long long* b, uint32_t parity, volatile int* abort_flag) {
    return mbar_try_wait(b, parity) || mbar_wait_slow(b, parity, abort_flag);
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(b))
                 : "memory");
}

// Stage tags: the producer publishes, after arming a stage's full barrier for
// chunk n, tag[stage] = n (release); a consumer of chunk n first waits for that
// tag (acquire) and only then tests the barrier's phase parity.  Without the tag
// a consumer group running ahead could test the parity of a use whose previous
// use has not landed yet, and parity alone cannot tell the two apart.
__device__ __forceinline__ void tag_publish(int* tag, int n) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tag)), "r"(n) : "memory");
}
__device__ __forceinline__ int tag_read(const int* tag) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(tag)) : "memory");
    return v;
}

// Bounded wait for chunk n (stage n mod NS, use n / NS): its tag, then its
// full-barrier phase.  Out of line: both consumer loops share one copy.
// Bounded wait (slow path, out of line) for a shared-memory tag to read `want`.
__device__ __noinline__ void tag_wait_slow(int* tag, int want, volatile int* abort_flag) {
    const unsigned long long t0 = globaltimer();
    while (tag_read(tag) != want)
        if (!wait_budget_left(t0, abort_flag)) return;
}

__device__ __forceinline__ void tag_wait(int* tag, int want, volatile int* abort_flag) {
    if (tag_read(tag) != want) tag_wait_slow(tag, want, abort_flag);
}

// Returns the stage; after an expired wait the CTA's abort flag is set and the
// stage's contents are not to be trusted (the caller finishes without waiting).
__device__ __noinline__ int chunk_wait(unsigned long long* full, int* tags, int n, FastDiv dv_ns, volatile int* abort_flag) {
    const int q = fdiv(n, dv_ns), s = n - q * (int)dv_ns.d;
    tag_wait(&tags[s], n, abort_flag);
    mbar_wait(&full[s], q & 1, abort_flag);
    return s;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(dk::NCW * 32) : "memory"); }
__device__ __forceinline__ void group_sync(int gi) {
    asm volatile("bar.sync %0, %1;" ::"r"(2 + gi), "n"(dk::WPG * 32) : "memory");
}

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

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return (i == 0) ? v.x : (i == 1) ? v.y : (i == 2) ? v.z : v.w;
}

// ---------------------------------------------------------------------------- staged activation rows

// Position (in halves) of element e of a row in the staged f16 layout: within
// each 128-element K-block, the 8-element piece i (0..3) of lane-quarter q
// (elements 32q + 8i .. +7) sits at piece (4i + q), so the four lanes of an mma
// row group read distinct banks for every i.
__device__ __forceinline__ int staged_pos(int e) {
    const int kb = e >> 7, w = e & 127;
    const int q = w >> 5, i = (w >> 3) & 3, r = w & 7;
    return (kb << 7) + (((i << 2) + q) << 3) + r;
}

// 2^e for the small exponents of the staging pre-scale (|e| < 126): exact.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& big) {
    const float lo = bf16_to_f32((uint16_t)(w & 0xFFFFu)), hi = bf16_to_f32((uint16_t)(w >> 16));
    big |= !(fabsf(lo) < 60000.0f) || !(fabsf(hi) < 60000.0f);
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Rare path of the staging: rows holding a value of magnitude >= 60000 are
// rescaled by a power of two so that they fit f16; exps[r] records it.  The
// caller synchronises before and after.  Source: bf16 rows (x), or h words.
__device__ __noinline__ void restage_scaled(int* exps, __half* dst, int stride, int n, int K, const uint16_t* xsrc,
                                            const unsigned long long* hw, int ti, int nthr, bool cta_wide) {
    auto val = [&](int r, int c) {
        if (xsrc) return bf16_to_f32(__ldcg(xsrc + (int64_t)r * K + c));
        const uint32_t w = (uint32_t)__ldcg(hw + (int64_t)r * (K / 2) + c / 2);
        return bf16_to_f32((uint16_t)((c & 1) ? (w >> 16) : (w & 0xFFFFu)));
    };
    const int w = ti >> 5, lane = ti & 31, nw = nthr >> 5;
#pragma unroll 1
    for (int r = w; r < n; r += nw) {
        float m = 0.0f;
#pragma unroll 1
        for (int i = lane; i < K; i += 32) m = fmaxf(m, fabsf(val(r, i)));
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) exps[r] = (m >= 16384.0f) ? ilogbf(m) - 14 : 0;
    }
    if (cta_wide) __syncthreads();
    else consumer_sync();
#pragma unroll 1
    for (int idx = ti; idx < n * K; idx += nthr) {
        const int r = idx / K, c = idx - r * K;
        dst[r * stride + staged_pos(c)] = __float2half_rn(val(r, c) * pow2i(-exps[r]));
    }
}

// Convert the n activation rows that landed as bf16 [n][K] in `raw` (shared
// memory, by one bulk copy) to f16 in dst (row stride `stride` halves,
// staged_pos order), with every thread of the CTA; `src` is the same rows in
// global memory, read again only on the rare rescaling path.
__device__ void stage_x(int* exps, volatile int* flag, __half* dst, int stride, const uint16_t* raw, const uint16_t* src,
                        int n, int K, FastDiv dv_row) {
    const int ti = threadIdx.x, nthr = blockDim.x;
    const int per_row = K >> 3, total = n * per_row;
    bool big = false;
#pragma unroll 1
    for (int idx = ti; idx < total; idx += nthr) {
        const int r = fdiv(idx, dv_row), c = idx - r * per_row;
        const uint4 v = *reinterpret_cast<const uint4*>(raw + (size_t)idx * 8);
        const uint4 o = make_uint4(bf16x2_to_f16x2(v.x, big), bf16x2_to_f16x2(v.y, big), bf16x2_to_f16x2(v.z, big),
                                   bf16x2_to_f16x2(v.w, big));
        *reinterpret_cast<uint4*>(dst + r * stride + staged_pos(c * 8)) = o;
    }
    if (big) *flag = 1;
    __syncthreads();
    if (*flag) {
        restage_scaled(exps, dst, stride, n, K, src, nullptr, ti, nthr, true);
        __syncthreads();
    }
}

// h words: the gate/up phase writes h as 64-bit words {bf16 h[2j], bf16 h[2j+1],
// uint32 epoch} (one single-copy-atomic store each), so the down phase can wait
// for exactly the words it reads instead of for a grid-wide barrier.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Stage all n h rows (I values each, nw = I/2 words per row) as f16 into dst,
// waiting (bounded) for each word to carry `epoch`; consumer threads only.
// Returns false if a wait gave up.
__device__ bool stage_h(int* exps, volatile int* flag, __half* dst, int stride, const unsigned long long* hw, int n, int I,
                        FastDiv dv_row, unsigned int epoch, volatile int* abort_flag) {
    const int ti = threadIdx.x, nthr = dk::NCW * 32;
    const int nw = I / 2, total = n * nw;
    constexpr int B = 8;  // 8-byte loads in flight per thread
    bool big = false, ok = true;
#pragma unroll 1
    for (int base = ti; base < total; base += B * nthr) {
        unsigned long long v[B];
        uint32_t pending = 0;
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int idx = base + u * nthr;
            if (idx < total) {
                v[u] = ld_relaxed_u64(hw + idx);
                if ((uint32_t)(v[u] >> 32) != epoch) pending |= 1u << u;
            }
        }
        if (pending) {
            const unsigned long long t0 = globaltimer();
            while (pending) {
#pragma unroll
                for (int u = 0; u < B; ++u)
                    if (pending & (1u << u)) {
                        v[u] = ld_relaxed_u64(hw + base + u * nthr);
                        if ((uint32_t)(v[u] >> 32) == epoch) pending &= ~(1u << u);
                    }
                if (pending && !wait_budget_left(t0, abort_flag)) {
                    ok = false;
                    break;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int idx = base + u * nthr;
            if (idx < total) {
                const int r = fdiv(idx, dv_row), c = idx - r * nw;
                *reinterpret_cast<uint32_t*>(dst + r * stride + staged_pos(2 * c)) = bf16x2_to_f16x2((uint32_t)v[u], big);
            }
        }
        if (!ok) break;
    }
    if (big) *flag = 1;
    consumer_sync();
    if (*flag) {
        restage_scaled(exps, dst, stride, n, I, nullptr, hw, ti, nthr, false);
        consumer_sync();
    }
    return ok;
}

// ---------------------------------------------------------------------------- tile math

// Partial products of one 16-row tile over K-blocks kb0, kb0+kstep, ... (K =
// 128*KB) against one staged f16 row per lane column (`xrow`, staged_pos
// order): the mma accumulator (rows g, g+8; token columns 2q, 2q+1) as
// {d0, d1, d2, d3}.  Out of line: one copy serves both phases.
//
// Lane L = 4g + q owns code bytes [16q, 16q+16) of rows g and g+8 in each
// K-block, i.e. elements 32q .. 32q+31.  mma s (of 8 per K-block) takes
// elements 32q + 4s .. +3 of them: the pair 4s, 4s+1 as the fragment's
// k = 2q, 2q+1 and the pair 4s+2, 4s+3 as k = 2q+8, 2q+9.  The activations are
// read at the same element positions, so the dot product is unchanged by this
// K order.  Two accumulators shorten the dependent mma chain.
__device__ __noinline__ float4 tile_partial(const uint8_t* tile, int KB, int kb0, int kstep, const __half* xrow) {
    const int lane = threadIdx.x & 31;
    const int q = lane & 3;
    const uint8_t* scl = tile + KB * 1024;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kb = kb0; kb < KB; kb += kstep) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(tile + kb * 1024 + lane * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(tile + kb * 1024 + 512 + lane * 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(scl + kb * 128 + lane * 4);
        const uint32_t sg0 = e4m3_to_f16x2_bcast(sc & 0xFFu), sg1 = e4m3_to_f16x2_bcast((sc >> 8) & 0xFFu);
        const uint32_t sh0 = e4m3_to_f16x2_bcast((sc >> 16) & 0xFFu), sh1 = e4m3_to_f16x2_bcast(sc >> 24);
        const __half* xr = xrow + kb * 128 + q * 8;
        uint4 xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = *reinterpret_cast<const uint4*>(xr + 32 * i);
        const uint32_t cw0[4] = {c0.x, c0.y, c0.z, c0.w};
        const uint32_t cw1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t sa = (s < 4) ? sg0 : sg1, sb = (s < 4) ? sh0 : sh1;
            const uint32_t w0 = cw0[s >> 1], w1 = cw1[s >> 1];
            const int sh = (s & 1) * 16;
            const uint32_t a0 = hmul2(e2m1x2_to_f16x2((w0 >> sh) & 0xFFu), sa);
            const uint32_t a2 = hmul2(e2m1x2_to_f16x2((w0 >> (sh + 8)) & 0xFFu), sa);
            const uint32_t a1 = hmul2(e2m1x2_to_f16x2((w1 >> sh) & 0xFFu), sb);
            const uint32_t a3 = hmul2(e2m1x2_to_f16x2((w1 >> (sh + 8)) & 0xFFu), sb);
            const uint32_t b0 = word_of(xv[s >> 1], (2 * s) & 3);
            const uint32_t b1 = word_of(xv[s >> 1], (2 * s + 1) & 3);
            if (s & 1)
                mma16816(e, a0, a1, a2, a3, b0, b1);
            else
                mma16816(d, a0, a1, a2, a3, b0, b1);
        }
    }
    return make_float4(d[0] + e[0], d[1] + e[1], d[2] + e[2], d[3] + e[3]);
}

// ---------------------------------------------------------------------------- routing

// 256 < E <= 1024: a lane rescans its (up to 32) logits, skipping the slots in
// `taken`.  Returns {expert of lane j < k, bad}.
__device__ __noinline__ uint2 select_topk_wide(const float* row, int E, int k) {
    const int lane = threadIdx.x & 31;
    const int EPL = (E + 31) >> 5;
    const int n = max(0, min(EPL, E - lane * EPL));
    const float* mine = row + lane * EPL;
    uint32_t taken = 0, bad = 0;
    int my_e = 0;
    uint32_t bk = 0;
    int bi = 0;
    bool dirty = true;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        if (dirty) {
            bk = 0;
#pragma unroll 1
            for (int i0 = 0; i0 < n; i0 += 4) {
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) x[u] = (i0 + u < n) ? mine[i0 + u] : 0.0f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u;
                    bad |= (i < n) && ((x[u] != x[u]) || (x[u] == INFINITY));
                    const uint32_t key = (i < n && !((taken >> i) & 1u)) ? logit_key(x[u]) : 0u;
                    if (key > bk) {
                        bk = key;
                        bi = i;
                    }
                }
            }
            dirty = false;
        }
        const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
        const int wl = __ffs(__ballot_sync(0xffffffffu, bk == gk)) - 1;
        const int we = __shfl_sync(0xffffffffu, lane * EPL + bi, wl);
        if (lane == wl) {
            taken |= 1u << bi;
            dirty = true;
        }
        if (lane == j) my_e = we;
    }
    return make_uint2((uint32_t)my_e, bad);
}

// Router of one token by one warp: top-k selection, then the weights
// exp(l_j - l_0) / sum over the k selected, with the same butterfly sum as
// ft_moe_route (every weight inv_k = 1/k when the largest logit is -inf).
__device__ __forceinline__ void route_token(const float* row, int E, int k, float inv_k, int& my_e, float& my_w, bool& bad) {
    const int lane = threadIdx.x & 31;
    bool b = false;
    if (E <= 256) {
        my_e = select_topk8(row, E, k, b);
    } else {
        const uint2 r = select_topk_wide(row, E, k);
        my_e = (int)r.x;
        b = r.y != 0u;
    }
    bad = __any_sync(0xffffffffu, b);
    const float my_v = (lane < k) ? row[my_e] : -INFINITY;
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    if (m == -INFINITY || m != m) {
        my_w = inv_k;
    } else {
        const float ej = (lane < k) ? expf(my_v - m) : 0.0f;
        const float s = warp_sum(ej);
        my_w = ej / s;
    }
}

// ---------------------------------------------------------------------------- kernel

__global__ void __launch_bounds__(dk::THREADS, 1) k_moe_decode(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t dsm[];
    const DecodePlan& P = a.P;
    unsigned long long* full = reinterpret_cast<unsigned long long*>(dsm + P.off_bars);
    unsigned long long* empty = full + dk::MAXNS;
    unsigned long long* xbar = full + 2 * dk::MAXNS;  // the bulk copy of x
    int* s_ids = reinterpret_cast<int*>(dsm + P.off_ids);      // [nf] expert of slot f (route mode)
    float* s_wts = reinterpret_cast<float*>(dsm + P.off_wts);  // [nf] weight of slot f
    int* s_plist = reinterpret_cast<int*>(dsm + P.off_plist);  // [nf] slot f of permuted row p
    int* s_ptok = reinterpret_cast<int*>(dsm + P.off_ptok);    // [nf] token of permuted row p
    int* s_pexp = reinterpret_cast<int*>(dsm + P.off_pexp);    // [nf] expert of permuted row p
    int* s_hexp = reinterpret_cast<int*>(dsm + P.off_hexp);    // [nf] pre-scale of staged h row p
    int* s_ulist = reinterpret_cast<int*>(dsm + P.off_ulist);  // [nf] selected experts, ascending
    int* s_ubeg = reinterpret_cast<int*>(dsm + P.off_ubeg);    // [nf+1] permuted-row range of each
    int* s_uwi = reinterpret_cast<int*>(dsm + P.off_uwi);      // [nf] weight index (-1: invalid slot)
    float* s_ts = reinterpret_cast<float*>(dsm + P.off_ts);   // [nf][4] tensor scales (gate, up, down) of each
    int* misc = reinterpret_cast<int*>(dsm + P.off_misc);
    volatile int* abort_flag = misc + M_ABORT;
    __half* xs = reinterpret_cast<__half*>(dsm + P.off_xs);  // x rows (phase 1)
    __half* hs = reinterpret_cast<__half*>(dsm + P.off_hs);  // h rows (phase 2); separate, so no CTA-wide sync between
    float* red = reinterpret_cast<float*>(dsm + P.off_red);
    float* ybuf = reinterpret_cast<float*>(dsm + P.off_ybuf);  // [max_ot][nf][16]
    uint8_t* ring = dsm + P.off_ring;

    const ft_moe_layer_weights& W = a.W;
    const int H = W.H, I = W.I, E = W.E, T = a.T, k = a.k;
    const int nf = T * k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int NS = P.nstages;

    if (tid == 0) {
#pragma unroll 1
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], dk::WPG);
        }
        mbar_init(xbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        misc[M_FLAG] = 0;
        misc[M_HFLAG] = 0;
        misc[M_ABORT] = 0;
        misc[M_TS] = 0;
    }
    if (tid < dk::MAXT) misc[M_XEXP + tid] = 0;
    if (tid < dk::MAXNS) misc[M_TAGS + tid] = -1;
#pragma unroll 1
    for (int i = tid; i < nf; i += dk::THREADS) s_hexp[i] = 0;
    __syncthreads();
    // inputs (and the workspace) may be written by the preceding kernel in the stream
    griddep_wait();
    // x lands as bf16 in the h staging area (unused until the down phase) by one bulk copy.
    // This call's epoch: calls sharing a workspace each add G to its counter.  The producer
    // lane takes it (off the router's path) and publishes it at the end of the prologue.
    // The logits, where the plan allows, land the same way in the ring (unused until the weights
    // stream); the router then reads them through a generic pointer either way.
    const bool route_mode = a.logits != nullptr;
    const uint16_t* xraw = reinterpret_cast<const uint16_t*>(hs);
    const float* lsrc = P.logits_bulk ? reinterpret_cast<const float*>(ring) : a.logits;
    unsigned int old_count = 0;
    if (tid == dk::NCW * 32) {
        const uint32_t xbytes = (uint32_t)(T * H * 2), lbytes = route_mode && P.logits_bulk ? (uint32_t)(T * E * 4) : 0u;
        mbar_arrive_expect_tx(xbar, xbytes + lbytes);
        bulk_g2s(hs, a.x, xbytes, xbar);
        if (lbytes) bulk_g2s(ring, a.logits, lbytes, xbar);
        old_count = atomicAdd(a.bar, 1u);
    }

    // ---------------- prologue: warps < T route their token once the inputs have landed, then all
    // threads stage x
    mbar_wait(xbar, 0, abort_flag);
    if (route_mode && warp < T) {
        int my_e = 0;
        float my_w = 0.0f;
        bool bad = false;
        route_token(lsrc + warp * E, E, k, P.inv_k, my_e, my_w, bad);
        if (bad && lane == 0) raise_dev_error(FT_DEVERR_NAN_LOGIT);
        if (lane < k) {
            s_ids[warp * k + lane] = my_e;
            s_wts[warp * k + lane] = my_w;
            if (c == 0 && a.ids_out) {
                a.ids_out[warp * k + lane] = my_e;
                a.w_out[warp * k + lane] = my_w;
            }
        }
    }
    // the ring is next written by the async proxy (the weight stream): order the reads before it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    stage_x(misc + M_XEXP, misc + M_FLAG, xs, P.xs_stride, xraw, a.x, T, H, P.dv_xrow);  // ends with __syncthreads
    // grouping: permuted row of slot f = #{f2 : e2 < e} + #{f2 < f : e2 == e}.  Up to 32 slots
    // one warp does it with shuffles and goes straight on to the scan below.
    const bool warp_grouping = route_mode && nf <= 32;
    if (warp_grouping) {
        if (warp == 0) {
            const int f = lane;
            const int e = (f < nf) ? s_ids[f] : 0x7fffffff;
            int pos = 0;
#pragma unroll 4
            for (int f2 = 0; f2 < nf; ++f2) {
                const int e2 = __shfl_sync(0xffffffffu, e, f2);
                pos += (e2 < e) || (e2 == e && f2 < f);
            }
            if (f < nf) {
                s_plist[pos] = f;
                s_ptok[pos] = fdiv(f, P.dv_k);
                s_pexp[pos] = e;
            }
            __syncwarp();
        }
    } else if (route_mode) {
#pragma unroll 1
        for (int f = tid; f < nf; f += dk::THREADS) {
            const int e = s_ids[f];
            int pos = 0;
#pragma unroll 1
            for (int f2 = 0; f2 < nf; ++f2) {
                const int e2 = s_ids[f2];
                pos += (e2 < e) || (e2 == e && f2 < f);
            }
            s_plist[pos] = f;
            s_ptok[pos] = fdiv(f, P.dv_k);
            s_pexp[pos] = e;
        }
    } else {
#pragma unroll 1
        for (int p = tid; p < nf; p += dk::THREADS) {
            int pf = a.perm[p];
            if (pf < 0 || pf >= nf) {
                raise_dev_error(FT_DEVERR_BAD_INDEX);
                pf = 0;
            }
            s_plist[p] = pf;
            s_ptok[p] = fdiv(pf, P.dv_k);
            s_wts[p] = a.w_in ? a.w_in[p] : 0.0f;  // indexed by slot f: w_in is [T][k]
            // expert owning row p: last e with offsets[e] <= p
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(a.offsets + mid) <= p) lo = mid;
                else hi = mid - 1;
            }
            if (__ldg(a.offsets + lo) > p || __ldg(a.offsets + lo + 1) <= p || __ldg(a.offsets + E) != nf)
                raise_dev_error(FT_DEVERR_BAD_INDEX);
            s_pexp[p] = lo;
        }
    }
    if (!warp_grouping) __syncthreads();
    // selected experts = segment starts of pexp (warp 0, ballot scan)
    if (warp == 0) {
        int run = 0;
#pragma unroll 1
        for (int p0 = 0; p0 < nf; p0 += 32) {
            const int p = p0 + lane;
            const bool start = p < nf && (p == 0 || s_pexp[p] != s_pexp[p - 1]);
            const uint32_t b = __ballot_sync(0xffffffffu, start);
            if (start) {
                const int u = run + __popc(b & ((1u << lane) - 1u));
                s_ulist[u] = s_pexp[p];
                s_ubeg[u] = p;
                s_uwi[u] = weight_index(W, s_pexp[p]);
            }
            run += __popc(b);
        }
        if (lane == 0) {
            misc[M_U] = run;
            s_ubeg[run] = nf;
        }
    }
    if (tid == dk::NCW * 32) misc[M_EPOCH] = (int)(old_count / (unsigned)G + 1u);
    __syncthreads();
    const int U = misc[M_U];
    const unsigned int epoch = (unsigned int)misc[M_EPOCH];

    // ---------------- work split
    const int tiles_gu = I >> 3;  // 16-row tiles of an expert's [2I][H] gate/up matrix
    const int KB1 = H >> 7, KB2 = I >> 7;
    const int bytes1 = 9 * H, bytes2 = 9 * I;  // one 16-row tile of [.][H] or [.][I]
    const int n1 = U * tiles_gu;                // <= 512 * 2048
    const int p1_beg = (int)((unsigned)(n1 * c) / (unsigned)G), p1_end = (int)((unsigned)(n1 * (c + 1)) / (unsigned)G);
    const int n2 = H >> 4;
    const int o_beg = fdiv(n2 * c, P.dv_g), o_end = fdiv(n2 * (c + 1), P.dv_g);
    const int J = P.J;
    const int n_p1 = p1_end - p1_beg;
    const int n_ot = o_end - o_beg;
    const int n_jg = fdiv(U + J - 1, P.dv_j);  // expert groups per output tile
    const int n_chunks = n_p1 + n_ot * n_jg;

    if (warp == dk::NCW) {
        // ---------------- producer: stream tiles into the ring
        if (lane == 0) {
            int n = 0, s = 0, use = 0;  // chunk, its stage and the stage's use
            int u = 0, lt = 0;          // gate/up chunk: expert and tile within it
            if (n_p1 > 0) {
                u = fdiv(p1_beg, P.dv_tgu);
                lt = p1_beg - u * tiles_gu;
            }
            int otl = 0, jg = 0;  // down chunk: output tile and expert group
#pragma unroll 1
            for (; n < n_chunks; ++n) {
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag)) break;
                uint8_t* dst = ring + (size_t)s * P.stage_bytes;
                if (n < n_p1) {
                    const int wi = s_uwi[u];
                    if (wi < 0) {
                        mbar_arrive(&full[s]);
                    } else {
                        mbar_arrive_expect_tx(&full[s], (uint32_t)bytes1);
                        bulk_g2s(dst, W.gu_codes + (int64_t)wi * W.gu_codes_stride + (int64_t)lt * bytes1,
                                 (uint32_t)bytes1, &full[s]);
                    }
                    if (++lt == tiles_gu) {
                        lt = 0;
                        ++u;
                    }
                } else {
                    const int ot = o_beg + otl;
                    const int u0 = jg * J, nj = min(J, U - u0);
                    uint32_t tx = 0;
#pragma unroll 1
                    for (int jj = 0; jj < nj; ++jj) tx += (s_uwi[u0 + jj] >= 0) ? (uint32_t)bytes2 : 0u;
                    mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll 1
                    for (int jj = 0; jj < nj; ++jj) {
                        const int wi = s_uwi[u0 + jj];
                        if (wi >= 0)
                            bulk_g2s(dst + jj * bytes2, W.d_codes + (int64_t)wi * W.d_codes_stride + (int64_t)ot * bytes2,
                                     (uint32_t)bytes2, &full[s]);
                    }
                    if (++jg == n_jg) {
                        jg = 0;
                        ++otl;
                    }
                }
                tag_publish(&misc[M_TAGS + s], n);
                if (++s == NS) {
                    s = 0;
                    ++use;
                }
            }
            // Once every CTA of this grid has started (the call counter reaches epoch * G), the
            // next kernel in the stream may be scheduled: it cannot take an SM one of ours still
            // needs, and it waits for our completion itself before reading anything.
            {
                const unsigned long long t0 = globaltimer();
                unsigned int v;
                do {
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.bar) : "memory");
                } while ((int)(v - epoch * (unsigned)G) < 0 && globaltimer() - t0 < 100000ull);
                if ((int)(v - epoch * (unsigned)G) >= 0) griddep_launch_dependents();
            }
            // the CTA must not exit with copies still landing in its shared memory: wait
            // (bounded, even after an abort) for the last use of every stage issued
            const unsigned long long t0 = globaltimer();
            int q = max(0, n - NS);
            const int uq = fdiv(q, P.dv_ns);
            int sq = q - uq * NS, pq = uq & 1;
#pragma unroll 1
            for (; q < n; ++q) {
                while (!mbar_try_wait(&full[sq], pq) && globaltimer() - t0 < dk::WAIT_NS) {
                }
                if (++sq == NS) {
                    sq = 0;
                    pq ^= 1;
                }
            }
        } else {
            // lanes 1..31: the tensor scales (gate, up, down) of the selected experts into shared
            // memory, published once all are there
#pragma unroll 1
            for (int u = lane - 1; u < U; u += 31) {
                const int wi = s_uwi[u];
                const float* ts = W.tscale + (int64_t)(wi >= 0 ? wi : 0) * W.tscale_stride;
                const float t0 = ts[0], t1 = ts[1], t2 = ts[2];
                s_ts[4 * u + 0] = (wi >= 0) ? t0 : 0.0f;
                s_ts[4 * u + 1] = (wi >= 0) ? t1 : 0.0f;
                s_ts[4 * u + 2] = (wi >= 0) ? t2 : 0.0f;
            }
            __syncwarp(0xfffffffeu);
            if (lane == 1) tag_publish(&misc[M_TS], 1);
        }
        return;
    }

    // ---------------- consumers (warps 0 .. NCW-1), phase 1: gate/up tiles -> h words
    const int gi = warp / dk::WPG, wig = warp % dk::WPG, gtid = tid % (dk::WPG * 32);
    const int g8 = lane >> 2, q4 = lane & 3;
    const int TC = P.tcol;
    const int hw_row = I / 2;  // h words per permuted row
    unsigned long long* hw = reinterpret_cast<unsigned long long*>(a.hbuf);
    float* gred = red + gi * 2 * dk::WPG * 16 * TC;  // this group's two partial buffers [WPG][16][TC]
    int buf = 0;
#pragma unroll 1
    for (int n = gi; n < n_p1; n += dk::NG) {
        const int t = p1_beg + n;
        const int u = fdiv(t, P.dv_tgu), lt = t - u * tiles_gu;
        const int wi = s_uwi[u];
        const int pb = s_ubeg[u], tu = s_ubeg[u + 1] - pb;
        const int s = chunk_wait(full, misc + M_TAGS, n, P.dv_ns, abort_flag);
        const uint8_t* tile = ring + (size_t)s * P.stage_bytes;
        float* rb = gred + buf * dk::WPG * 16 * TC;
#pragma unroll 1
        for (int c0 = 0; c0 < tu; c0 += 8) {
            const int nt = min(8, tu - c0);
            const int col = min(g8, nt - 1);
            const int xr = s_ptok[pb + c0 + col];  // token of this lane's column
            float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (wi >= 0) dv = tile_partial(tile, KB1, wig, dk::WPG, xs + xr * P.xs_stride);
            const float d[4] = {dv.x, dv.y, dv.z, dv.w};
            float* r = rb + wig * 16 * TC;
            if (2 * q4 < nt) {
                r[g8 * TC + c0 + 2 * q4] = d[0];
                r[(g8 + 8) * TC + c0 + 2 * q4] = d[2];
            }
            if (2 * q4 + 1 < nt) {
                r[g8 * TC + c0 + 2 * q4 + 1] = d[1];
                r[(g8 + 8) * TC + c0 + 2 * q4 + 1] = d[3];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        group_sync(gi);
        // h = silu(g) * u for the tile's 8 (gate, up) row pairs: word j holds pairs 2j, 2j+1
        tag_wait(&misc[M_TS], 1, abort_flag);
        const float tsg = s_ts[4 * u + 0], tsu = s_ts[4 * u + 1];
#pragma unroll 1
        for (int idx = gtid; idx < 4 * tu; idx += dk::WPG * 32) {
            const int j = idx & 3, tt = idx >> 2;
            float hv[2] = {0.0f, 0.0f};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int p = 2 * j + h2;
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int w = 0; w < dk::WPG; ++w) {
                    gs += rb[(w * 16 + 2 * p) * TC + tt];
                    us += rb[(w * 16 + 2 * p + 1) * TC + tt];
                }
                if (wi >= 0) {
                    const float sc = pow2i(misc[M_XEXP + s_ptok[pb + tt]]);
                    hv[h2] = silu_f32(gs * tsg * sc) * (us * tsu * sc);
                }
            }
            const unsigned long long word = (unsigned long long)bf16_bits(hv[0]) |
                                            ((unsigned long long)bf16_bits(hv[1]) << 16) | ((unsigned long long)epoch << 32);
            st_relaxed_u64(hw + (int64_t)(pb + tt) * hw_row + lt * 4 + j, word);
        }
        buf ^= 1;
    }

    // ---------------- phase 2: down projection over this CTA's output rows
    if (n_ot > 0)  // all h rows (permuted order), as each becomes available
        stage_h(s_hexp, misc + M_HFLAG, hs, P.hs_stride, hw, nf, I, P.dv_hrow, epoch, abort_flag);
    tag_wait(&misc[M_TS], 1, abort_flag);
    {
        // chunks n_p1 .. n_chunks-1, round robin over the groups continuing phase 1's order;
        // chunk n_p1 + m is (output tile m / n_jg, expert group m mod n_jg)
        int n = n_p1 + ((gi - n_p1) % dk::NG + dk::NG) % dk::NG;
        int otl = 0, jg = n - n_p1;
        while (n_jg > 0 && jg >= n_jg) {
            jg -= n_jg;
            ++otl;
        }
#pragma unroll 1
        for (; n < n_chunks; n += dk::NG) {
            const int ot = o_beg + otl;
            const int u0 = jg * J, nj = min(J, U - u0);
            // warps per expert tile: with one or two experts in the chunk the group's four warps
            // split each tile's K-blocks, and their partials are summed through shared memory
            const int wpe = (nj == 1) ? dk::WPG : (nj == 2) ? dk::WPG / 2 : (nj <= 4 && dk::WPG >= 8) ? dk::WPG / 4 : 1;
            const int s = chunk_wait(full, misc + M_TAGS, n, P.dv_ns, abort_flag);
            const uint8_t* slot = ring + (size_t)s * P.stage_bytes;
            float* rb = gred + buf * dk::WPG * 16 * TC;
#pragma unroll 1
            for (int jj = wig / wpe; jj < nj; jj += dk::WPG / wpe) {
                const int u = u0 + jj;
                const int wi = s_uwi[u];
                const int pb = s_ubeg[u], tu = s_ubeg[u + 1] - pb;
                const float tsd = s_ts[4 * u + 2];
#pragma unroll 1
                for (int c0 = 0; c0 < tu; c0 += 8) {
                    const int nt = min(8, tu - c0);
                    const int col = min(g8, nt - 1);
                    float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (wi >= 0)
                        dv = tile_partial(slot + jj * bytes2, KB2, wig & (wpe - 1), wpe, hs + (pb + c0 + col) * P.hs_stride);
                    const float d[4] = {dv.x, dv.y, dv.z, dv.w};
                    if (wpe > 1) {  // this warp's share of the K-blocks, summed below
                        float* r = rb + wig * 16 * TC;
                        if (2 * q4 < nt) {
                            r[g8 * TC + c0 + 2 * q4] = d[0];
                            r[(g8 + 8) * TC + c0 + 2 * q4] = d[2];
                        }
                        if (2 * q4 + 1 < nt) {
                            r[g8 * TC + c0 + 2 * q4 + 1] = d[1];
                            r[(g8 + 8) * TC + c0 + 2 * q4 + 1] = d[3];
                        }
                        continue;
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int cc = c0 + 2 * q4 + h2;  // column of d[h2] (row g8) and d[2 + h2] (row g8 + 8)
                        if (2 * q4 + h2 < nt) {
                            const int p = pb + cc;
                            const float sc = (wi >= 0) ? tsd * pow2i(s_hexp[p]) : 0.0f;
                            const int f = s_plist[p];
                            const float y0 = d[h2] * sc, y1 = d[2 + h2] * sc;
                            ybuf[(otl * nf + f) * 16 + g8] = y0;
                            ybuf[(otl * nf + f) * 16 + g8 + 8] = y1;
                            if (a.y) {
                                a.y[(int64_t)p * H + ot * 16 + g8] = y0;
                                a.y[(int64_t)p * H + ot * 16 + g8 + 8] = y1;
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (wpe > 1) {
                group_sync(gi);
                // item idx of expert e2: row idx & 15, column idx >> 4
#pragma unroll 1
                for (int e2 = 0; e2 < nj; ++e2) {
                    const int u = u0 + e2;
                    const int wi = s_uwi[u];
                    const int pb = s_ubeg[u], tu = s_ubeg[u + 1] - pb;
                    const float tsd = s_ts[4 * u + 2];
#pragma unroll 1
                    for (int idx = gtid; idx < 16 * tu; idx += dk::WPG * 32) {
                        const int r = idx & 15, tt = idx >> 4;
                        float ys = 0.0f;
#pragma unroll 1
                        for (int w = 0; w < wpe; ++w) ys += rb[((e2 * wpe + w) * 16 + r) * TC + tt];
                        const int p = pb + tt;
                        ys = (wi >= 0) ? ys * (tsd * pow2i(s_hexp[p])) : 0.0f;
                        ybuf[(otl * nf + s_plist[p]) * 16 + r] = ys;
                        if (a.y) a.y[(int64_t)p * H + ot * 16 + r] = ys;
                    }
                }
                buf ^= 1;
            }
            jg += dk::NG;
            while (jg >= n_jg) {
                jg -= n_jg;
                ++otl;
            }
        }
    }
    consumer_sync();
    // combine: out[t][row] = bf16(sum_j w[t][j] * y[t*k + j][row]) in slot order j;
    // item i = (otl * T + tok) * 16 + row
    if (a.out) {
#pragma unroll 1
        for (int i = tid; i < n_ot * 16 * T; i += dk::NCW * 32) {
            const int q = i >> 4, r = i & 15;
            const int otl = fdiv(q, P.dv_t), tok = q - otl * T;
            float acc = 0.0f;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const int f = tok * k + j;
                acc += s_wts[f] * ybuf[(otl * nf + f) * 16 + r];
            }
            a.out[(int64_t)tok * H + (o_beg + otl) * 16 + r] = bf16_bits(acc);
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
        if (r < KB * 64) {  // code piece (kb, h, g, q): bytes 16q..16q+15 of row 8h+g's 64 bytes in block kb
            const int64_t kb = r / 64;
            const int rem = (int)(r % 64);
            const int h = rem / 32, g = (rem / 4) & 7, q = rem & 3;
            const int64_t row = tile * 16 + 8 * h + g;
            const uint4 v = *reinterpret_cast<const uint4*>(codes + row * codes_ld + kb * 64 + 16 * q);
            *reinterpret_cast<uint4*>(dst + kb * 1024 + h * 512 + (g * 4 + q) * 16) = v;
        } else {  // scale word (kb, g, q): blocks 2q, 2q+1 of rows g and g+8
            r -= KB * 64;
            const int64_t kb = r / 32;
            const int rem = (int)(r % 32);
            const int g = rem / 4, q = rem & 3;
            const uint8_t* s0 = scales + (tile * 16 + g) * scales_ld + kb * 8 + 2 * q;
            const uint8_t* s1 = scales + (tile * 16 + 8 + g) * scales_ld + kb * 8 + 2 * q;
            const uint32_t w = (uint32_t)s0[0] | ((uint32_t)s0[1] << 8) | ((uint32_t)s1[0] << 16) | ((uint32_t)s1[1] << 24);
            *reinterpret_cast<uint32_t*>(dst + KB * 1024 + kb * 128 + (g * 4 + q) * 4) = w;
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

// Shared memory: barriers and routing tables, staged activations (x in phase
// 1, h in phase 2, same area), the groups' partial tiles, the per-slot down
// outputs, and the ring (one 16-row tile of the wider matrix per stage).
static bool plan_decode(int T, int k, int H, int I, int G, DecodePlan& p, std::string& why) {
    const int nf = T * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 128);
        return (int)o;
    };
    p.off_bars = take((2 * dk::MAXNS + 1) * 8);
    p.off_ids = take((size_t)nf * 4);
    p.off_wts = take((size_t)nf * 4);
    p.off_plist = take((size_t)nf * 4);
    p.off_ptok = take((size_t)nf * 4);
    p.off_pexp = take((size_t)nf * 4);
    p.off_hexp = take((size_t)nf * 4);
    p.off_ulist = take((size_t)nf * 4);
    p.off_ubeg = take((size_t)(nf + 1) * 4);
    p.off_uwi = take((size_t)nf * 4);
    p.off_misc = take((4 + dk::MAXT + dk::MAXNS + 2) * 4);
    p.off_ts = take((size_t)nf * 16);
    p.xs_stride = H + dk::XPAD;
    p.hs_stride = I + dk::XPAD;
    // the h staging area first receives x as bf16 [T][H] (the prologue's bulk copy)
    const size_t xs = (size_t)T * p.xs_stride * 2, hs = std::max((size_t)nf * p.hs_stride * 2, (size_t)T * H * 2);
    if (xs + hs > dk::XS_BUDGET) {
        why = "activations of " + std::to_string(T) + " tokens and their " + std::to_string(nf) +
              " expert rows do not fit the fused kernel's staging area";
        return false;
    }
    p.off_xs = take(xs);
    p.off_hs = take(hs);
    p.tcol = T;
    p.off_red = take((size_t)dk::NG * 2 * dk::WPG * 16 * T * 4);
    const int n2 = H / 16;
    p.max_ot = (n2 + G - 1) / G;
    p.off_ybuf = take((size_t)p.max_ot * nf * 16 * 4);
    p.stage_bytes = (int)align_up((size_t)9 * std::max(H, I), 128);
    p.off_ring = (int)off;
    if (off + 2 * (size_t)p.stage_bytes > dk::SMEM_BUDGET) {
        why = "layer too large for the fused kernel's shared memory";
        return false;
    }
    p.nstages = (int)std::min<size_t>(dk::MAXNS, (dk::SMEM_BUDGET - off) / p.stage_bytes);
    p.smem = (int)(off + (size_t)p.nstages * p.stage_bytes);
    // down tiles per stage: as many as a stage holds; for long down rows (8+ K-blocks) few enough
    // that every group gets a chunk per output tile and splits its tiles' K-blocks
    p.J = std::max(1, std::min(p.stage_bytes / (9 * I), 16));
    if (I / 128 >= 8) p.J = std::max(1, std::min(p.J, (nf + dk::NG - 1) / dk::NG));
    p.dv_ns = make_fastdiv((uint32_t)p.nstages);
    p.dv_tgu = make_fastdiv((uint32_t)(I / 8));
    p.dv_k = make_fastdiv((uint32_t)k);
    p.dv_xrow = make_fastdiv((uint32_t)(H / 8));
    p.dv_hrow = make_fastdiv((uint32_t)(I / 2));
    p.dv_g = make_fastdiv((uint32_t)G);
    p.dv_t = make_fastdiv((uint32_t)T);
    p.dv_j = make_fastdiv((uint32_t)p.J);
    p.inv_k = 1.0f / (float)k;
    return true;
}

static ft_status launch_decode(const DecodeArgs& args0, ft_stream_t stream, const char* fn) {
    const ft_moe_layer_weights& W = args0.W;
    const int G = sm_count();
    DecodeArgs a = args0;
    std::string why;
    if (!plan_decode(a.T, a.k, W.H, W.I, G, a.P, why)) return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": " + why);
    // the router's logits come in by one bulk copy when their address and size allow it
    const size_t lbytes = (size_t)a.T * W.E * 4;
    a.P.logits_bulk = a.logits && aligned(a.logits, 16) && lbytes % 16 == 0 &&
                      lbytes <= (size_t)a.P.nstages * a.P.stage_bytes;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(k_moe_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dk::SMEM_BUDGET);
    });
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(dk::THREADS);
    cfg.dynamicSmemBytes = a.P.smem;
    cfg.stream = cu(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_moe_decode, a);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
    return check_launch(fn);
}

ft_status validate_weights(const ft_moe_layer_weights* W, const char* fn);

// Workspace: [0, 256) call counter (zero before first use), then the h words
// (8 bytes per two h values).
static size_t fused_workspace_size(int T, int k, int I) { return 256 + align_up((size_t)T * k * I * 4, 256); }

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
    if (out && !w) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": out needs w");
    DecodeArgs a{};
    a.W = *W;
    a.offsets = offsets;
    a.perm = perm;
    a.w_in = w;
    a.x = x;
    a.out = out;
    a.y = y;
    a.bar = static_cast<unsigned int*>(ws);
    a.hbuf = static_cast<char*>(ws) + 256;
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

}  // extern "C"

// ---------------------------------------------------------------------------- variant without allocation

namespace ft {

// Scratch of ft_moe_layer_decode_noalloc: the call counter and the h words of
// one call, in a file-scope device array (every device that loads the library
// holds it until the process exits).  In host code the name is only a stand-in:
// the device address comes from cudaGetSymbolAddress, resolved once per device.
constexpr size_t kNoAllocScratchBytes = FT_NOALLOC_DECODE_MAX_SCRATCH;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (resolved on the first call there).
static ft_status noalloc_scratch(void** out, const char* fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": device ordinal beyond 63");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(FT_ERR_CUDA, std::string(fn) + ": cudaGetSymbolAddress failed: " + cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FT_OK;
}

}  // namespace ft

extern "C" {

ft_status ft_moe_layer_decode_noalloc(const ft_moe_layer_weights* W, const float* logits, const uint16_t* x, int T,
                                      int k, uint16_t* out, int32_t* ids, float* w, ft_stream_t stream) {
    const char* fn = "ft_moe_layer_decode_noalloc";
    ft_status st = validate_weights(W, fn);
    if (st != FT_OK) return st;
    if (T < 0 || T > dk::MAXT || k <= 0 || k > W->E || k > dk::MAXK)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 0 <= T <= 16 and 1 <= k <= min(E, 32)");
    if (T == 0) return FT_OK;
    const size_t need = fused_workspace_size(T, k, W->I);
    if (need > kNoAllocScratchBytes)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": T*k*I = " + std::to_string((size_t)T * k * W->I) +
                                            " needs " + std::to_string(need) + " bytes of scratch; the built-in scratch holds " +
                                            std::to_string(kNoAllocScratchBytes) + " (T*k*I <= 262144)");
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch, fn);
    if (st != FT_OK) return st;
    // every call starts from a zeroed counter and zeroed h words, whatever earlier calls left there
    const cudaError_t e = cudaMemsetAsync(scratch, 0, need, cu(stream));
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, std::string(fn) + ": clearing the scratch: " + cudaGetErrorString(e));
    return ft_moe_layer_decode(W, logits, x, T, k, out, ids, w, scratch, need, stream);
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
    // Tokens are independent in this step (each one's output depends only on its own routing),
    // so a batch whose activations do not fit the shared-memory staging runs as consecutive
    // launches over the largest token chunks that do, in order on the stream.
    int Tc = T;
    {
        DecodePlan probe;
        std::string why;
        while (Tc > 0 && !plan_decode(Tc, k, W->H, W->I, sm_count(), probe, why)) --Tc;
        if (Tc == 0) return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": " + why);
    }
    for (int t0 = 0; t0 < T; t0 += Tc) {
        DecodeArgs a{};
        a.W = *W;
        a.logits = logits + (int64_t)t0 * W->E;
        a.x = x + (int64_t)t0 * W->H;
        a.out = out + (int64_t)t0 * W->H;
        a.ids_out = ids ? ids + (int64_t)t0 * k : nullptr;
        a.w_out = w ? w + (int64_t)t0 * k : nullptr;
        a.bar = static_cast<unsigned int*>(ws);
        a.hbuf = static_cast<char*>(ws) + 256;
        a.T = std::min(Tc, T - t0);
        a.k = k;
        st = launch_decode(a, stream, fn);
        if (st != FT_OK) return st;
    }
    return FT_OK;
}

}  // extern "C"
