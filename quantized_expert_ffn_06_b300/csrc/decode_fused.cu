// decode_fused.cu -- one launch per MoE layer for small token counts (decode):
// router top-k, grouping by expert, NVFP4 gate/up projection with SwiGLU, down
// projection and the routing-weighted combine.
//
// The step follows the page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算"
// (MoE core mechanism: linear + softmax router, top-K experts, weighted sum of
// independent expert FFNs).  At batch 1 a layer of the 35B-class shape moves
// ~14 MB of expert weights, a few microseconds of HBM time, so the kernel is a
// chain of latencies around that stream, and two costs dominate that chain
// besides the stream itself: round trips to memory and instruction fetch (the
// control code runs once per launch, so every instruction on the path is
// fetched cold).  The kernel is built for both:
//
//  * Code size.  Control loops stay rolled, divisions by per-launch constants
//    are host-computed multiply-high divisors, and one out-of-line routine
//    computes a K-block for both projections.
//  * Inputs.  Right after the dependency wait one thread issues one bulk copy of
//    x and one of the router logits on an mbarrier.
//  * Router (every CTA, redundantly: no inter-CTA traffic before the weight
//    stream).  One token of at most 256 logits: warp 0 keeps each lane's eight
//    keys sorted and takes each rank with two warp reductions (the largest key,
//    then the lowest expert holding it) while the other warps stage x, and the
//    work split, a function of k alone, is made before the inputs arrive.
//    Several tokens: each warp ranks a block of 32 logits by 32 shuffles and
//    keeps its k best as sorted candidates, then eight lanes per candidate count
//    the candidates that beat it.  Keys order the fp32 logits exactly, equal
//    logits going to the lower expert id.
//  * Work split.  Phase 1 is the gate/up tiles of the selected experts, phase 2
//    the down projection of 16-row output tiles over all selected experts.  A
//    CTA's phase-1 share is balanced by bytes against its phase-2 share.
//  * Weight stream.  Each warp copies its own K-blocks (1152 bytes each) from
//    HBM into a shared-memory ring of R slots with per-lane async copies
//    (cp.async, one commit group per K-block), so R K-blocks per warp are in
//    flight; a lane reads back only the bytes it copied itself.  The ring runs
//    straight on from the gate/up K-blocks into the down K-blocks, which thus
//    land while the gate/up results are handed over.
//  * Inner loop.  A code word is split into its four bytes in one move, each
//    byte (two E2M1 codes) converts exactly to f16x2 (cvt.rn.f16x2.e2m1x2) and
//    is multiplied by its E4M3 block scale in f16 (exact: at most 6 significant
//    bits, magnitudes in [2^-10, 2688]); mma.sync m16n8k16 accumulates in fp32
//    with tokens as N.  Warps that share a tile sum their partials in shared
//    memory in a fixed order.
//  * Hand-off.  h = bf16(silu(g) * u) goes to global memory as 64-bit words
//    {bf16, bf16, call epoch}; phase 2 of every CTA waits (bounded) for exactly
//    the words it reads, so no grid-wide barrier separates the phases.
//  * Combine.  A token's k expert outputs are summed in slot order j in fp32
//    from shared memory and rounded once to bf16.
//  * MXFP4 weights run through the same kernel with 1088-byte K-blocks (UE8M0
//    scales: a per-row reference exponent, the residual in f16, 2^r on the fp32
//    partial).
//  * Grid = one CTA per SM (its shared memory admits one), all co-resident,
//    which the hand-off relies on: while another kernel holds SMs, resident CTAs
//    wait for the h of CTAs not yet started.  Every wait is bounded by a
//    %globaltimer budget; on expiry the kernel sets FT_DEVERR_TIMEOUT and
//    finishes without trapping.  The launch allows programmatic dependent
//    launch (griddepcontrol).
#include "common.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace ft {

namespace dk {
constexpr int NW = 16;                 // warps per CTA
constexpr int LOG_NW = 4;
constexpr int THREADS = 32 * NW;
constexpr int MAXT = 16;               // tokens per launch
constexpr int MAXK = 32;               // experts per token
constexpr int ITEM = 1152;             // bytes of one K-block (128 elements) of a 16-row tile: NVFP4 (MXFP4: 1088)
constexpr int ITEM8 = 2112;            // MXFP8: 2048 code bytes + 64 scale bytes
constexpr int XPAD = 32;               // halves of padding per staged f16 row
constexpr int MINSLOT = 2 * NW;        // partial-sum slots of a phase split across warps: at least,
constexpr int MAXSLOT = 4 * NW;        // and at most (one- and two-token launches)
constexpr size_t SMEM_BUDGET = 227 * 1024;
constexpr unsigned long long WAIT_NS = 2000000000ull;  // default bound on any single wait
}  // namespace dk

// Test hooks (off by default): a shorter wait bound, and a wait made to expire.
static std::atomic<unsigned long long> g_wait_ns{dk::WAIT_NS};
static std::atomic<int> g_wait_site{FT_WAIT_SITE_NONE};
unsigned long long wait_hook_ns() { return g_wait_ns.load(); }
int wait_hook_site() { return g_wait_site.load(); }

// Division by a divisor fixed per launch: q = x / d as one multiply-high with
// m = ceil(2^32 / d), exact whenever x * d < 2^32 (every use below stays far
// inside that).
struct FastDiv {
    uint32_t d, m;  // m == 0 encodes d == 1
};

static FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.m = (d <= 1) ? 0u : (uint32_t)((0x100000000ull + d - 1) / d);
    return f;
}

__device__ __forceinline__ int fdiv(int x, const FastDiv& f) { return f.m ? (int)__umulhi((uint32_t)x, f.m) : x; }

// Shared-memory plan and per-launch constants, computed on the host.
struct DecodePlan {
    int ring;                  // K-block slots per warp (R)
    int xs_stride, hs_stride;  // halves per staged x / h row
    int tc;                    // token columns of a partial tile (T)
    int nb, kk;                // router: 32-logit blocks per token, candidates per block (min(k, 32))
    int max_ot;                // output tiles per CTA, at most
    int off_misc, off_ids, off_wts, off_plist, off_ptok, off_pexp, off_hexp, off_ulist, off_ubeg, off_uwi, off_ts;
    int off_rank, off_xs, off_big, off_xraw, off_cand, off_slot, off_wscr, off_ybuf, off_ring;
    int smem;
    FastDiv dv_k;     // slots per token
    FastDiv dv_xrow;  // 16-byte pieces per x row (H/8)
    FastDiv dv_hrow;  // h words per row (I/2)
    FastDiv dv_g;     // CTAs in the grid
    FastDiv dv_t;     // tokens
    FastDiv dv_nb;    // router blocks per token
    FastDiv dv_c;     // router candidates per token (nb * kk)
    FastDiv dv_tgu;   // gate/up tiles per expert (I/8)
    FastDiv dv_kb1;   // K-blocks per gate/up tile (H/128)
    FastDiv dv_kb2;   // K-blocks per down tile (I/128)
    unsigned long long dv_g64;  // ceil(2^64 / G): call number = mulhi(counter, dv_g64)
    float inv_k;      // 1/k, rounded to nearest (the weight of every slot of a -inf row)
    unsigned long long wait_ns;  // bound on any single wait
    int wait_site;               // FT_WAIT_SITE_DECODE_H: the h hand-off waits for an epoch nobody writes
    int logits_bulk;             // the logits come in by one bulk copy (16-byte aligned, size a multiple of 16)
    int solo;                    // one routed token of at most 256 logits: one warp routes it, and the work split
                                 // (U = k distinct experts) is made before the inputs arrive
    int mx;                      // 0 NVFP4; 1 MXFP4 (1088-byte K-blocks), 2 MXFP8 (2112-byte K-blocks): no tensor scale
    int item;                    // bytes of a ring slot (one K-block of the format, rounded up to ITEM)
    int nslot;                   // partial-tile slots (a phase of n runs is split over the warps if n + NW <= nslot)
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
    unsigned long long* bar;  // call counter (monotonic, starts at 0): one per CTA per call
    int T, k;
    DecodePlan P;
};

// misc ints in shared memory (XEXP: pre-scale exponent of each staged x row)
enum { M_U = 0, M_FLAG = 1, M_HFLAG = 2, M_ABORT = 3, M_EPOCH = 4, M_XEXP = 8, M_BAR = 8 + dk::MAXT, M_COUNT = M_BAR + 2 };

// ---------------------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// per-thread async copies global -> shared (cp.async): 16 bytes (L2 only) or 4 bytes
__device__ __forceinline__ void cp16(void* s, const void* g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp4(void* s, const void* g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// the same copies to a shared-memory address given as such
__device__ __forceinline__ void cp16s(uint32_t s, const void* g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(g) : "memory");
}
__device__ __forceinline__ void cp4s(uint32_t s, const void* g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(g) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// wait until at most n of this thread's commit groups are pending (n clamped to [0, 15])
__device__ __forceinline__ void cp_wait_upto(int n) {
    switch (n <= 0 ? 0 : n >= 15 ? 15 : n) {
        case 0: cp_wait<0>(); break;
        case 1: cp_wait<1>(); break;
        case 2: cp_wait<2>(); break;
        case 3: cp_wait<3>(); break;
        case 4: cp_wait<4>(); break;
        case 5: cp_wait<5>(); break;
        case 6: cp_wait<6>(); break;
        case 7: cp_wait<7>(); break;
        case 8: cp_wait<8>(); break;
        case 9: cp_wait<9>(); break;
        case 10: cp_wait<10>(); break;
        case 11: cp_wait<11>(); break;
        case 12: cp_wait<12>(); break;
        case 13: cp_wait<13>(); break;
        case 14: cp_wait<14>(); break;
        default: cp_wait<15>(); break;
    }
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The four bytes of a code word (eight E2M1 codes) as four f16x2 (exact).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&f)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
        : "r"(w));
}

// A lane's four E4M3 block scales (one word) as f16x2, each value in both halves (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2_bcast(uint32_t sc, uint32_t& s0, uint32_t& s1, uint32_t& s2,
                                                      uint32_t& s3) {
    const uint32_t lo = __byte_perm(sc, 0u, 0x1100), hi = __byte_perm(sc, 0u, 0x3322);
    asm("{\n\t.reg .b16 a, b, c, d;\n\tmov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 %2, c;\n\tcvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
        : "=r"(s0), "=r"(s1), "=r"(s2), "=r"(s3)
        : "r"(lo), "r"(hi));
}

// Four E4M3 bytes (one word, byte 0 first) as two f16x2: bytes 0, 1 and bytes 2, 3 (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
// caller synchronises the CTA before and after.  Source: bf16 rows (x), or h words.
__device__ __noinline__ void restage_scaled(int* exps, __half* dst, int stride, int n, int K, const uint16_t* xsrc,
                                            const unsigned long long* hw) {
    auto val = [&](int r, int c) {
        if (xsrc) return bf16_to_f32(__ldcg(xsrc + (int64_t)r * K + c));
        const uint32_t w = (uint32_t)__ldcg(hw + (int64_t)r * (K / 2) + c / 2);
        return bf16_to_f32((uint16_t)((c & 1) ? (w >> 16) : (w & 0xFFFFu)));
    };
    const int ti = threadIdx.x, w = ti >> 5, lane = ti & 31;
#pragma unroll 1
    for (int r = w; r < n; r += dk::NW) {
        float m = 0.0f;
#pragma unroll 1
        for (int i = lane; i < K; i += 32) m = fmaxf(m, fabsf(val(r, i)));
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) exps[r] = (m >= 16384.0f) ? ilogbf(m) - 14 : 0;
    }
    __syncthreads();
#pragma unroll 1
    for (int idx = ti; idx < n * K; idx += dk::THREADS) {
        const int r = idx / K, c = idx - r * K;
        dst[r * stride + staged_pos(c)] = __float2half_rn(val(r, c) * pow2i(-exps[r]));
    }
}

// ---------------------------------------------------------------------------- one K-block of a 16-row tile

// Partial products of one K-block (128 elements x 16 rows) held in shared
// memory as laid out in HBM: lane L = 4g + q owns the code bytes [16q, 16q+16)
// of rows g and g+8 (at L*16 and 512 + L*16) and the scale word of blocks 2q,
// 2q+1 of both rows (at 1024 + L*4), i.e. elements 32q .. 32q+31.  x: the
// lane's staged f16 row (its token column) at this K-block, + 8q halves.  mma s
// (8 per K-block) takes elements 32q + 4s .. +3: the pair 4s, 4s+1 as the
// fragment's k = 2q, 2q+1 and the pair 4s+2, 4s+3 as k = 2q+8, 2q+9; the
// activations are read at the same element positions, so the dot product is
// unchanged by this K order.  Returns the accumulator (rows g, g+8; columns
// 2q, 2q+1) as {d0, d1, d2, d3}.  Out of line: one copy serves both phases.
__device__ __noinline__ float4 kblock_partial(const uint8_t* item, const __half* x) {
    const int lane = threadIdx.x & 31;
    uint32_t sg0, sg1, sh0, sh1;
    e4m3x4_to_f16x2_bcast(*reinterpret_cast<const uint32_t*>(item + 1024 + lane * 4), sg0, sg1, sh0, sh1);
    // the lane's 16 code bytes of each row in one 16-byte load each, the loop fully unrolled
    const uint4 w0 = *reinterpret_cast<const uint4*>(item + lane * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(item + 512 + lane * 16);
    const uint32_t c0[4] = {w0.x, w0.y, w0.z, w0.w}, c1[4] = {w1.x, w1.y, w1.z, w1.w};
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t f0[4], f1[4];
        e2m1x8_to_f16x2x4(c0[s2], f0);
        e2m1x8_to_f16x2x4(c1[s2], f1);
        const uint32_t sa = (s2 < 2) ? sg0 : sg1, sb = (s2 < 2) ? sh0 : sh1;
        const uint4 xv = *reinterpret_cast<const uint4*>(x + 32 * s2);
        mma16816(d, hmul2(f0[0], sa), hmul2(f1[0], sb), hmul2(f0[1], sa), hmul2(f1[1], sb), xv.x, xv.y);
        mma16816(e, hmul2(f0[2], sa), hmul2(f1[2], sb), hmul2(f0[3], sa), hmul2(f1[3], sb), xv.z, xv.w);
    }
    return make_float4(d[0] + e[0], d[1] + e[1], d[2] + e[2], d[3] + e[3]);
}

// 2^d (d <= 0) as f16 in both halves: exact down to 2^-24 (subnormals), 0 below.
__device__ __forceinline__ uint32_t pow2_f16x2(int d) {
    const uint32_t b = (d >= -14) ? (uint32_t)(d + 15) << 10 : (d >= -24) ? 1u << (d + 24) : 0u;
    return b | (b << 16);
}
// The power of two a UE8M0 byte stands for, 2^(s - 127), as an fp32 (s = 0: the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t s) {
    return s ? __uint_as_float(s << 23) : __uint_as_float(1u << 22);
}

// The MXFP4 form of kblock_partial: item = 1024 code bytes as above, then the
// UE8M0 scale bytes of rows g and g+8 for lane L = 4g + q at 1024 + 2L (lane
// L's 32 elements of a row are exactly one MX block).  Row g's reference
// exponent r is the largest of its four blocks (lanes 4g .. 4g+3); the codes
// are scaled by 2^(x - r) in f16 (exact unless x - r < -22), the fp32 partial
// by 2^(r - 127).
__device__ __noinline__ float4 kblock_partial_mx(const uint8_t* item, const __half* x) {
    const int lane = threadIdx.x & 31;
    const uint32_t sp = *reinterpret_cast<const uint16_t*>(item + 1024 + lane * 2);
    const uint32_t own = (sp & 0xFFu) | ((sp >> 8) << 16);  // {row g, row g+8} as 16-bit halves
    uint32_t ref = __vmaxu2(own, __shfl_xor_sync(0xffffffffu, own, 1));
    ref = __vmaxu2(ref, __shfl_xor_sync(0xffffffffu, ref, 2));
    const int rg = (int)(ref & 0xFFFFu), rh = (int)(ref >> 16);
    const uint32_t sa = pow2_f16x2((int)(own & 0xFFFFu) - rg), sb = pow2_f16x2((int)(own >> 16) - rh);
    const uint4 w0 = *reinterpret_cast<const uint4*>(item + lane * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(item + 512 + lane * 16);
    const uint32_t c0[4] = {w0.x, w0.y, w0.z, w0.w}, c1[4] = {w1.x, w1.y, w1.z, w1.w};
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t f0[4], f1[4];
        e2m1x8_to_f16x2x4(c0[s2], f0);
        e2m1x8_to_f16x2x4(c1[s2], f1);
        const uint4 xv = *reinterpret_cast<const uint4*>(x + 32 * s2);
        mma16816(d, hmul2(f0[0], sa), hmul2(f1[0], sb), hmul2(f0[1], sa), hmul2(f1[1], sb), xv.x, xv.y);
        mma16816(e, hmul2(f0[2], sa), hmul2(f1[2], sb), hmul2(f0[3], sa), hmul2(f1[3], sb), xv.z, xv.w);
    }
    const float fg = ue8m0_to_f32((uint32_t)rg), fh = ue8m0_to_f32((uint32_t)rh);
    return make_float4((d[0] + e[0]) * fg, (d[1] + e[1]) * fg, (d[2] + e[2]) * fh, (d[3] + e[3]) * fh);
}

// The MXFP8 form: item = 2048 code bytes (one E4M3 byte per element; lane L =
// 4g + q owns the 32 bytes of row g at L*32 and of row g+8 at 1024 + L*32, i.e.
// elements 32q .. 32q+31, exactly one MX block of each row), then the UE8M0
// pairs at 2048 + 2L.  E4M3 converts exactly to f16; the scales are applied as
// for MXFP4 (exact unless a block is more than 2^15 below the largest of its
// row's K-block).
__device__ __noinline__ float4 kblock_partial_mx8(const uint8_t* item, const __half* x) {
    const int lane = threadIdx.x & 31;
    const uint32_t sp = *reinterpret_cast<const uint16_t*>(item + 2048 + lane * 2);
    const uint32_t own = (sp & 0xFFu) | ((sp >> 8) << 16);
    uint32_t ref = __vmaxu2(own, __shfl_xor_sync(0xffffffffu, own, 1));
    ref = __vmaxu2(ref, __shfl_xor_sync(0xffffffffu, ref, 2));
    const int rg = (int)(ref & 0xFFFFu), rh = (int)(ref >> 16);
    const uint32_t sa = pow2_f16x2((int)(own & 0xFFFFu) - rg), sb = pow2_f16x2((int)(own >> 16) - rh);
    const uint4 g0 = *reinterpret_cast<const uint4*>(item + lane * 32);
    const uint4 g1 = *reinterpret_cast<const uint4*>(item + lane * 32 + 16);
    const uint4 h0 = *reinterpret_cast<const uint4*>(item + 1024 + lane * 32);
    const uint4 h1 = *reinterpret_cast<const uint4*>(item + 1024 + lane * 32 + 16);
    const uint32_t c0[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t c1[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
        uint32_t f0[4], f1[4];
        e4m3x4_to_f16x2x2(c0[2 * s2], f0[0], f0[1]);
        e4m3x4_to_f16x2x2(c0[2 * s2 + 1], f0[2], f0[3]);
        e4m3x4_to_f16x2x2(c1[2 * s2], f1[0], f1[1]);
        e4m3x4_to_f16x2x2(c1[2 * s2 + 1], f1[2], f1[3]);
        const uint4 xv = *reinterpret_cast<const uint4*>(x + 32 * s2);
        mma16816(d, hmul2(f0[0], sa), hmul2(f1[0], sb), hmul2(f0[1], sa), hmul2(f1[1], sb), xv.x, xv.y);
        mma16816(e, hmul2(f0[2], sa), hmul2(f1[2], sb), hmul2(f0[3], sa), hmul2(f1[3], sb), xv.z, xv.w);
    }
    const float fg = ue8m0_to_f32((uint32_t)rg), fh = ue8m0_to_f32((uint32_t)rh);
    return make_float4((d[0] + e[0]) * fg, (d[1] + e[1]) * fg, (d[2] + e[2]) * fh, (d[3] + e[3]) * fh);
}

// ---------------------------------------------------------------------------- kernel

// FMT: 0 NVFP4, 1 MXFP4, 2 MXFP8 (a template parameter: each format's kernel carries only its own code)
template <int R, int FMT>
__global__ void __launch_bounds__(dk::THREADS, 1) k_moe_decode(const DecodeArgs a) {
    constexpr int ITEMB = FMT == 2 ? dk::ITEM8 : dk::ITEM;  // bytes of a ring slot
    extern __shared__ __align__(128) uint8_t dsm[];
    const DecodePlan& P = a.P;
    int* misc = reinterpret_cast<int*>(dsm + P.off_misc);
    volatile int* abort_flag = misc + M_ABORT;
    int* s_ids = reinterpret_cast<int*>(dsm + P.off_ids);      // [nf] expert of slot f (route mode)
    float* s_wts = reinterpret_cast<float*>(dsm + P.off_wts);  // [nf] weight of slot f
    int* s_plist = reinterpret_cast<int*>(dsm + P.off_plist);  // [nf] slot f of permuted row p
    int* s_ptok = reinterpret_cast<int*>(dsm + P.off_ptok);    // [nf] token of permuted row p
    int* s_pexp = reinterpret_cast<int*>(dsm + P.off_pexp);    // [nf] expert of permuted row p
    int* s_hexp = reinterpret_cast<int*>(dsm + P.off_hexp);    // [nf] pre-scale of staged h row p
    int* s_ulist = reinterpret_cast<int*>(dsm + P.off_ulist);  // [nf] selected experts, ascending
    int* s_ubeg = reinterpret_cast<int*>(dsm + P.off_ubeg);    // [nf+1] permuted-row range of each
    int* s_uwi = reinterpret_cast<int*>(dsm + P.off_uwi);      // [nf] weight index (-1: invalid slot)
    float* s_ts = reinterpret_cast<float*>(dsm + P.off_ts);    // [nf][4] tensor scales (gate, up, down)
    int* s_rank = reinterpret_cast<int*>(dsm + P.off_rank);    // [T][nb*kk] router candidate ranks
    __half* xs = reinterpret_cast<__half*>(dsm + P.off_xs);    // x rows, f16, staged layout
    float* lg = reinterpret_cast<float*>(dsm + P.off_big);     // raw logits [T][E] (router), then ...
    __half* hs = reinterpret_cast<__half*>(dsm + P.off_big);   // ... h rows, f16, staged layout (phase 2)
    uint16_t* xraw = reinterpret_cast<uint16_t*>(dsm + P.off_xraw);                       // x as loaded, bf16
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(dsm + P.off_cand);  // [T][nb][kk]
    float* slots = reinterpret_cast<float*>(dsm + P.off_slot);  // [nslot][16][tc] partial tiles
    float* wscr = reinterpret_cast<float*>(dsm + P.off_wscr);   // [NW][16][tc] a warp's finished tile
    float* ybuf = reinterpret_cast<float*>(dsm + P.off_ybuf);   // [max_ot][nf][16] expert outputs

    const ft_moe_layer_weights& W = a.W;
    const int H = W.H, I = W.I, E = W.E, T = a.T, k = a.k;
    const int nf = T * k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int TC = P.tc;
    const bool route_mode = a.logits != nullptr;
    uint8_t* ring = dsm + P.off_ring + warp * (R * ITEMB);

    // ---------------- work split over U selected experts: CTA c takes phase-1 tiles [p1_beg, p1_end) and
    // output tiles [o_beg, o_end); its warps split the K-blocks of each phase.  With one routed token U = k
    // is known before the inputs arrive, and the split is made there.
    const int tiles_gu = I >> 3;  // 16-row tiles of an expert's [2I][H] gate/up matrix
    const int KB1 = H >> 7, KB2 = I >> 7;
    const int n2 = H >> 4;
    const int o_beg = fdiv(n2 * c, P.dv_g), o_end = fdiv(n2 * (c + 1), P.dv_g);
    const int n_ot = o_end - o_beg;
    int U = 0, n1 = 0, p1_beg = 0, p1_end = 0, n_t1 = 0, nr2 = 0, ni1 = 0, ni2 = 0;
    int ib1 = 0, ie1 = 0, ib2 = 0, ie2 = 0, cnt1 = 0, cnt = 0;
    bool split1 = false, split2 = false;
    float inv_u = 1.0f;
    // r / U for 0 <= r < 2^20: float estimate, corrected by one step
    auto div_u = [&](int r) {
        int q = (int)((float)r * inv_u);
        const int rem = r - q * U;
        q += (rem >= U) - (rem < 0);
        return q;
    };
    auto work_split = [&](int u_count) {
        U = u_count;
        n1 = U * tiles_gu;
        inv_u = __fdividef(1.0f, (float)max(U, 1));
        // phase-1 share balanced by bytes against the phase-2 share: CTA c's boundary is
        // proportional to c * tgt - (bytes of the down tiles of CTAs < c), in units of 9 bytes.
        // Float rounding can move a boundary by a tile; both neighbours compute a boundary from
        // the same expression, so the tiles still partition (at worst a tile is done twice).
        const float b1 = (float)H, b2 = (float)I * (float)U;
        float tgt = __fdividef((float)n1 * b1 + (float)n2 * b2, (float)G);
        tgt = fmaxf(tgt, (float)P.max_ot * b2);
        const float scale = __fdividef((float)n1, (float)G * tgt - (float)n2 * b2);
        p1_beg = c == 0 ? 0 : min(n1, __float2int_rn(((float)c * tgt - (float)o_beg * b2) * scale));
        p1_end = c == G - 1 ? n1 : min(n1, __float2int_rn(((float)(c + 1) * tgt - (float)o_end * b2) * scale));
        p1_end = max(p1_end, p1_beg);
        n_t1 = p1_end - p1_beg;
        nr2 = n_ot * U;  // phase-2 runs (output tile, expert), run r = otl * U + u
        // this warp's K-block ranges: split evenly (runs shared by neighbouring warps; run r of warp w
        // sums into slot r + w), or whole runs per warp when the slots cannot hold a split
        split1 = n_t1 + dk::NW <= P.nslot;
        split2 = nr2 + dk::NW <= P.nslot;
        ni1 = n_t1 * KB1;
        ni2 = nr2 * KB2;
        if (split1) {
            ib1 = (warp * ni1) >> dk::LOG_NW;
            ie1 = ((warp + 1) * ni1) >> dk::LOG_NW;
        } else {
            ib1 = ((warp * n_t1) >> dk::LOG_NW) * KB1;
            ie1 = (((warp + 1) * n_t1) >> dk::LOG_NW) * KB1;
        }
        if (split2) {
            ib2 = (warp * ni2) >> dk::LOG_NW;
            ie2 = ((warp + 1) * ni2) >> dk::LOG_NW;
        } else {
            ib2 = ((warp * nr2) >> dk::LOG_NW) * KB2;
            ie2 = (((warp + 1) * nr2) >> dk::LOG_NW) * KB2;
        }
        cnt1 = ie1 - ib1;
        cnt = cnt1 + (ie2 - ib2);  // this warp's K-blocks, phase 1 then 2
    };
    if (P.solo) work_split(k);

    unsigned long long* ibar = reinterpret_cast<unsigned long long*>(misc + M_BAR);  // the inputs' bulk copies
    if (tid < M_BAR) misc[tid] = 0;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(ibar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
#pragma unroll 1
    for (int i = tid; i < nf; i += dk::THREADS) s_hexp[i] = 0;
    if (route_mode && !P.solo) {
#pragma unroll 1
        for (int i = tid; i < T * P.nb * P.kk; i += dk::THREADS) s_rank[i] = 0;
    }
    __syncthreads();
    // inputs (and the workspace) may be written by the preceding kernel in the stream
    griddep_wait();
    griddep_launch_dependents();
    unsigned long long old_count = 0;
    // this call's epoch (thread 0, which drew old_count): calls sharing a workspace each add G to its 64-bit
    // counter; the tag runs through 1 .. 2^32-1 (never 0, the value of a zeroed word):
    // (call mod (2^32 - 1)) + 1, with call = counter / G and 2^32 = 1 mod (2^32 - 1)
    auto set_epoch = [&]() {
        const unsigned long long call = __umul64hi(old_count, P.dv_g64);
        unsigned long long f = (call >> 32) + (call & 0xFFFFFFFFull);
        f = (f >> 32) + (f & 0xFFFFFFFFull);
        if (f >= 0xFFFFFFFFull) f -= 0xFFFFFFFFull;
        misc[M_EPOCH] = (int)(uint32_t)(f + 1ull);
    };

    // ---------------- inputs: x (and the logits, when aligned) by one bulk copy each
    {
        const int nx = T * (H >> 3);  // 16-byte pieces of x
        const bool lbulk = route_mode && P.logits_bulk;
        if (tid == 0) {
            const uint32_t xbytes = (uint32_t)(T * H * 2), lbytes = lbulk ? (uint32_t)(T * E * 4) : 0u;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(ibar)),
                         "r"(xbytes + lbytes) : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                             smem_u32(xraw)), "l"(a.x), "r"(xbytes), "r"(smem_u32(ibar)) : "memory");
            if (lbulk)
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 smem_u32(lg)), "l"(a.logits), "r"(lbytes), "r"(smem_u32(ibar)) : "memory");
            old_count = atomicAdd(a.bar, 1ull);
        }
        if (route_mode && !lbulk) {  // unaligned logits: 4-byte async copies
            const int nl = T * E;
#pragma unroll 1
            for (int i = tid; i < nl; i += dk::THREADS) cp4(lg + i, a.logits + i);
            cp_commit();
            cp_wait<0>();
        }
        {  // bounded wait for the bulk copies
            uint32_t ok = 0;
            const unsigned long long t0 = globaltimer();
#pragma unroll 1
            while (true) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                    : "=r"(ok)
                    : "r"(smem_u32(ibar))
                    : "memory");
                if (ok || *abort_flag) break;
                if (globaltimer() - t0 > P.wait_ns) {
                    *abort_flag = 1;
                    raise_dev_error(FT_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        if (route_mode && !lbulk) __syncthreads();
        bool big = false;
        const int st0 = P.solo ? 32 : 0;  // one routed token: warp 0 routes while the other warps stage x
#pragma unroll 1
        for (int i = tid - st0; i >= 0 && i < nx; i += dk::THREADS - st0) {
            const int r = fdiv(i, P.dv_xrow), cp = i - r * (H >> 3);
            const uint4 v = *reinterpret_cast<const uint4*>(xraw + i * 8);
            const uint4 o = make_uint4(bf16x2_to_f16x2(v.x, big), bf16x2_to_f16x2(v.y, big), bf16x2_to_f16x2(v.z, big),
                                       bf16x2_to_f16x2(v.w, big));
            *reinterpret_cast<uint4*>(xs + r * P.xs_stride + staged_pos(cp * 8)) = o;
        }
        if (big) misc[M_FLAG] = 1;
    }

    if (P.solo) {
        if (warp == 0) {
            // one routed token: warp 0 takes its top k (one warp reduction per rank), orders the k distinct
            // experts by id (permuted row = rank of the id among them) and writes the selected-expert list
            bool bad = false;
            const int e = select_topk8(lg, E, k, bad);  // lane j < k: expert of rank j
            if (__any_sync(0xffffffffu, bad) && lane == 0) raise_dev_error(FT_DEVERR_NAN_LOGIT);
            const int ej = (lane < k) ? e : 0x7fffffff;
            int pos = 0;
#pragma unroll 4
            for (int i = 0; i < k; ++i) pos += __shfl_sync(0xffffffffu, ej, i) < ej;
            if (lane < k) {
                const int wi = weight_index(W, e);
                s_ids[lane] = e;
                s_plist[pos] = lane;
                s_ptok[pos] = 0;
                s_pexp[pos] = e;
                s_ulist[pos] = e;
                s_ubeg[pos] = pos;
                s_uwi[pos] = wi;
            }
            if (lane == 0) {
                misc[M_U] = k;
                s_ubeg[k] = k;
                set_epoch();
            }
        }
    } else {
    // ---------------- router: top-k of every token (route mode)
    if (route_mode) {
        const int nb = P.nb, kk = P.kk, C = nb * kk;
        // level 1: rank within each block of 32 logits; the kk best become sorted candidates.
        // Key = (order-preserving key of the fp32 logit, then ~expert): larger is better, and
        // equal logits rank the lower expert id first.
        bool bad = false;
#pragma unroll 1
        for (int b = warp; b < T * nb; b += dk::NW) {
            const int t = fdiv(b, P.dv_nb), bb = b - t * nb;
            const int e = bb * 32 + lane;
            const float v = (e < E) ? lg[t * E + e] : 0.0f;
            const uint32_t key = (e < E) ? logit_key(v) : 0u;
            bad |= (e < E) && ((v != v) || (v == INFINITY));
            int rank = 0;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) {
                const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
                rank += (kj > key) || (kj == key && j < lane);
            }
            if (rank < kk)
                cand[b * kk + rank] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_dev_error(FT_DEVERR_NAN_LOGIT);
        __syncthreads();
        if (C <= 64) {
            // level 2 over the whole CTA: eight consecutive lanes per candidate, each comparing it with an
            // eighth of the token's C candidates; the eight counts summed by shuffles give its rank (keys
            // are distinct, so the ranks are too)
            const int per = (C + 7) >> 3;
#pragma unroll 1
            for (int base = 0; base < T * C * 8; base += dk::THREADS) {
                const int idx = base + tid;
                const bool in = idx < T * C * 8;
                const int tc = idx >> 3, part = idx & 7;
                const int t = in ? fdiv(tc, P.dv_c) : 0;
                const unsigned long long* ct = cand + t * C;
                const unsigned long long key = in ? cand[tc] : 0ull;
                int r = 0;
                const int j0 = part * per, j1 = min(C, j0 + per);
#pragma unroll 4
                for (int j = j0; j < j1; ++j) r += ct[j] > key;
                r += __shfl_xor_sync(0xffffffffu, r, 1);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                r += __shfl_xor_sync(0xffffffffu, r, 4);
                if (in && part == 0 && r < k) s_ids[t * k + r] = (int)(0xFFFFFFFFu - (uint32_t)key);
            }
            __syncthreads();
        } else {
            // level 2: rank of a candidate = sum over the token's blocks of the number of that
            // block's candidates that beat it (binary search in the sorted list)
#pragma unroll 1
            for (int i = tid; i < T * C * nb; i += dk::THREADS) {
                const int tc = fdiv(i, P.dv_nb), L = i - tc * nb;
                const int t = fdiv(tc, P.dv_c);
                const unsigned long long key = cand[tc];
                const unsigned long long* list = cand + t * C + L * kk;
                int lo = 0, hi = kk;
#pragma unroll 1
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (list[mid] > key) lo = mid + 1;
                    else hi = mid;
                }
                if (lo) atomicAdd(&s_rank[tc], lo);
            }
            __syncthreads();
            // the k best of token t, in order, by warp t mod NW
#pragma unroll 1
            for (int t = warp; t < T; t += dk::NW) {
#pragma unroll 1
                for (int i = lane; i < C; i += 32) {
                    const int r = s_rank[t * C + i];
                    if (r < k) s_ids[t * k + r] = (int)(0xFFFFFFFFu - (uint32_t)cand[t * C + i]);
                }
            }
            __syncthreads();
        }
    }

    // ---------------- grouping: permuted row of slot f = #{f2 : e2 < e} + #{f2 < f : e2 == e} (every
    // token's ids are in: the router ends with a CTA barrier)
    if (!route_mode) __syncthreads();
    if (route_mode && nf <= 32) {
        if (warp == 0) {  // one warp, shuffles
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
#pragma unroll 1
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
    if (!(route_mode && nf <= 32)) __syncthreads();
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
                const int wi = weight_index(W, s_pexp[p]);
                s_ulist[u] = s_pexp[p];
                s_ubeg[u] = p;
                s_uwi[u] = wi;
            }
            run += __popc(b);
        }
        if (lane == 0) {
            misc[M_U] = run;
            s_ubeg[run] = nf;
            set_epoch();
        }
    }
    }  // general routing and grouping
    __syncthreads();
    if (misc[M_FLAG]) {  // rare: x rows with values beyond the f16 range
        restage_scaled(misc + M_XEXP, xs, P.xs_stride, T, H, a.x, nullptr);
        __syncthreads();
    }
    if (!P.solo) work_split(misc[M_U]);
    const unsigned int epoch = (unsigned int)misc[M_EPOCH];


    // ---------------- weight stream: per-lane async copies into this warp's ring.  The issue
    // cursor walks this warp's K-blocks: within a run (a tile, or an (output tile, expert) pair)
    // consecutive K-blocks are 1024 code bytes and 128 scale bytes apart.
    int is_n = 0, is_left = 0, is_ph = 1, is_run = 0, is_kb0 = 0;
    // bytes of a 16-row tile (gate/up, down) and of a K-block's scales: NVFP4 1152-byte K-blocks (128
    // scale bytes), MXFP4 1088-byte ones (64)
    // MXFP8: 2112-byte K-blocks (2048 code bytes)
    constexpr int cb_kb = FMT == 2 ? 2048 : 1024;  // code bytes of a K-block
    const int tile_b1 = FMT == 2 ? (33 * H) >> 1 : FMT ? (17 * H) >> 1 : 9 * H;
    const int tile_b2 = FMT == 2 ? (33 * I) >> 1 : FMT ? (17 * I) >> 1 : 9 * I;
    constexpr int sc_kb = FMT ? 64 : 128;
    const uint8_t* is_cb = nullptr;  // this lane's codes of the next K-block (nullptr: expert without weights)
    const uint8_t* is_sb = nullptr;  // this lane's scale word of it
    // shared address of this lane's code piece in ring slot 0 (16 bytes per lane and half tile; MXFP8: 32);
    // its scale word is sc_off further
    const uint32_t ring_l = smem_u32(ring) + lane * (cb_kb >> 6);
    const int sc_off = cb_kb + lane * 4 - lane * (cb_kb >> 6);
    // first K-block `kb` of run `run` of phase `ph` (run: local tile, or local (output tile, expert))
    auto open_run = [&](int ph, int run, int kb, int left) {
        is_ph = ph;
        is_run = run;
        is_left = left;
        int wi, KB;
        const uint8_t* base;
        if (ph == 1) {
            const int t = p1_beg + run;
            const int u = fdiv(t, P.dv_tgu);
            wi = s_uwi[u];
            KB = KB1;
            base = W.gu_codes + (int64_t)max(wi, 0) * W.gu_codes_stride + (int64_t)(t - u * tiles_gu) * tile_b1;
        } else {
            const int otl = div_u(run), u = run - otl * U;
            wi = s_uwi[u];
            KB = KB2;
            base = W.d_codes + (int64_t)max(wi, 0) * W.d_codes_stride + (int64_t)(o_beg + otl) * tile_b2;
        }
        is_cb = (wi >= 0) ? base + kb * cb_kb + lane * (cb_kb >> 6) : nullptr;  // this lane's first code byte
        is_sb = base + KB * cb_kb + kb * sc_kb + lane * 4;                        // and scale word
    };
    const bool sc_lane = lane * 4 < sc_kb;  // lanes holding a scale word of a K-block
    auto issue = [&]() {
        if (is_n < cnt) {
            if (is_left == 0 || is_n == cnt1) {
                if (is_n == cnt1) {  // this warp's first down K-block
                    const int r = ib2 / KB2, kb = ib2 - r * KB2;
                    open_run(2, r, kb, KB2 - kb);
                } else {  // next run of the same phase
                    open_run(is_ph, is_run + 1, 0, is_ph == 1 ? KB1 : KB2);
                }
            }
            const uint32_t d = ring_l + (uint32_t)((is_n & (R - 1)) * ITEMB);
            if (is_cb) {
                if (FMT == 2) {  // 32 code bytes per lane and half tile
                    cp16s(d, is_cb);
                    cp16s(d + 16, is_cb + 16);
                    cp16s(d + 1024, is_cb + 1024);
                    cp16s(d + 1040, is_cb + 1040);
                } else {
                    cp16s(d, is_cb);
                    cp16s(d + 512, is_cb + 512);
                }
                if (sc_lane) cp4s(d + sc_off, is_sb);
                is_cb += cb_kb;
            } else {  // no weights behind this expert: zeros
                uint8_t* slot = ring + (is_n & (R - 1)) * ITEMB;
#pragma unroll 1
                for (int o = lane * 16; o < cb_kb; o += 512) *reinterpret_cast<uint4*>(slot + o) = make_uint4(0u, 0u, 0u, 0u);
                if (sc_lane) *reinterpret_cast<uint32_t*>(slot + cb_kb + lane * 4) = 0u;
            }
            is_sb += sc_kb;
            --is_left;
            ++is_n;
            cp_commit();  // one group per K-block: the waits count groups
        }
    };
    if (cnt1 > 0) {
        const int tl = ib1 / KB1, kb = ib1 - tl * KB1;
        open_run(1, tl, kb, KB1 - kb);
    }
    // the gate/up K-blocks go first; the down K-blocks follow as the ring frees up, the rest of them
    // once this warp's gate/up K-blocks are all consumed (they land during the hand-off)
#pragma unroll 1
    for (int j = 0; j < min(R, cnt1 > 0 ? cnt1 : cnt); ++j) issue();
    // with the weights on their way: the routing weights exp(l_j - l_0) / sum over the k selected (the
    // router's arithmetic), token t by warp t mod NW, and the tensor scales of the selected experts
    if (route_mode) {
#pragma unroll 1
        for (int t = warp; t < T; t += dk::NW) {
            const int e = (lane < k) ? s_ids[t * k + lane] : 0;
            const float v = (lane < k) ? lg[t * E + e] : -INFINITY;
            const float m = __shfl_sync(0xffffffffu, v, 0);
            float w;
            if (m == -INFINITY || m != m) {
                w = P.inv_k;
            } else {
                const float ej = (lane < k) ? expf(v - m) : 0.0f;
                const float s = warp_sum(ej);
                w = ej / s;
            }
            if (lane < k) {
                s_wts[t * k + lane] = w;
                if (c == 0 && a.ids_out) {
                    a.ids_out[t * k + lane] = e;
                    a.w_out[t * k + lane] = w;
                }
            }
        }
    }
#pragma unroll 1
    for (int u = tid; u < U; u += dk::THREADS) {
        const int wi = s_uwi[u];
        const float* ts = FMT ? nullptr : W.tscale + (int64_t)(wi >= 0 ? wi : 0) * W.tscale_stride;
        s_ts[4 * u + 0] = (wi >= 0) ? (FMT ? 1.0f : __ldg(ts + 0)) : 0.0f;
        s_ts[4 * u + 1] = (wi >= 0) ? (FMT ? 1.0f : __ldg(ts + 1)) : 0.0f;
        s_ts[4 * u + 2] = (wi >= 0) ? (FMT ? 1.0f : __ldg(ts + 2)) : 0.0f;
    }

    const int g8 = lane >> 2, q4 = lane & 3;
    const int hw_row = I >> 1;  // h words per permuted row
    unsigned long long* hw = reinterpret_cast<unsigned long long*>(a.hbuf);

    // partial tiles [16][TC]: this lane's accumulator (rows g8, g8+8; columns cg*8 + 2q4, +1)
    auto store_acc = [&](float* dst, int cg, const float4& v, int tu) {
        const int col = cg * 8 + 2 * q4;
        if (col < tu) {
            dst[g8 * TC + col] = v.x;
            dst[(g8 + 8) * TC + col] = v.z;
        }
        if (col + 1 < tu) {
            dst[g8 * TC + col + 1] = v.y;
            dst[(g8 + 8) * TC + col + 1] = v.w;
        }
    };
    // tensor scale j of expert index u: from shared memory once a CTA barrier has passed since it
    // was stored (split phases), else from global memory
    auto tscale = [&](int u, int j, bool shared) {
        if (shared) return s_ts[4 * u + j];
        const int wi = s_uwi[u];
        if (wi < 0) return 0.0f;
        return FMT ? 1.0f : __ldg(W.tscale + (int64_t)wi * W.tscale_stride + j);
    };
    // is warp w without K-blocks in a split phase of ni K-blocks?
    auto empty_warp = [&](int w, int ni) { return ni && ((w * ni) >> dk::LOG_NW) == (((w + 1) * ni) >> dk::LOG_NW); };
    // phase-1 epilogue of tile t (global index) from the partial tiles at tile + w*16*TC, w in
    // [wlo, whi] (skipping warps without K-blocks of a split phase of ni K-blocks; ni = 0: none):
    // h of the tile's 8 (gate, up) row pairs for its tu tokens, as h words; items (token, pair)
    auto finish1 = [&](int t, const float* tile, int wlo, int whi, int ni, bool shared) {
        const int u = fdiv(t, P.dv_tgu), lt = t - u * tiles_gu;
        const int wi = s_uwi[u];
        const int pb = s_ubeg[u], tu = s_ubeg[u + 1] - pb;
        const float tsg = tscale(u, 0, shared), tsu = tscale(u, 1, shared);
        // lane 8*tt' + pr handles pair pr of token tt; the 32 lanes cover 4 tokens per pass
#pragma unroll 1
        for (int idx0 = 0; idx0 < 8 * tu; idx0 += 32) {
            const int idx = idx0 + lane;
            const int pr = idx & 7, tt = idx >> 3;
            float hv = 0.0f;
            if (idx < 8 * tu) {
                float gs = 0.0f, us = 0.0f;
#pragma unroll 1
                for (int w = wlo; w <= whi; ++w) {
                    if (empty_warp(w, ni)) continue;
                    const float* s = tile + w * 16 * TC;
                    gs += s[(2 * pr) * TC + tt];
                    us += s[(2 * pr + 1) * TC + tt];
                }
                if (wi >= 0) {
                    const float sc = pow2i(misc[M_XEXP + s_ptok[pb + tt]]);
                    hv = silu_f32(gs * tsg * sc) * (us * tsu * sc);
                }
            }
            // lanes of pairs 2j, 2j+1 are neighbours: the even one stores the word
            const uint32_t hb = bf16_bits(hv);
            const uint32_t hb1 = __shfl_down_sync(0xffffffffu, hb, 1);
            if (idx < 8 * tu && !(pr & 1))
                st_relaxed_u64(hw + (int64_t)(pb + tt) * hw_row + lt * 4 + (pr >> 1),
                               (unsigned long long)(hb | (hb1 << 16)) | ((unsigned long long)epoch << 32));
        }
    };
    // phase-2 epilogue of run r (local index: output tile r / U, expert r % U)
    auto finish2 = [&](int r, const float* tile, int wlo, int whi, int ni, bool shared) {
        const int otl = div_u(r), u = r - otl * U;
        const int wi = s_uwi[u];
        const int pb = s_ubeg[u], tu = s_ubeg[u + 1] - pb;
        const float tsd = tscale(u, 2, shared);
#pragma unroll 1
        for (int idx = lane; idx < 16 * tu; idx += 32) {
            const int row = idx & 15, tt = idx >> 4;
            float ys = 0.0f;
#pragma unroll 1
            for (int w = wlo; w <= whi; ++w)
                if (!empty_warp(w, ni)) ys += tile[w * 16 * TC + row * TC + tt];
            const int p = pb + tt;
            ys = (wi >= 0) ? ys * (tsd * pow2i(s_hexp[p])) : 0.0f;
            ybuf[(otl * nf + s_plist[p]) * 16 + row] = ys;
            if (a.y) a.y[(int64_t)p * H + (o_beg + otl) * 16 + row] = ys;
        }
    };
    // warps whose K-block range of a split phase covers run r (KB K-blocks per run, ni in all):
    // warp(i) = floor(((i + 1) * NW - 1) / ni) covers K-block i
    auto cover = [&](int r, int KB, int ni, int& wlo, int& whi) {
        wlo = ((r * KB + 1) * dk::NW - 1) / ni;
        whi = (((r + 1) * KB) * dk::NW - 1) / ni;
    };

    // this warp's K-blocks [ib, ie) of a phase (KB per run), consumed in ring order n0, n0+1, ...:
    // runs in turn, each accumulated in registers, then flushed into its slot (split phase) or
    // finished in the warp (whole runs)
    auto run_phase = [&](int ph, int n0, int ib, int ie, int KB, bool split) {
        int n = n0;
#pragma unroll 1
        for (int i = ib; i < ie;) {
            const int run = fdiv(i, ph == 1 ? P.dv_kb1 : P.dv_kb2);
            const int kb0 = i - run * KB, kb1 = min(KB, kb0 + (ie - i));
            int pb, tu;
            const __half* r0;
            const __half* r1;
            if (ph == 1) {
                const int u = fdiv(p1_beg + run, P.dv_tgu);
                pb = s_ubeg[u];
                tu = s_ubeg[u + 1] - pb;
                r0 = xs + s_ptok[pb + min(g8, tu - 1)] * P.xs_stride + q4 * 8;
                r1 = xs + s_ptok[pb + min(8 + g8, tu - 1)] * P.xs_stride + q4 * 8;
            } else {
                const int u = run - div_u(run) * U;
                pb = s_ubeg[u];
                tu = s_ubeg[u + 1] - pb;
                r0 = hs + (pb + min(g8, tu - 1)) * P.hs_stride + q4 * 8;
                r1 = hs + (pb + min(8 + g8, tu - 1)) * P.hs_stride + q4 * 8;
            }
            float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 1
            for (int kb = kb0; kb < kb1; ++kb, ++n) {
                // K-block n of this lane has landed: R - 1 younger groups in flight in the steady state
                if (is_n - n - 1 >= R - 1) cp_wait<R - 1>();
                else cp_wait_upto(is_n - n - 1);
                const uint8_t* slot = ring + (n & (R - 1)) * ITEMB;
                const float4 v = FMT == 2 ? kblock_partial_mx8(slot, r0 + kb * 128)
                                 : FMT    ? kblock_partial_mx(slot, r0 + kb * 128)
                                          : kblock_partial(slot, r0 + kb * 128);
                acc0.x += v.x, acc0.y += v.y, acc0.z += v.z, acc0.w += v.w;
                if (tu > 8) {
                    const float4 v1 = FMT == 2 ? kblock_partial_mx8(slot, r1 + kb * 128)
                                      : FMT    ? kblock_partial_mx(slot, r1 + kb * 128)
                                               : kblock_partial(slot, r1 + kb * 128);
                    acc1.x += v1.x, acc1.y += v1.y, acc1.z += v1.z, acc1.w += v1.w;
                }
                issue();  // into the slot just read (this lane's own bytes)
            }
            float* dst = split ? slots + (run + warp) * 16 * TC : wscr + warp * 16 * TC;
            store_acc(dst, 0, acc0, tu);
            if (tu > 8) store_acc(dst, 1, acc1, tu);
            if (!split) {
                __syncwarp();
                if (ph == 1) finish1(p1_beg + run, dst, 0, 0, 0, false);
                else finish2(run, dst, 0, 0, 0, false);
                __syncwarp();
            }
            i += kb1 - kb0;
        }
    };

    // ---------------- phase 1: gate/up K-blocks -> partial tiles -> h words
    run_phase(1, 0, ib1, ie1, KB1, split1);
#pragma unroll 1
    while (is_n < min(cnt, cnt1 + R)) issue();  // the ring full of down K-blocks before the hand-off
    if (split1) {
        __syncthreads();
        // tiles shared by warps: sum the slots in warp order
#pragma unroll 1
        for (int tl = warp; tl < n_t1; tl += dk::NW) {
            int wlo, whi;
            cover(tl, KB1, ni1, wlo, whi);
            finish1(p1_beg + tl, slots + tl * 16 * TC, wlo, whi, ni1, true);
        }
    }
    if (n_ot == 0) {
        cp_wait<0>();  // no copy may land after the CTA exits
        return;
    }

    // ---------------- phase 2: all h rows (permuted order) staged as f16, as each becomes available (over
    // the raw logits: every warp has read them by the barrier)
    if (!split1) __syncthreads();
    {
        const unsigned int want = (P.wait_site == FT_WAIT_SITE_DECODE_H) ? (epoch ^ 0x80000000u) : epoch;
        const int total = nf * hw_row;
        bool big = false;
        // B loads in flight per thread; words whose tag is not there yet are read again, all
        // together, until they are (bounded)
        constexpr int B = 4;
#pragma unroll 1
        for (int base = tid; base < total; base += B * dk::THREADS) {
            unsigned long long v[B];
            uint32_t pending = 0;
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int idx = base + u * dk::THREADS;
                if (idx < total) {
                    v[u] = ld_relaxed_u64(hw + idx);
                    pending |= ((uint32_t)(v[u] >> 32) != want) << u;
                }
            }
            if (pending) {
                const unsigned long long t0 = globaltimer();
#pragma unroll 1
                while (pending) {
                    if (*abort_flag) break;
                    if (globaltimer() - t0 > P.wait_ns) {
                        *abort_flag = 1;
                        raise_dev_error(FT_DEVERR_TIMEOUT);
                        break;
                    }
#pragma unroll
                    for (int u = 0; u < B; ++u)
                        if (pending & (1u << u)) v[u] = ld_relaxed_u64(hw + base + u * dk::THREADS);
#pragma unroll
                    for (int u = 0; u < B; ++u)
                        if ((pending & (1u << u)) && (uint32_t)(v[u] >> 32) == want) pending &= ~(1u << u);
                }
            }
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int idx = base + u * dk::THREADS;
                if (idx < total) {
                    const int r = fdiv(idx, P.dv_hrow), cc = idx - r * hw_row;
                    *reinterpret_cast<uint32_t*>(hs + r * P.hs_stride + staged_pos(2 * cc)) =
                        bf16x2_to_f16x2((uint32_t)v[u], big);
                }
            }
        }
        if (big) misc[M_HFLAG] = 1;
        __syncthreads();
        if (misc[M_HFLAG]) {
            restage_scaled(s_hexp, hs, P.hs_stride, nf, I, nullptr, hw);
            __syncthreads();
        }
    }
    run_phase(2, cnt1, ib2, ie2, KB2, split2);
    cp_wait<0>();
    __syncthreads();
    if (split2) {
#pragma unroll 1
        for (int r = warp; r < nr2; r += dk::NW) {
            int wlo, whi;
            cover(r, KB2, ni2, wlo, whi);
            finish2(r, slots + r * 16 * TC, wlo, whi, ni2, true);
        }
        __syncthreads();
    }
    // combine: out[t][row] = bf16(sum_j w[t][j] * y[t*k + j][row]) in slot order j;
    // item i = (otl * T + tok) * 16 + row
    if (a.out) {
#pragma unroll 1
        for (int i = tid; i < n_ot * 16 * T; i += dk::THREADS) {
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

// Shared memory: routing and grouping tables, staged x, one area that holds the
// raw inputs and the router's candidates and later the staged h rows, the
// partial-tile slots, the warps' scratch tiles, the per-slot down outputs and
// the warps' K-block rings (R slots each: 16, else 8, 4 or 2, whichever fits).
static int item_bytes(int layout) { return layout == FT_LAYOUT_MXFP8_DECODE_TILES ? dk::ITEM8 : dk::ITEM; }

static bool plan_decode(int T, int k, int E, int H, int I, int G, bool route_mode, int item, DecodePlan& p,
                        std::string& why) {
    const int nf = T * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 128);
        return (int)o;
    };
    p.nb = (E + 31) / 32;
    p.kk = std::min(k, 32);
    const int C = p.nb * p.kk;
    p.off_misc = take(M_COUNT * 4);
    p.off_ids = take((size_t)nf * 4);
    p.off_wts = take((size_t)nf * 4);
    p.off_plist = take((size_t)nf * 4);
    p.off_ptok = take((size_t)nf * 4);
    p.off_pexp = take((size_t)nf * 4);
    p.off_hexp = take((size_t)nf * 4);
    p.off_ulist = take((size_t)nf * 4);
    p.off_ubeg = take((size_t)(nf + 1) * 4);
    p.off_uwi = take((size_t)nf * 4);
    p.off_ts = take((size_t)nf * 16);
    p.off_rank = take(route_mode ? (size_t)T * C * 4 : 4);
    p.xs_stride = H + dk::XPAD;
    p.hs_stride = I + dk::XPAD;
    p.off_xs = take((size_t)T * p.xs_stride * 2);
    const size_t lg_bytes = route_mode ? align_up((size_t)T * E * 4, 16) : 0;
    const size_t xraw_bytes = align_up((size_t)T * H * 2, 16);
    const size_t cand_bytes = route_mode ? (size_t)T * C * 8 : 0;
    const size_t big = std::max((size_t)nf * p.hs_stride * 2, lg_bytes + xraw_bytes + cand_bytes);
    p.off_big = take(big);
    p.off_xraw = p.off_big + (int)lg_bytes;
    p.off_cand = p.off_xraw + (int)xraw_bytes;
    p.tc = T;
    {
        // enough slots for a split of either phase when the CTA's share allows it: at most
        // ceil(n1 / G) + 2 gate/up tiles (float rounding of the byte balance) and max_ot * U runs
        const int umax = std::min(E, nf);
        const int t1max = (umax * (I / 8) + G - 1) / G + 2, r2max = ((H / 16 + G - 1) / G) * umax;
        p.nslot = std::max(dk::MINSLOT, std::min(T <= 2 ? dk::MAXSLOT : dk::MINSLOT, dk::NW + std::max(t1max, r2max)));
    }
    p.off_slot = take((size_t)p.nslot * 16 * T * 4);
    p.off_wscr = take((size_t)dk::NW * 16 * T * 4);
    const int n2 = H / 16;
    p.max_ot = (n2 + G - 1) / G;
    p.off_ybuf = take((size_t)p.max_ot * nf * 16 * 4);
    p.off_ring = (int)off;
    p.ring = 0;
    for (int r : {16, 8, 4, 2})
        if (off + (size_t)dk::NW * r * item <= dk::SMEM_BUDGET) {
            p.ring = r;
            break;
        }
    if (!p.ring) {
        why = "activations of " + std::to_string(T) + " tokens and their " + std::to_string(nf) +
              " expert rows do not fit the fused kernel's shared memory";
        return false;
    }
    p.smem = (int)(off + (size_t)dk::NW * p.ring * item);
    p.item = item;
    p.dv_k = make_fastdiv((uint32_t)k);
    p.dv_xrow = make_fastdiv((uint32_t)(H / 8));
    p.dv_hrow = make_fastdiv((uint32_t)(I / 2));
    p.dv_g = make_fastdiv((uint32_t)G);
    p.dv_t = make_fastdiv((uint32_t)T);
    p.dv_nb = make_fastdiv((uint32_t)p.nb);
    p.dv_c = make_fastdiv((uint32_t)C);
    p.dv_tgu = make_fastdiv((uint32_t)(I / 8));
    p.dv_kb1 = make_fastdiv((uint32_t)(H / 128));
    p.dv_kb2 = make_fastdiv((uint32_t)(I / 128));
    // ceil(2^64 / G): mulhi(x, m) = floor(x / G) for every x below 2^64 / G (the error of m, under G,
    // times x stays under 2^64)
    p.dv_g64 = (G <= 1) ? ~0ull : (~0ull / (unsigned long long)G) + 1ull;
    p.inv_k = 1.0f / (float)k;
    p.wait_ns = g_wait_ns.load();
    p.wait_site = g_wait_site.load();
    p.logits_bulk = 0;
    p.solo = (route_mode && T == 1 && E <= 256) ? 1 : 0;
    p.mx = 0;
    return true;
}

// The kernels' shared-memory limit, set once per device before the first launch there.
static ft_status decode_attributes(const char* fn) {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(FT_ERR_CUDA, std::string(fn) + ": no current device");
    }
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return FT_OK;
    const int lim = (int)dk::SMEM_BUDGET;
    const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    const cudaError_t errs[10] = {
        cudaFuncSetAttribute(k_moe_decode<16, 0>, attr, lim), cudaFuncSetAttribute(k_moe_decode<8, 0>, attr, lim),
        cudaFuncSetAttribute(k_moe_decode<4, 0>, attr, lim),  cudaFuncSetAttribute(k_moe_decode<2, 0>, attr, lim),
        cudaFuncSetAttribute(k_moe_decode<16, 1>, attr, lim), cudaFuncSetAttribute(k_moe_decode<8, 1>, attr, lim),
        cudaFuncSetAttribute(k_moe_decode<4, 1>, attr, lim),  cudaFuncSetAttribute(k_moe_decode<2, 1>, attr, lim),
        cudaFuncSetAttribute(k_moe_decode<4, 2>, attr, lim),  cudaFuncSetAttribute(k_moe_decode<2, 2>, attr, lim)};
    for (cudaError_t e : errs)
        if (e != cudaSuccess) {
            cudaGetLastError();  // not sticky: leave no error behind for the launch check
            return fail(FT_ERR_CUDA, std::string(fn) + ": setting the shared-memory limit: " + cudaGetErrorString(e));
        }
    done[dev] = true;
    return FT_OK;
}

static ft_status launch_decode(DecodeArgs a, ft_stream_t stream, const char* fn) {
    const ft_moe_layer_weights& W = a.W;
    const int G = sm_count();
    std::string why;
    if (!plan_decode(a.T, a.k, W.E, W.H, W.I, G, a.logits != nullptr, item_bytes(W.layout), a.P, why))
        return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": " + why);
    a.P.logits_bulk = a.logits && aligned(a.logits, 16) && ((size_t)a.T * W.E * 4) % 16 == 0;
    a.P.mx = W.layout == FT_LAYOUT_MXFP4_DECODE_TILES ? 1 : W.layout == FT_LAYOUT_MXFP8_DECODE_TILES ? 2 : 0;
    ft_status st = decode_attributes(fn);
    if (st != FT_OK) return st;
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
    cudaError_t e;
    // (an MXFP8 ring of 2112-byte slots holds at most 4 per warp in the shared-memory budget)
    const int R = a.P.ring, F = a.P.mx;
    if (F == 2) e = cudaLaunchKernelEx(&cfg, R >= 4 ? k_moe_decode<4, 2> : k_moe_decode<2, 2>, a);
    else if (F == 1)
        e = cudaLaunchKernelEx(&cfg, R == 16 ? k_moe_decode<16, 1> : R == 8 ? k_moe_decode<8, 1> :
                                     R == 4 ? k_moe_decode<4, 1> : k_moe_decode<2, 1>, a);
    else
        e = cudaLaunchKernelEx(&cfg, R == 16 ? k_moe_decode<16, 0> : R == 8 ? k_moe_decode<8, 0> :
                                     R == 4 ? k_moe_decode<4, 0> : k_moe_decode<2, 0>, a);
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
    a.bar = static_cast<unsigned long long*>(ws);
    a.hbuf = static_cast<char*>(ws) + 256;
    a.T = T;
    a.k = k;
    return launch_decode(a, stream, fn);
}

// Argument checks of the fused decode step (shared by both entry points).
static ft_status check_layer_decode_args(const ft_moe_layer_weights* W, const float* logits, const uint16_t* x, int T,
                                         int k, uint16_t* out, int32_t* ids, float* w, const char* fn) {
    ft_status st = validate_weights(W, fn);
    if (st != FT_OK) return st;
    if (W->layout != FT_LAYOUT_DECODE_TILES && W->layout != FT_LAYOUT_MXFP4_DECODE_TILES &&
        W->layout != FT_LAYOUT_MXFP8_DECODE_TILES)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weights must use FT_LAYOUT_DECODE_TILES or an MX tile layout");
    if (T < 0 || T > dk::MAXT || k <= 0 || k > W->E || k > dk::MAXK)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 0 <= T <= 16 and 1 <= k <= min(E, 32)");
    if (T == 0) return FT_OK;
    if (!logits || !x || !out) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if ((ids == nullptr) != (w == nullptr))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": give both ids and w or neither");
    if (!aligned(x, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": x needs 16-byte alignment");
    if (!aligned(logits, 4)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": logits need 4-byte alignment");
    return FT_OK;
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

ft_status ft_debug_inject_wait_expiry(int site, uint64_t limit_ns) {
    if (site != FT_WAIT_SITE_NONE && site != FT_WAIT_SITE_DECODE_H && site != FT_WAIT_SITE_PREFILL_TOKEN)
        return fail(FT_ERR_INVALID_ARG, "ft_debug_inject_wait_expiry: unknown wait site");
    if (site != FT_WAIT_SITE_NONE && (limit_ns == 0 || limit_ns > dk::WAIT_NS))
        return fail(FT_ERR_INVALID_ARG, "ft_debug_inject_wait_expiry: need 0 < limit_ns <= 2 s");
    g_wait_ns.store(site == FT_WAIT_SITE_NONE ? dk::WAIT_NS : limit_ns);
    g_wait_site.store(site);
    return FT_OK;
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
    // every argument check comes before any CUDA call
    ft_status st = check_layer_decode_args(W, logits, x, T, k, out, ids, w, fn);
    if (st != FT_OK || T == 0) return st;
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
    ft_status st = check_layer_decode_args(W, logits, x, T, k, out, ids, w, fn);
    if (st != FT_OK || T == 0) return st;
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
        while (Tc > 0 && !plan_decode(Tc, k, W->E, W->H, W->I, sm_count(), true, item_bytes(W->layout), probe, why))
            --Tc;
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
        a.bar = static_cast<unsigned long long*>(ws);
        a.hbuf = static_cast<char*>(ws) + 256;
        a.T = std::min(Tc, T - t0);
        a.k = k;
        st = launch_decode(a, stream, fn);
        if (st != FT_OK) return st;
    }
    return FT_OK;
}

}  // extern "C"
