// prefill.cu -- grouped expert FFN for many tokens (prefill) on the 5th-
// generation tensor cores: block-scaled FP4 MMA (tcgen05.mma kind::mxf4nvf4,
// E2M1 operands, one UE4M3 scale per 16 elements), fp32 accumulators in TMEM.
//
// Each expert is an independent FFN applied to the tokens routed to it (page
// "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", MoE core mechanism);
// the weights are NVFP4 (page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把
// frontier MoE 拉回本地", sections on the evaluation and the limits).  The FP4
// MMA takes FP4 on both sides, so the activations x and h are quantised to
// NVFP4 with unit tensor scale (E4M3 scale per 16 along the reduction
// dimension); the weights' fp32 tensor scales are applied in the epilogues.
//
// Steps (one stream):
//  1. k_pf_plan: every expert's permuted rows are padded to whole 128-row
//     tiles; tile_off[e] = first tile of expert e (exclusive scan).
//  2. k_pf_quant_tokens + k_pf_gather_x: each token's x quantised once, then
//     copied in permuted order into operand tiles, with a (token, weight) table
//     of the padded rows; the gather also zeroes the fp32 output accumulator.
//  3. k_pf_gemm_res<1>: h = silu(Wg x) * (Wu x) per (expert, 128 gate/up rows,
//     128 tokens) tile, rounded to bf16 and quantised into operand tiles.
//  4. k_pf_gemm_res<2>: y = Wd h per (expert, 128 output rows, 128 tokens)
//     tile; the epilogue adds w[t][j] * y into an fp32 accumulator of the
//     output (red.global.add, whole 128-byte lines through a shared-memory
//     transpose), i.e. the routing-weighted combine.
//  5. k_pf_out: the accumulator rounded to bf16.
//
// Operand tiles ("UMMA tiles"): an [R][K] NVFP4 matrix (R a multiple of 128,
// K of 128) is stored as blocks of 128 rows x 128 K, 9216 bytes each, block
// (rt, ks) at (rt*(K/128) + ks)*9216.  In a block, code byte b (0..63) of row r
// sits at (b/16)*2048 + (r/8)*128 + (r%8)*16 + b%16 -- the tensor core's
// K-major layout without swizzle: 8-row x 16-byte core matrices, 128 bytes
// apart along the rows and 2048 bytes apart along K -- and scale j (0..7) of
// row r at 8192 + (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4, the layout that
// tcgen05.cp .32x128b.warpx4 moves into TMEM (4 columns per 64 K).  A block is
// one contiguous bulk copy.
//
// The GEMM kernels are persistent (one CTA per SM).  In k_pf_gemm_res (K up to
// 2048) the token tile stays resident in shared memory while warp 0 streams the
// weight blocks through a ring of bulk copies (cp.async.bulk + mbarriers; four
// K blocks per copy, since a bulk copy costs about the same whatever its size);
// k_pf_gemm_stream (longer K) streams both operands through a 3-stage ring.
// Warp 1 allocates TMEM and one of its threads issues
// the MMAs (two per K block, K = 64 each, scales copied to TMEM with
// tcgen05.cp) into one of two 128-column accumulators, and warps 2-17 (four per
// TMEM lane quadrant, 32 columns each) drain the other accumulator (tcgen05.ld)
// through the epilogue, so MMA and epilogue overlap.  The token tile is the
// MMA's M side: each TMEM lane is one token and its columns are weight rows, so
// the SwiGLU + NVFP4 quantisation of h and the weighted combine run without
// leaving the thread.  Every wait is bounded; on expiry
// the kernel sets FT_DEVERR_TIMEOUT and finishes, freeing its TMEM.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace ft {

namespace pf {
constexpr int BLK = 9216;           // one 128 x 128 operand block
constexpr int KPS = 4;              // K blocks per ring stage: a bulk copy costs about the same whatever
                                    // its size, so A and B each come in one copy of up to 4 blocks
constexpr int NS = 3;               // ring stages (KPS A blocks + KPS B blocks each)
constexpr int STAGE = 2 * KPS * BLK;
constexpr int EPI_WARPS = 16;       // four per TMEM lane quadrant, each draining 32 of the 128 columns
constexpr int THREADS = 32 * (2 + EPI_WARPS);  // warp 0 producer, warp 1 MMA, warps 2.. epilogue
constexpr uint32_t TMEM_COLS = 512; // 2 x 128 accumulator columns + scale-factor columns
constexpr uint32_t SF_COL0 = 256;   // 16 scale-factor columns per K block of a ring stage
constexpr unsigned long long WAIT_NS = 2000000000ull;
constexpr size_t SMEM = (size_t)NS * STAGE + 1024;
constexpr int RES_MAXKSN = 16;      // resident token tile: up to 16 K blocks (H or I up to 2048)
constexpr int RES_MAXNS = 8;        // its weight ring: up to 8 stages of KPS blocks
constexpr size_t SMEM_LIMIT = 227 * 1024 - 1024;  // dynamic shared memory, leaving room for the static part
}  // namespace pf

struct PfGemmArgs {
    const uint8_t* A;        // weights in UMMA tiles, expert e at A + e*a_stride
    int64_t a_stride;
    const float* tscale;     // per expert {gate, up, down}
    int64_t ts_stride;
    const uint8_t* B;        // activation tiles [tiles][KSN] blocks
    int MT, KSN;             // M tiles per expert, K blocks
    int E;
    const int32_t* offsets;  // [E+1] permuted rows per expert
    const int32_t* tile_off; // [E+1] padded tiles per expert (exclusive scan)
    // SwiGLU epilogue: h tiles [tiles][KSN2] blocks
    uint8_t* hq;
    int KSN2;
    // combine epilogue
    const int2* rowmeta;     // [tiles*128] (token, routing weight bits) per padded row, token -1 for padding
    float* out32;            // [T][H], or nullptr: no combine
    int H;
    int nstages;             // ring stages (resident-token-tile kernel)
    int tbufs;               // resident kernel: token-tile buffers (2: the next item's tile loads during this one)
    const int32_t* e2s;      // optional expert -> weight index (slot table); validated by the plan
    const int4* tinfo;       // [tiles] {expert, first permuted row, real rows, 0}
    float* y;                // optional [T*k][H] fp32 per-row expert outputs (tensor scale applied, no routing weight)
    int parts;               // resident kernel: work items per token tile, each a contiguous part of the weight tiles
    unsigned long long wait_ns;  // bound on any single wait (2 s; shorter under the wait-expiry test hook)
    int wait_site;           // FT_WAIT_SITE_PREFILL_TOKEN: the gate/up MMA issuer waits on a barrier nothing completes
    int cstage;              // resident kernel, down GEMM: 32 or 16 = the combine goes through a shared-memory
                             // transpose, that many columns per pass; 0 = reductions straight from the thread's row
};

// weight index of expert e (identity without a slot table; the plan has checked every expert with rows)
__device__ __forceinline__ int64_t pf_widx(const PfGemmArgs& a, int e) { return a.e2s ? (int64_t)__ldg(a.e2s + e) : e; }

// ---------------------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t pf_su(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long pf_gt() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// try_wait with a suspend-time hint: a waiting thread sleeps (up to ~1 us) instead of
// spinning, leaving issue slots to the epilogue warps; it wakes when the phase completes.
__device__ __forceinline__ bool pf_try_wait(unsigned long long* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(pf_su(b)), "r"(parity), "n"(1000)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool pf_wait(unsigned long long* b, uint32_t parity, volatile int* abort_flag,
                                        unsigned long long limit_ns) {
    if (pf_try_wait(b, parity)) return true;
    const unsigned long long t0 = pf_gt();
    while (!pf_try_wait(b, parity)) {
        if (*abort_flag) return false;
        if (pf_gt() - t0 > limit_ns) {
            *abort_flag = 1;
            raise_dev_error(FT_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Shared-memory operand descriptor of the 5th-generation tensor core, no swizzle:
// start address, leading (K-direction) and stride (row-direction) core-matrix offsets.
__device__ __forceinline__ uint64_t umma_desc(const void* p, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((pf_su(p) & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor: kind::mxf4nvf4, E2M1 x E2M1, UE4M3 scales, M = 128, N = 128, both K-major.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// A descriptor's address field counts 16-byte units, so a descriptor moves by adding the byte
// offset / 16 (shared-memory addresses stay below 256 KB: no carry out of the field).
constexpr uint64_t kDescBlk = 9216 / 16, kDescHalf = 4096 / 16, kDescSfHalf = 512 / 16;

__device__ __forceinline__ void sf_copy(uint32_t tcol, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tcol), "l"(desc));
}

__device__ __forceinline__ void mma_fp4(uint32_t dcol, uint64_t da, uint64_t db, uint32_t sfa, uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(dcol),
        "l"(da), "l"(db), "r"(kIdesc), "r"(sfa), "r"(sfb), "r"(acc));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Offset of code byte b (0..63) / scale j (0..7) of row r within a 128 x 128 block.
__host__ __device__ __forceinline__ int blk_code_off(int r, int b) {
    return (b >> 4) * 2048 + (r >> 3) * 128 + (r & 7) * 16 + (b & 15);
}
__host__ __device__ __forceinline__ int blk_scale_off(int r, int j) {
    return 8192 + (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

// ---------------------------------------------------------------------------- plan and activation tiles

// tile_off[e] = first tile of expert e (exclusive scan of its tile counts);
// tinfo[tile] = {expert, first permuted row, real rows in the tile, 0}.  With a
// slot table, an expert with rows whose slot is out of [0, n_weights) raises
// FT_DEVERR_BAD_INDEX and gets no tiles.
// offsets must partition [0, P) in order; otherwise FT_DEVERR_BAD_INDEX is
// raised and every tile count is zero, so the later kernels do nothing.
__global__ void __launch_bounds__(1024) k_pf_plan(const int32_t* __restrict__ offsets, int E, int P, int max_tiles,
                                                  const int32_t* __restrict__ e2s, int n_weights,
                                                  int32_t* __restrict__ tile_off, int4* __restrict__ tinfo) {
    __shared__ int wsum[33];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    // experts per thread: E <= 1024, so one each
    const int o0 = (tid < E) ? offsets[tid] : 0;
    const int o1 = (tid < E) ? offsets[tid + 1] : 0;
    if (tid < E && (o0 < 0 || o1 < o0 || o1 > P || (tid == 0 && o0 != 0) || (tid == E - 1 && o1 != P))) s_bad = 1;
    int n = max(o1 - o0, 0);
    if (e2s && n > 0) {  // an expert whose slot is invalid gets no tiles: its rows contribute nothing
        const int sl = e2s[tid];
        if (sl < 0 || sl >= n_weights) {
            raise_dev_error(FT_DEVERR_BAD_INDEX);
            n = 0;
        }
    }
    const int nt = (n + 127) / 128;
    int incl = nt;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = wsum[lane], si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += v;
        }
        wsum[lane] = si - s;
        if (lane == 31) wsum[32] = si;
    }
    __syncthreads();
    if (s_bad || wsum[32] > max_tiles) {
        if (tid <= E) tile_off[tid] = 0;
        if (tid == 0) raise_dev_error(FT_DEVERR_BAD_INDEX);
        return;
    }
    const int first = wsum[wid] + incl - nt;
    if (tid < E) tile_off[tid] = first;
    if (tid == 0) tile_off[E] = wsum[32];
    for (int i = 0; i < nt; ++i) tinfo[first + i] = make_int4(tid, o0 + 128 * i, min(128, n - 128 * i), 0);
}

// x[t] quantised once (unit tensor scale) into a compact row of H/2 code bytes
// followed by H/16 scale bytes.  A warp covers 1024 elements of one token, 32
// per lane (two blocks of 16), spread over as many warps as the rows allow.
__global__ void __launch_bounds__(256) k_pf_quant_tokens(const uint16_t* __restrict__ x, int T, int H,
                                                         uint8_t* __restrict__ xc) {
    const int wpt = (H + 1023) / 1024;  // warps per token
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (int64_t)T * wpt) return;
    const int t = (int)(gw / wpt), sub = (int)(gw - (int64_t)t * wpt);
    const int e0 = sub * 1024 + lane * 32;
    if (e0 >= H) return;
    uint8_t* row = xc + (int64_t)t * (H / 2 + H / 16);
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)t * H + e0);
    uint32_t cw[4], sw = 0;
#pragma unroll
    for (int bl = 0; bl < 2; ++bl) {
        float v[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint4 u = __ldg(src + 2 * bl + hh);
            const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[8 * hh + 2 * i] = __uint_as_float(words[i] << 16);
                v[8 * hh + 2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
            }
        }
        uint2 c;
        uint32_t sb;
        quant_block16_bf16(v, c, sb);
        cw[2 * bl] = c.x;
        cw[2 * bl + 1] = c.y;
        sw |= sb << (8 * bl);
    }
    *reinterpret_cast<uint4*>(row + e0 / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    *reinterpret_cast<uint16_t*>(row + H / 2 + e0 / 16) = (uint16_t)sw;
}

// Two blocks per 128-row operand tile, one per half of K: the compact quantised
// rows of the tile's tokens copied into the tile, and each row's (token,
// routing weight) for the combine (token -1 for padding rows, whose tile rows
// keep whatever they held: every output row depends only on its own tile row,
// and padding rows are skipped).  Each block resolves the tile's tokens, then
// every thread copies 16-byte pieces, many in flight.  Every block (used tile
// or not) first zeroes its share of the fp32 output accumulator (n4 float4s in
// all), which the down GEMM's combine adds into: the stores overlap the
// block's first dependent loads.
__global__ void __launch_bounds__(256, 4) k_pf_gather_x(const uint8_t* __restrict__ xc, int H, int k, int E,
                                                     const int32_t* __restrict__ perm, const float* __restrict__ w,
                                                     const int32_t* __restrict__ tile_off, const int4* __restrict__ tinfo,
                                                     uint8_t* __restrict__ xq, int2* __restrict__ rowmeta,
                                                     float4* __restrict__ out32, int64_t n4) {
    __shared__ int s_tok[128];
    {
        const int64_t per = (n4 + gridDim.x - 1) / gridDim.x, z0 = (int64_t)blockIdx.x * per;
        const int64_t z1 = min(n4, z0 + per);
        for (int64_t i = z0 + threadIdx.x; i < z1; i += blockDim.x) out32[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    // two blocks per tile, each copying half of its K blocks (H is a multiple of 256, so the halves are whole
    // K blocks); the first also writes the row table
    const int rt = blockIdx.x >> 1, kp = blockIdx.x & 1, tid = threadIdx.x;
    const int ntiles = __ldg(tile_off + E);
    const int4 ti = __ldg(tinfo + rt);  // beyond the used tiles it is never read past the check below
    if (rt >= ntiles) return;
    int t = -1;
    float wt = 0.0f;
    if (tid < 128) {
        if (tid < ti.z) {
            const int f = __ldg(perm + ti.y + tid);
            t = f / k;
            wt = __ldg(w + f);  // consumed only by the row table, written last
        }
        s_tok[tid] = t;
    }
    __syncthreads();
    const int KSN = H / 128, pieces = H / 32;  // per row: 16-byte code pieces
    const int64_t rowb = H / 2 + H / 16;
    uint8_t* tile = xq + (int64_t)rt * KSN * pf::BLK;
    // codes: lanes 8a .. 8a+7 take eight consecutive rows of one 16-byte piece, i.e. one whole
    // 128-byte line of the tile; thread t: row t & 7 of the eight row groups 8 ((t >> 3) & 1) .., and
    // a pair of adjacent pieces (one 32-byte sector of the source row, so the second load is served
    // by L1 and L2 sees one request per sector), pairs t >> 4, +16, ...  Four row groups are loaded
    // before any is stored (eight loads in flight, few enough registers for four blocks per SM; no
    // runtime division either: this copy is instruction-heavy).
    {
        const int r_lo = tid & 7, rgh = (tid >> 3) & 1, npair = H / 128;  // pairs of pieces in this half
        for (int pp = tid >> 4; pp < npair; pp += blockDim.x >> 4) {
            const int pc = kp * (pieces / 2) + 2 * pp;  // even: both pieces lie in one K block
            uint8_t* dst = tile + (pc >> 2) * pf::BLK + blk_code_off(r_lo, (pc & 3) * 16);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint4 v0[4], v1[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tk = s_tok[(rgh * 8 + hb * 4 + j) * 8 + r_lo];
                    if (tk >= 0) {
                        const uint4* src = reinterpret_cast<const uint4*>(xc + (int64_t)tk * rowb) + pc;
                        v0[j] = __ldg(src);
                        v1[j] = __ldg(src + 1);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int rg = rgh * 8 + hb * 4 + j;
                    if (s_tok[rg * 8 + r_lo] >= 0) {
                        *reinterpret_cast<uint4*>(dst + rg * 128) = v0[j];
                        *reinterpret_cast<uint4*>(dst + rg * 128 + 2048) = v1[j];
                    }
                }
            }
        }
    }
    // scale words: two threads per row (t >> 1), each loading its half of this half-row's H / 128
    // words as 16-byte pieces (4-byte words when H / 256 is not a multiple of four) and storing
    // every word where the tile layout puts it
    {
        const int r = tid >> 1, tk = s_tok[r], wpt = H / 256, w0 = kp * (H / 128) + (tid & 1) * wpt;
        if (tk >= 0) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(xc + (int64_t)tk * rowb + H / 2) + w0;
            if ((wpt & 3) == 0) {
                for (int c = 0; c < wpt; c += 4) {
                    const uint4 q = __ldg(reinterpret_cast<const uint4*>(src + c));
                    const uint32_t ww[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int wd = w0 + c + u;
                        *reinterpret_cast<uint32_t*>(tile + (wd >> 1) * pf::BLK + blk_scale_off(r, (wd & 1) * 4)) = ww[u];
                    }
                }
            } else {
                for (int c = 0; c < wpt; ++c) {
                    const int wd = w0 + c;
                    *reinterpret_cast<uint32_t*>(tile + (wd >> 1) * pf::BLK + blk_scale_off(r, (wd & 1) * 4)) = __ldg(src + c);
                }
            }
        }
    }
    if (kp == 0 && tid < 128) rowmeta[(int64_t)rt * 128 + tid] = make_int2(t, __float_as_int(wt));
}

// Each warp converts segments of 4 x 32 float4s (four coalesced loads in flight per lane, then four stores).
__global__ void __launch_bounds__(256) k_pf_out(const float4* __restrict__ out32, int64_t n4, uint2* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t nseg = (n4 + 127) / 128, wstep = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t sg = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; sg < nseg; sg += wstep) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t i = sg * 128 + j * 32 + lane;
            if (i < n4) v[j] = out32[i];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t i = sg * 128 + j * 32 + lane;
            if (i < n4)
                out[i] = make_uint2((uint32_t)bf16_bits(v[j].x) | ((uint32_t)bf16_bits(v[j].y) << 16),
                                    (uint32_t)bf16_bits(v[j].z) | ((uint32_t)bf16_bits(v[j].w) << 16));
        }
    }
}

// ---------------------------------------------------------------------------- epilogues

// The MMA puts the token tile on the M side, so TMEM lane r of the accumulator is
// token row r of the tile and its columns are the 128 weight rows of the m tile:
// a thread that loads 32 columns holds 32 consecutive weight rows of one token.

// SwiGLU + h quantisation.  Weight rows come as (gate, up) pairs, so the 32
// columns c0 .. c0+31 of a thread are the 16 h features m*64 + c0/2 .. +15 of its
// token: exactly one NVFP4 block, quantised without leaving the thread (the
// quantiser's codes with one reciprocal per block: quant_block16_bf16).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ void epi_swiglu(const PfGemmArgs& a, const uint32_t (&v)[32], int m, int ntg, int r, int c0,
                                           float tsg, float tsu) {
    float hb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float g = __uint_as_float(v[2 * i]) * tsg, u = __uint_as_float(v[2 * i + 1]) * tsu;
        hb[i] = bf16_to_f32(bf16_bits(silu_fast(g) * u));
    }
    uint2 cw;
    uint32_t sb;
    quant_block16_bf16(hb, cw, sb);  // hb is bf16-valued, unit tensor scale
    const uint32_t w[2] = {cw.x, cw.y};
    const int f0 = m * 64 + c0 / 2;  // first feature: block f0 / 128 of the h row, bytes (f0 % 128) / 2 ..
    uint8_t* blk = a.hq + ((int64_t)ntg * a.KSN2 + f0 / 128) * pf::BLK;
    *reinterpret_cast<uint2*>(blk + blk_code_off(r, (f0 & 127) / 2)) = make_uint2(w[0], w[1]);
    blk[blk_scale_off(r, (f0 & 127) / 16)] = (uint8_t)sb;
}

// Down projection + combine: out32[t][m*128 + c0 .. +31] += w * tsd * y for the
// thread's token row (row table entry: token, routing weight; token -1 for
// padding), as eight 16-byte vector reductions.
// With a y output, the row's y = tsd * acc (no routing weight) also goes to y[prow][...].
__device__ __forceinline__ void epi_combine(const PfGemmArgs& a, const uint32_t (&v)[32], int2 meta, int prow, int m,
                                            int c0, float tsd) {
    if (meta.x < 0) return;
    if (a.y) {
        float4* yd = reinterpret_cast<float4*>(a.y + (int64_t)prow * a.H + m * 128 + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            yd[i] = make_float4(__uint_as_float(v[4 * i]) * tsd, __uint_as_float(v[4 * i + 1]) * tsd,
                                __uint_as_float(v[4 * i + 2]) * tsd, __uint_as_float(v[4 * i + 3]) * tsd);
    }
    if (!a.out32) return;
    const float wt = __int_as_float(meta.y) * tsd;
    float* dst = a.out32 + (int64_t)meta.x * a.H + m * 128 + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * i),
                     "f"(__uint_as_float(v[4 * i]) * wt), "f"(__uint_as_float(v[4 * i + 1]) * wt),
                     "f"(__uint_as_float(v[4 * i + 2]) * wt), "f"(__uint_as_float(v[4 * i + 3]) * wt)
                     : "memory");
}

// The same combine with coalesced reductions.  A thread holds 32 columns of one token row, so the warp's direct
// reductions touch 32 rows with 16 bytes each.  Here the warp's 32 rows x 32 columns, already scaled by each
// row's w * tsd, pass through a per-warp shared-memory block (32 rows, row stride LD floats) in 32 / CW passes of
// CW columns; read back with CW / 4 lanes per row, each reduction instruction covers 4 CW contiguous bytes of
// 128 / CW output rows (whole 128-byte lines for CW = 32).  Row strides 36 (CW = 32) and 20 (CW = 16) floats:
// both the row-wise writes and the column-wise reads take the minimum of four shared-memory wavefronts per
// 512 bytes.
namespace pf {
template <int CW>
__host__ __device__ constexpr int cst_ld() { return CW == 32 ? 36 : 20; }
template <int CW>
__host__ __device__ constexpr size_t cst_bytes() { return (size_t)EPI_WARPS * 32 * cst_ld<CW>() * 4; }  // 72 KB (CW 32), 40 KB (CW 16)
}  // namespace pf

template <int CW>
__device__ __forceinline__ void epi_combine_staged(const PfGemmArgs& a, const uint32_t (&v)[32], int2 meta, int m,
                                                   int c0, float tsd, float* st, int lane) {
    constexpr int LD = pf::cst_ld<CW>(), LPR = CW / 4, RPI = 32 / LPR;  // lanes per row, rows per instruction
    const float wt = meta.x < 0 ? 0.0f : __int_as_float(meta.y) * tsd;
#pragma unroll
    for (int hh = 0; hh < 32 / CW; ++hh) {
#pragma unroll
        for (int q = 0; q < CW / 4; ++q)
            *reinterpret_cast<float4*>(st + lane * LD + 4 * q) =
                make_float4(__uint_as_float(v[CW * hh + 4 * q]) * wt, __uint_as_float(v[CW * hh + 4 * q + 1]) * wt,
                            __uint_as_float(v[CW * hh + 4 * q + 2]) * wt, __uint_as_float(v[CW * hh + 4 * q + 3]) * wt);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32 / RPI; ++i) {
            const int row = RPI * i + lane / LPR, cq = lane % LPR;
            const int tok = __shfl_sync(0xffffffffu, meta.x, row);
            const float4 val = *reinterpret_cast<const float4*>(st + row * LD + 4 * cq);
            if (tok >= 0)
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(
                                 a.out32 + (int64_t)tok * a.H + m * 128 + c0 + CW * hh + 4 * cq),
                             "f"(val.x), "f"(val.y), "f"(val.z), "f"(val.w)
                             : "memory");
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------- grouped GEMM

template <int EPI>
__global__ void __launch_bounds__(pf::THREADS, 1) k_pf_gemm_stream(const PfGemmArgs a) {
    extern __shared__ __align__(1024) uint8_t pf_smem[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_smem) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) unsigned long long full[pf::NS], empty[pf::NS], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < pf::NS; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&empty[s])));
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&acc_full[b])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pf_su(&acc_empty[b])), "n"(pf::EPI_WARPS));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_s = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(pf_su(&tmem_base)),
                     "n"(pf::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = tmem_base;
    const int n_items = a.MT * __ldg(a.tile_off + a.E);

    // decode item i -> (expert, m tile, global token tile)
    auto item = [&](int i, int& e, int& m, int& ntg) {
        const int v = i / a.MT;
        e = __ldg(a.tinfo + v).x;
        const int t0 = __ldg(a.tile_off + e), nt = __ldg(a.tile_off + e + 1) - t0;
        const int local = i - a.MT * t0;
        m = local / nt;
        ntg = t0 + (local - m * nt);
    };

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int sc = 0;
            for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x) {
                int e, m, ntg;
                item(i, e, m, ntg);
                const uint8_t* ab = a.A + pf_widx(a, e) * a.a_stride + (int64_t)m * a.KSN * pf::BLK;
                const uint8_t* bb = a.B + (int64_t)ntg * a.KSN * pf::BLK;
                // a tile's K blocks are contiguous: KPS of them (A, then B) per stage
                for (int ks = 0; ks < a.KSN; ks += pf::KPS, ++sc) {
                    const int s = sc % pf::NS, use = sc / pf::NS;
                    if (use > 0 && !pf_wait(&empty[s], (use - 1) & 1, abort_flag, a.wait_ns)) break;
                    uint8_t* dst = ring + (size_t)s * pf::STAGE;
                    const uint32_t bytes = (uint32_t)(min(pf::KPS, a.KSN - ks) * pf::BLK);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(pf_su(&full[s])),
                                 "r"(2 * bytes) : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            pf_su(dst)), "l"(ab + (int64_t)ks * pf::BLK), "r"(bytes), "r"(pf_su(&full[s]))
                        : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            pf_su(dst + pf::KPS * pf::BLK)), "l"(bb + (int64_t)ks * pf::BLK), "r"(bytes), "r"(pf_su(&full[s]))
                        : "memory");
                }
            }
            // do not leave copies landing after exit: wait (bounded) for the last stages issued
            const unsigned long long t0 = pf_gt();
            for (int n = max(0, sc - pf::NS); n < sc; ++n)
                while (!pf_try_wait(&full[n % pf::NS], (n / pf::NS) & 1) && pf_gt() - t0 < pf::WAIT_NS) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int sc = 0, it = 0;
            for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x, ++it) {
                const int buf = it & 1, useb = it >> 1;
                if (useb > 0 && !pf_wait(&acc_empty[buf], (useb - 1) & 1, abort_flag, a.wait_ns)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dcol = tbase + (uint32_t)(buf * 128);
                for (int ks = 0; ks < a.KSN; ks += pf::KPS, ++sc) {
                    const int s = sc % pf::NS;
                    if (!pf_wait(&full[s], (sc / pf::NS) & 1, abort_flag, a.wait_ns)) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const int nkb = min(pf::KPS, a.KSN - ks);
                    for (int bi = 0; bi < nkb; ++bi) {
                        const uint8_t* sa = ring + (size_t)s * pf::STAGE + bi * pf::BLK;
                        const uint8_t* sbp = sa + pf::KPS * pf::BLK;
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            // M side: the token tile (ring B half); N side: the weight tile (A half)
                            const uint32_t tsfa = tbase + pf::SF_COL0 + (uint32_t)((s * pf::KPS + bi) * 16 + kb * 8), tsfb = tsfa + 4;
                            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsfa),
                                         "l"(umma_desc(sbp + 8192 + kb * 512, 0, 128)));
                            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsfb),
                                         "l"(umma_desc(sa + 8192 + kb * 512, 0, 128)));
                            const uint64_t da = umma_desc(sbp + kb * 4096, 2048, 128), db = umma_desc(sa + kb * 4096, 2048, 128);
                            const uint32_t acc = (ks | bi | kb) ? 1u : 0u;
                            asm volatile(
                                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                                    dcol), "l"(da), "l"(db), "r"(kIdesc), "r"(tsfa), "r"(tsfb), "r"(acc));
                        }
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     pf_su(&empty[s])) : "memory");
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 pf_su(&acc_full[buf])) : "memory");
            }
        }
    } else {
        // ---------------- epilogue warps 2..17: TMEM lane quadrant qd = warp % 4 (token rows
        // 32 qd .. +31), 32 columns (weight rows c0 .. +31) each
        const int qd = warp & 3, c0 = 32 * ((warp - 2) >> 2);
        const int r = 32 * qd + lane;
        int it = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++it) {
            const int buf = it & 1;
            // everything that does not depend on the accumulator is loaded before waiting for it
            int e, m, ntg;
            item(i, e, m, ntg);
            const float* ts = a.tscale + pf_widx(a, e) * a.ts_stride;
            const float t0s = __ldg(ts + 0), t1s = __ldg(ts + 1), t2s = __ldg(ts + 2);
            int2 meta = make_int2(-1, 0);
            int prow = -1;  // permuted row of this token row of the tile (y output)
            if (EPI == 2) {
                meta = __ldg(a.rowmeta + (int64_t)ntg * 128 + r);
                if (a.y) prow = __ldg(a.tinfo + ntg).y + r;
            }
            if (!pf_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, a.wait_ns)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // the accumulator is in registers once the load has completed: hand the TMEM columns back to
            // the MMA before the epilogue's math and stores
            uint32_t v[32];
            tmem_ld32(tbase + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * 128 + c0), v);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pf_su(&acc_empty[buf])) : "memory");
            if (EPI == 1) epi_swiglu(a, v, m, ntg, r, c0, t0s, t1s);
            else epi_combine(a, v, meta, prow, m, c0, t2s);
        }
    }
    // all MMAs have completed once the epilogue has consumed every accumulator; on an abort
    // wait (bounded) for the last commit before the TMEM is released
    if (warp == 1 && lane == 0 && *abort_flag) {
        const unsigned long long t0 = pf_gt();
        int it = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) ++it;
        if (it > 0)
            while (!pf_try_wait(&acc_full[(it - 1) & 1], ((it - 1) >> 1) & 1) && pf_gt() - t0 < pf::WAIT_NS) {
            }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(pf::TMEM_COLS));
    }
}

// Resident-token-tile variant (K <= 2048): a work item is (token tile, a part of
// the weight row tiles: all of them for gate/up, half for down).  The token tile's K blocks are copied once into shared
// memory and stay there (scale factors copied once into TMEM) while the item's
// weight tiles stream through the ring, KPS blocks per stage: half as many bulk
// copies per token tile as streaming both operands.
// The item's token tile and weight-tile range; its expert (tinfo[ntg].x) is loaded only by the roles that need it,
// so the MMA issuer's per-item work has no global load.
__device__ __forceinline__ bool pf_res_item(const PfGemmArgs& a, int i, int& ntg, int& mlo, int& mhi) {
    ntg = i / a.parts;
    const int part = i - ntg * a.parts, per = (a.MT + a.parts - 1) / a.parts;
    mlo = part * per;
    mhi = min(a.MT, mlo + per);
    return mlo < mhi;
}

template <int EPI>
__global__ void __launch_bounds__(pf::THREADS, 1) k_pf_gemm_res(const PfGemmArgs a) {
    extern __shared__ __align__(1024) uint8_t pf_smem[];
    uint8_t* btile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_smem) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = btile + (size_t)a.tbufs * a.KSN * pf::BLK;  // after the token-tile buffer(s)
    float* cst = reinterpret_cast<float*>(ring + (size_t)a.nstages * pf::KPS * pf::BLK);  // combine staging (cstage)
    __shared__ __align__(8) unsigned long long full[pf::RES_MAXNS], empty[pf::RES_MAXNS], acc_full[2], acc_empty[2],
        bfull[2], bfree[2], never;  // per token-tile buffer; never: the wait-expiry test hook's barrier
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NSr = a.nstages;
    // TMEM columns: accumulators [0, 256), token-tile scale factors (8 per K block, per buffer), then the
    // weight scale factors of the ring stages (8 per K block of a stage)
    const int TB = a.tbufs;
    const uint32_t SFT0 = 256, SFW0 = 256 + 8 * (uint32_t)(a.KSN * TB);
    if (tid == 0) {
        for (int s = 0; s < NSr; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&empty[s])));
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&acc_full[b])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pf_su(&acc_empty[b])), "n"(pf::EPI_WARPS));
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&bfull[b])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&bfree[b])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pf_su(&never)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_s = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(pf_su(&tmem_base)),
                     "n"(pf::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = tmem_base;
    const int n_items = a.parts * __ldg(a.tile_off + a.E);
    const uint32_t tile_bytes = (uint32_t)a.KSN * pf::BLK;
    int bfree_commits = 0;  // MMA thread: token-tile releases committed

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int sc = 0, bi = 0;
            int ps = 0, puse = 0;  // ring slot of stage sc and how many times it was filled before (sc % NSr, sc / NSr)
            for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x) {
                int ntg, mlo, mhi;
                if (!pf_res_item(a, i, ntg, mlo, mhi)) continue;
                // the token tile into buffer bi % TB, once the MMAs of the item that last used that buffer are done
                const int tb = bi % TB, tuse = bi / TB;
                if (tuse > 0 && !pf_wait(&bfree[tb], (tuse - 1) & 1, abort_flag, a.wait_ns)) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(pf_su(&bfull[tb])),
                             "r"(tile_bytes) : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        pf_su(btile + (size_t)tb * tile_bytes)), "l"(a.B + (int64_t)ntg * a.KSN * pf::BLK), "r"(tile_bytes),
                    "r"(pf_su(&bfull[tb]))
                    : "memory");
                ++bi;
                const uint8_t* ae = a.A + pf_widx(a, __ldg(a.tinfo + ntg).x) * a.a_stride;
                bool stop = false;
                for (int m = mlo; m < mhi && !stop; ++m) {
                    // warm L2 with the item's next weight tile, or with the next item's token tile,
                    // while this one streams through the two or so stages shared memory leaves
                    if (m + 1 < mhi) {
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ae + (int64_t)(m + 1) * a.KSN * pf::BLK),
                                     "r"(tile_bytes) : "memory");
                    } else if (i + (int)gridDim.x < n_items) {
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                         a.B + (int64_t)((i + (int)gridDim.x) / a.parts) * a.KSN * pf::BLK),
                                     "r"(tile_bytes) : "memory");
                    }
                    for (int ks = 0; ks < a.KSN; ks += pf::KPS, ++sc) {
                        const int s = ps, use = puse;
                        if (use > 0 && !pf_wait(&empty[s], (use - 1) & 1, abort_flag, a.wait_ns)) {
                            stop = true;
                            break;
                        }
                        const uint32_t bytes = (uint32_t)(min(pf::KPS, a.KSN - ks) * pf::BLK);
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(pf_su(&full[s])),
                                     "r"(bytes) : "memory");
                        asm volatile(
                            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                pf_su(ring + (size_t)s * pf::KPS * pf::BLK)),
                            "l"(ae + ((int64_t)m * a.KSN + ks) * pf::BLK), "r"(bytes), "r"(pf_su(&full[s]))
                            : "memory");
                        if (++ps == NSr) {
                            ps = 0;
                            ++puse;
                        }
                    }
                }
                if (stop) break;
            }
            // do not leave copies landing after exit: wait (bounded) for the last ring stages and
            // the last token tile issued
            const unsigned long long t0 = pf_gt();
            for (int n = max(0, sc - NSr); n < sc; ++n)
                while (!pf_try_wait(&full[n % NSr], (n / NSr) & 1) && pf_gt() - t0 < pf::WAIT_NS) {
                }
            for (int n = max(0, bi - TB); n < bi; ++n)  // the last token tile of each buffer
                while (!pf_try_wait(&bfull[n % TB], (n / TB) & 1) && pf_gt() - t0 < pf::WAIT_NS) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the token tile is the M side, the weight tile the N side
        if (lane == 0) {
            int sc = 0, it = 0, bi = 0;
            int ms = 0;
            uint32_t mph = 0;  // ring slot and phase parity of stage sc (sc % NSr, (sc / NSr) & 1)
            bool stop = false;
            const uint64_t dW0 = umma_desc(ring, 2048, 128), sW0 = umma_desc(ring + 8192, 0, 128);
            const uint64_t dTb = umma_desc(btile, 2048, 128), sTb = umma_desc(btile + 8192, 0, 128);
            for (int i = blockIdx.x; i < n_items && !stop && !*abort_flag; i += gridDim.x) {
                int ntg, mlo, mhi;
                if (!pf_res_item(a, i, ntg, mlo, mhi)) continue;
                // under the wait-expiry test hook the gate/up GEMM first waits on a barrier that nothing
                // completes: the bound runs out and every role winds down
                if (EPI == 1 && a.wait_site == FT_WAIT_SITE_PREFILL_TOKEN && !pf_wait(&never, 0, abort_flag, a.wait_ns))
                    break;
                const int tb = bi % TB;
                if (!pf_wait(&bfull[tb], (bi / TB) & 1, abort_flag, a.wait_ns)) break;
                const uint64_t dT0 = dTb + (uint64_t)tb * (tile_bytes >> 4), sT0 = sTb + (uint64_t)tb * (tile_bytes >> 4);
                const uint32_t SFTb = SFT0 + (uint32_t)(tb * 8 * a.KSN);
                ++bi;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int ks = 0; ks < a.KSN; ++ks) {
                    sf_copy(tbase + SFTb + (uint32_t)(ks * 8), sT0 + (uint64_t)ks * kDescBlk);
                    sf_copy(tbase + SFTb + (uint32_t)(ks * 8 + 4), sT0 + (uint64_t)ks * kDescBlk + kDescSfHalf);
                }
                for (int m = mlo; m < mhi && !stop; ++m, ++it) {
                    const int buf = it & 1, useb = it >> 1;
                    if (useb > 0 && !pf_wait(&acc_empty[buf], (useb - 1) & 1, abort_flag, a.wait_ns)) {
                        stop = true;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t dcol = tbase + (uint32_t)(buf * 128);
                    for (int ks = 0; ks < a.KSN; ks += pf::KPS, ++sc) {
                        const int s = ms;
                        if (!pf_wait(&full[s], mph, abort_flag, a.wait_ns)) {
                            stop = true;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        // A single thread issues every MMA, so its instruction count between MMAs
                        // sets their rate: descriptors advance by constant offsets, the loops unroll,
                        // and the stage's scale-factor copies go first.
                        const int nkb = min(pf::KPS, a.KSN - ks);
                        const uint64_t dW = dW0 + (uint64_t)(s * pf::KPS) * kDescBlk, sW = sW0 + (uint64_t)(s * pf::KPS) * kDescBlk;
                        const uint64_t dT = dT0 + (uint64_t)ks * kDescBlk;
                        const uint32_t cW = tbase + SFW0 + (uint32_t)(s * pf::KPS * 8), cT = tbase + SFTb + (uint32_t)(ks * 8);
                        if (nkb == pf::KPS) {  // a full stage: no per-block predicates
#pragma unroll
                            for (int bq = 0; bq < pf::KPS; ++bq) {
                                sf_copy(cW + bq * 8, sW + bq * kDescBlk);
                                sf_copy(cW + bq * 8 + 4, sW + bq * kDescBlk + kDescSfHalf);
                            }
#pragma unroll
                            for (int bq = 0; bq < pf::KPS; ++bq)
#pragma unroll
                                for (int kb = 0; kb < 2; ++kb)
                                    mma_fp4(dcol, dT + bq * kDescBlk + kb * kDescHalf, dW + bq * kDescBlk + kb * kDescHalf,
                                            cT + bq * 8 + kb * 4, cW + bq * 8 + kb * 4, (ks | bq | kb) ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int bq = 0; bq < pf::KPS; ++bq)
                                if (bq < nkb) {
                                    sf_copy(cW + bq * 8, sW + bq * kDescBlk);
                                    sf_copy(cW + bq * 8 + 4, sW + bq * kDescBlk + kDescSfHalf);
                                }
#pragma unroll
                            for (int bq = 0; bq < pf::KPS; ++bq)
                                if (bq < nkb) {
#pragma unroll
                                    for (int kb = 0; kb < 2; ++kb)
                                        mma_fp4(dcol, dT + bq * kDescBlk + kb * kDescHalf,
                                                dW + bq * kDescBlk + kb * kDescHalf, cT + bq * 8 + kb * 4,
                                                cW + bq * 8 + kb * 4, (ks | bq | kb) ? 1u : 0u);
                                }
                        }
                        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                         pf_su(&empty[s])) : "memory");
                        if (++ms == NSr) {
                            ms = 0;
                            mph ^= 1u;
                        }
                    }
                    if (stop) break;
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     pf_su(&acc_full[buf])) : "memory");
                }
                // the token tile may be replaced once this item's MMAs are done
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 pf_su(&bfree[tb])) : "memory");
                ++bfree_commits;
            }
        }
    } else {
        // ---------------- epilogue warps 2..17: TMEM lane quadrant qd = warp % 4 (token rows
        // 32 qd .. +31), 32 columns (weight rows c0 .. +31) each
        const int qd = warp & 3, c0 = 32 * ((warp - 2) >> 2);
        const int r = 32 * qd + lane;
        int it = 0;
        bool stop = false;
        for (int i = blockIdx.x; i < n_items && !stop; i += gridDim.x) {
            int ntg, mlo, mhi;
            if (!pf_res_item(a, i, ntg, mlo, mhi)) continue;
            const float* ts = a.tscale + pf_widx(a, __ldg(a.tinfo + ntg).x) * a.ts_stride;
            const float t0s = __ldg(ts + 0), t1s = __ldg(ts + 1), t2s = __ldg(ts + 2);
            int2 meta = make_int2(-1, 0);
            int prow = -1;  // permuted row of this token row of the tile (y output)
            if (EPI == 2) {
                meta = __ldg(a.rowmeta + (int64_t)ntg * 128 + r);
                if (a.y) prow = __ldg(a.tinfo + ntg).y + r;
            }
            for (int m = mlo; m < mhi; ++m, ++it) {
                const int buf = it & 1;
                if (!pf_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, a.wait_ns)) {
                    stop = true;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // the accumulator is in registers once the load has completed: hand the TMEM columns back to
                // the MMA before the epilogue's math and stores
                uint32_t v[32];
                tmem_ld32(tbase + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * 128 + c0), v);
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pf_su(&acc_empty[buf])) : "memory");
                if (EPI == 1) epi_swiglu(a, v, m, ntg, r, c0, t0s, t1s);
                else {
                    if (a.y) epi_combine(a, v, meta, prow, m, c0, t2s);  // y rows (and the combine, unstaged)
                    else if (a.cstage == 32)
                        epi_combine_staged<32>(a, v, meta, m, c0, t2s, cst + (warp - 2) * 32 * pf::cst_ld<32>(), lane);
                    else if (a.cstage == 16)
                        epi_combine_staged<16>(a, v, meta, m, c0, t2s, cst + (warp - 2) * 32 * pf::cst_ld<16>(), lane);
                    else epi_combine(a, v, meta, prow, m, c0, t2s);
                }
            }
        }
    }
    // all MMAs have completed once the epilogue has consumed every accumulator; on an abort
    // wait (bounded) for the last commit before the TMEM is released
    if (warp == 1 && lane == 0 && *abort_flag && bfree_commits > 0) {
        const int lb = (bfree_commits - 1) % TB;
        // the last commit covers every MMA issued before it
        const unsigned long long t0 = pf_gt();
        while (!pf_try_wait(&bfree[lb], ((bfree_commits - 1) / TB) & 1) && pf_gt() - t0 < pf::WAIT_NS) {
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(pf::TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------- weight packing

// [N][K] row-major codes/scales -> UMMA tiles (N, K multiples of 128).
__global__ void __launch_bounds__(256) k_pack_umma(const uint8_t* __restrict__ codes, int64_t codes_ld,
                                                   const uint8_t* __restrict__ scales, int64_t scales_ld, int64_t N,
                                                   int64_t K, uint8_t* __restrict__ out) {
    const int64_t KSN = K / 128;
    const int64_t per_row = 4 + 1;  // four 16-byte code pieces and one 8-byte scale group per 128 K
    const int64_t total = N * KSN * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / (KSN * per_row);
        const int64_t rem = i % (KSN * per_row);
        const int64_t ks = rem / per_row;
        const int piece = (int)(rem % per_row);
        uint8_t* blk = out + ((row / 128) * KSN + ks) * pf::BLK;
        const int r = (int)(row % 128);
        if (piece < 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(codes + row * codes_ld + ks * 64 + piece * 16);
            *reinterpret_cast<uint4*>(blk + blk_code_off(r, piece * 16)) = v;
        } else {
            const uint8_t* s = scales + row * scales_ld + ks * 8;
            for (int j = 0; j < 8; ++j) blk[blk_scale_off(r, j)] = s[j];
        }
    }
}

// ---------------------------------------------------------------------------- host side

static int pf_sm_count() {
    static int cached = 0;
    if (!cached) {
        int dev = 0, n = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached = n > 0 ? n : 148;
    }
    return cached;
}

static size_t a256(size_t v) { return (v + 255) / 256 * 256; }

struct PfWs {
    size_t tile_off, tinfo, xc, xq, hq, rowmeta, out32, total;
    int max_tiles;
};

static PfWs pf_ws_layout(int T, int k, int E, int H, int I) {
    PfWs w;
    const int64_t P = (int64_t)T * k;
    w.max_tiles = (int)((P + 127) / 128 + std::min<int64_t>(E, P));
    size_t off = 0;
    w.tile_off = off;
    off += a256((size_t)(E + 1) * 4);
    w.tinfo = off;
    off += a256((size_t)w.max_tiles * 16);
    w.xc = off;
    off += a256((size_t)T * (H / 2 + H / 16));
    w.xq = off;
    off += a256((size_t)w.max_tiles * (H / 128) * pf::BLK);
    w.rowmeta = off;
    off += a256((size_t)w.max_tiles * 128 * 8);
    w.hq = off;
    off += a256((size_t)w.max_tiles * (I / 128) * pf::BLK);
    w.out32 = off;
    off += a256((size_t)T * H * 4);
    w.total = off;
    return w;
}

ft_status validate_weights(const ft_moe_layer_weights* W, const char* fn);

// Resident token tile when it fits with a ring of at least two stages (shared memory) and the
// scale factors fit TMEM; otherwise both operands stream through the ring.
template <int EPI>
static void launch_pf_gemm(PfGemmArgs g, int G, cudaStream_t s) {
    const size_t tile = (size_t)g.KSN * pf::BLK, stage = (size_t)pf::KPS * pf::BLK;
    int ns = 0;
    size_t extra = 0;
    g.cstage = 0;
    g.tbufs = 1;
    if (g.KSN <= pf::RES_MAXKSN && tile + 1024 < pf::SMEM_LIMIT) {
        // the down GEMM's combine (without y rows) goes through shared memory when two stages still fit beside it
        if (EPI == 2 && g.out32 && !g.y) {
            for (int cw : {32, 16}) {
                const size_t b = cw == 32 ? pf::cst_bytes<32>() : pf::cst_bytes<16>();
                if (tile + 2 * stage + b + 1024 <= pf::SMEM_LIMIT) {
                    g.cstage = cw;
                    extra = b;
                    break;
                }
            }
        }
        // a second token-tile buffer when two stages still fit beside it: the next item's tile loads while this
        // item's MMAs run
        if (EPI == 2 && 2 * tile + 2 * stage + extra + 1024 <= pf::SMEM_LIMIT &&
            256 + 16 * (uint32_t)g.KSN + 2 * 8 * pf::KPS <= pf::TMEM_COLS)
            g.tbufs = 2;
        const int by_tmem = (int)((pf::TMEM_COLS - 256 - 8 * (uint32_t)(g.KSN * g.tbufs)) / (8 * pf::KPS));
        const int by_smem = (int)((pf::SMEM_LIMIT - 1024 - tile * g.tbufs - extra) / stage);
        ns = std::min({by_smem, by_tmem, pf::RES_MAXNS});
    }
    if (ns >= 2) {
        g.nstages = ns;
        g.parts = EPI == 1 ? 1 : 2;  // measured: whole token tiles for gate/up (one token-tile load each), halves for down
        k_pf_gemm_res<EPI><<<G, pf::THREADS, tile * g.tbufs + (size_t)ns * stage + extra + 1024, s>>>(g);
    } else {
        g.cstage = 0;
        k_pf_gemm_stream<EPI><<<G, pf::THREADS, pf::SMEM, s>>>(g);
    }
}

}  // namespace ft

using namespace ft;

extern "C" {

ft_status ft_nvfp4_pack_umma(const uint8_t* codes, int64_t codes_ld, const uint8_t* scales, int64_t scales_ld,
                             int64_t N, int64_t K, uint8_t* tiles, ft_stream_t stream) {
    if (N <= 0 || K <= 0 || N % 128 || K % 128)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_umma: need N and K multiples of 128");
    if (!codes || !scales || !tiles) return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_umma: null pointer");
    if (!aligned(codes, 16) || codes_ld % 16 || !aligned(tiles, 16) || codes_ld < K / 2 || scales_ld < K / 16)
        return fail(FT_ERR_INVALID_ARG, "ft_nvfp4_pack_umma: codes/tiles need 16-byte alignment and row strides");
    const int64_t total = N * (K / 128) * 5;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 64);
    k_pack_umma<<<(unsigned)blocks, 256, 0, cu(stream)>>>(codes, codes_ld, scales, scales_ld, N, K, tiles);
    return check_launch("ft_nvfp4_pack_umma");
}

size_t ft_moe_prefill_workspace_size(int T, int k, int E, int H, int I) {
    if (T <= 0 || k <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
    return pf_ws_layout(T, k, E, H, I).total;
}

ft_status ft_moe_expert_ffn_nvfp4_prefill(const ft_moe_layer_weights* W, const uint16_t* x, int T, int k,
                                          const int32_t* offsets, const int32_t* perm, const float* w, float* y,
                                          uint16_t* out, void* ws, size_t ws_bytes, ft_stream_t stream) {
    const char* fn = "ft_moe_expert_ffn_nvfp4_prefill";
    ft_status st = validate_weights(W, fn);
    if (st != FT_OK) return st;
    if (W->layout != FT_LAYOUT_UMMA_TILES)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": weights must use FT_LAYOUT_UMMA_TILES");
    if (W->H % 128 || W->I % 64 || (2 * W->I) % 128)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need H a multiple of 128 and I of 64");
    if (W->I % 128) return fail(FT_ERR_UNSUPPORTED, std::string(fn) + ": I must be a multiple of 128");
    if (T < 0 || k <= 0 || k > W->E || k > 32) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need T >= 0, 1 <= k <= min(E, 32)");
    if (T == 0) return FT_OK;
    if ((int64_t)T * k > INT32_MAX) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": T*k must fit in int32");
    if (!x || !offsets || !perm || (out && !w)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (!y && !out) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need y or out");
    if (!aligned(x, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": x needs 16-byte alignment");
    if (out && !aligned(out, 8)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": out needs 8-byte alignment");
    if (y && !aligned(y, 16)) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": y needs 16-byte alignment");
    const int E = W->E, H = W->H, I = W->I;
    const PfWs L = pf_ws_layout(T, k, E, H, I);
    if (!ws || ws_bytes < L.total || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": workspace missing, too small or not 256-byte aligned");
    uint8_t* base = static_cast<uint8_t*>(ws);
    int32_t* tile_off = reinterpret_cast<int32_t*>(base + L.tile_off);
    int4* tinfo = reinterpret_cast<int4*>(base + L.tinfo);
    uint8_t* xq = base + L.xq;
    uint8_t* xc = base + L.xc;
    int2* rowmeta = reinterpret_cast<int2*>(base + L.rowmeta);
    uint8_t* hq = base + L.hq;
    float* out32 = reinterpret_cast<float*>(base + L.out32);
    cudaStream_t s = cu(stream);
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(k_pf_gemm_stream<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pf::SMEM);
        cudaFuncSetAttribute(k_pf_gemm_stream<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pf::SMEM);
        cudaFuncSetAttribute(k_pf_gemm_res<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pf::SMEM_LIMIT);
        cudaFuncSetAttribute(k_pf_gemm_res<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pf::SMEM_LIMIT);
    });
    k_pf_plan<<<1, 1024, 0, s>>>(offsets, E, (int)((int64_t)T * k), L.max_tiles, W->expert_to_slot, W->n_weights,
                                  tile_off, tinfo);
    {
        const int64_t warps = (int64_t)T * ((H + 1023) / 1024);
        k_pf_quant_tokens<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(x, T, H, xc);
    }
    k_pf_gather_x<<<(unsigned)(2 * L.max_tiles), 256, 0, s>>>(xc, H, k, E, perm, w, tile_off, tinfo, xq, rowmeta,
                                                               reinterpret_cast<float4*>(out32), (int64_t)T * H / 4);
    PfGemmArgs g{};
    g.tscale = W->tscale;
    g.ts_stride = W->tscale_stride;
    g.E = E;
    g.offsets = offsets;
    g.tile_off = tile_off;
    g.hq = hq;
    g.KSN2 = I / 128;
    g.rowmeta = rowmeta;
    g.out32 = out ? out32 : nullptr;
    g.H = H;
    g.e2s = W->expert_to_slot;
    g.tinfo = tinfo;
    g.y = y;
    g.wait_ns = wait_hook_ns();
    g.wait_site = wait_hook_site();
    const int G = pf_sm_count();
    // gate/up + SwiGLU
    g.A = W->gu_codes;
    g.a_stride = W->gu_codes_stride;
    g.B = xq;
    g.MT = 2 * I / 128;
    g.KSN = H / 128;
    launch_pf_gemm<1>(g, G, s);
    // down + combine
    g.A = W->d_codes;
    g.a_stride = W->d_codes_stride;
    g.B = hq;
    g.MT = H / 128;
    g.KSN = I / 128;
    launch_pf_gemm<2>(g, G, s);
    if (!out) return check_launch(fn);
    const int64_t n4 = (int64_t)T * H / 4;  // H is a multiple of 128
    k_pf_out<<<(unsigned)std::min<int64_t>((n4 + 1023) / 1024, 148 * 8), 256, 0, s>>>(
        reinterpret_cast<const float4*>(out32), n4, reinterpret_cast<uint2*>(out));
    return check_launch(fn);
}

}  // extern "C"
