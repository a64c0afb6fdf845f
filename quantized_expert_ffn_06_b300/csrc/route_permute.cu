// route_permute.cu -- router top-k (warp per token), the stable expert
// permutation, and the routing-weighted combine.
//
// Router: page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", MoE core
// mechanism: linear + softmax gives per-expert probabilities, the top-K
// experts are taken and their outputs weighted.  Selection is on the fp32
// logits (softmax is monotone), equal logits go to the lower expert id, and
// the selected probabilities are renormalised to sum to 1.
// Permutation: page xxmr.cn/news/175150 §2.2 -- tokens are dispatched to the
// few selected experts; here a stable counting sort by expert id.
#include "common.cuh"

#include <algorithm>
#include <cfloat>
#include <climits>
#include <mutex>

namespace ft {

// ----------------------------------------------------------------------------
// route
// ----------------------------------------------------------------------------

// One warp per token.  Each lane holds logits e = lane + 32*i; k rounds of a
// warp arg-max on (value, lower index wins) pick the experts in order.
template <int EPL>
__global__ void __launch_bounds__(256) k_route(const float* __restrict__ logits, int T, int E, int k,
                                               int32_t* __restrict__ ids, float* __restrict__ w) {
    const int t = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* row = logits + (int64_t)t * E;
    float v[EPL];
    bool live[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        live[i] = e < E;
        v[i] = live[i] ? row[e] : -INFINITY;
        if (live[i] && (v[i] != v[i] || v[i] == INFINITY)) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_dev_error(FT_DEVERR_NAN_LOGIT);

    float my_val = -INFINITY;
    int my_id = -1;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (live[i] && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi != INT_MAX && (bi & 31) == lane) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == (bi >> 5)) live[i] = false;
        }
        if (lane == j) {
            my_val = bv;
            my_id = bi;
        }
    }
    const float m = __shfl_sync(0xffffffffu, my_val, 0);
    float wj;
    if (m == -INFINITY) {
        wj = 1.0f / (float)k;
    } else {
        const float ej = (lane < k) ? expf(my_val - m) : 0.0f;
        const float s = warp_sum(ej);
        wj = ej / s;
    }
    if (lane < k) {
        ids[(int64_t)t * k + lane] = my_id;
        w[(int64_t)t * k + lane] = wj;
    }
}

// E <= 256: the selection of select_topk8 (each lane's eight keys sorted once,
// then k rounds of two warp reductions over the lanes' heads); same experts, same
// order and the same weights as k_route.
__global__ void __launch_bounds__(256) k_route_sorted(const float* __restrict__ logits, int T, int E, int k,
                                                      int32_t* __restrict__ ids, float* __restrict__ w) {
    const int t = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* row = logits + (int64_t)t * E;
    bool bad = false;
    const int my_id = select_topk8(row, E, k, bad);
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_dev_error(FT_DEVERR_NAN_LOGIT);
    const float my_val = (lane < k) ? __ldg(row + my_id) : -INFINITY;
    const float m = __shfl_sync(0xffffffffu, my_val, 0);
    float wj;
    if (m == -INFINITY || m != m) {
        wj = 1.0f / (float)k;
    } else {
        const float ej = (lane < k) ? expf(my_val - m) : 0.0f;
        const float s = warp_sum(ej);
        wj = ej / s;
    }
    if (lane < k) {
        ids[(int64_t)t * k + lane] = my_id;
        w[(int64_t)t * k + lane] = wj;
    }
}

// ----------------------------------------------------------------------------
// permute: stable counting sort of f = t*k + j by ids[f]
// ----------------------------------------------------------------------------

constexpr int kPermChunk = 1024;  // slots per block

// Block-wide exclusive scan of cnt[0..E) in shared memory (E <= 1024), in place;
// returns the total.  Deterministic.
__device__ int block_exclusive_scan(int* cnt, int E, int* warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x;
    int v = (tid < E) ? cnt[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int nw = nthreads / 32;
        int s = (lane < nw) ? warp_tot[lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        if (lane < nw) warp_tot[lane] = si - s;  // exclusive warp base
        if (lane == nw - 1) warp_tot[32] = si;   // total
    }
    __syncthreads();
    if (tid < E) cnt[tid] = warp_tot[wid] + incl - v;
    const int total = warp_tot[32];
    __syncthreads();
    return total;
}

__device__ __forceinline__ int load_id(const int32_t* ids, int64_t f, int E) {
    const int e = ids[f];
    if (e < 0 || e >= E) {
        raise_dev_error(FT_DEVERR_BAD_INDEX);
        return -1;
    }
    return e;
}

// Rank of slot f among the earlier slots of the same expert within its chunk
// (brute force over the chunk held in shared memory; broadcast reads).
__device__ __forceinline__ int chunk_rank(const int* sid, int pos, int e) {
    int r = 0;
    for (int i = 0; i < pos; ++i) r += (sid[i] == e);
    return r;
}

// Single-block path (n <= kPermChunk): histogram, scan, stable placement.
__global__ void __launch_bounds__(1024) k_permute_small(const int32_t* __restrict__ ids, int n, int E,
                                                        int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                        int32_t* __restrict__ inv, int32_t* __restrict__ active) {
    __shared__ int cnt[1024];
    __shared__ int flag[1024];
    __shared__ int sid[kPermChunk];
    __shared__ int warp_tot[33];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int e_me = (tid < n) ? load_id(ids, tid, E) : -1;
    sid[tid] = e_me;
    if (e_me >= 0) atomicAdd(&cnt[e_me], 1);
    __syncthreads();
    const int has = (tid < E && cnt[tid] > 0) ? 1 : 0;
    if (tid < E) flag[tid] = has;
    block_exclusive_scan(cnt, E, warp_tot);  // cnt[e] <- first permuted row of expert e
    if (tid < E) offsets[tid] = cnt[tid];
    if (tid == 0) offsets[E] = n;
    if (active) {
        const int nact = block_exclusive_scan(flag, E, warp_tot);
        if (has) active[1 + flag[tid]] = tid;
        if (tid == 0) active[0] = nact;
    }
    if (e_me >= 0) {
        const int p = cnt[e_me] + chunk_rank(sid, tid, e_me);
        perm[p] = tid;
        inv[tid] = p;
    }
}

// Multi-block path: (A) per-chunk histograms, (B) scan into per-chunk bases,
// (C) stable placement within each chunk.
__global__ void __launch_bounds__(1024) k_permute_hist(const int32_t* __restrict__ ids, int n, int E,
                                                       int32_t* __restrict__ chunk_cnt) {
    __shared__ int cnt[1024];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int64_t f = (int64_t)blockIdx.x * kPermChunk + tid;
    if (f < n) {
        const int e = load_id(ids, f, E);
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) chunk_cnt[(int64_t)blockIdx.x * E + e] = cnt[e];
}

// One thread per expert: its chunk counts are loaded 32 at a time (independent loads, one round trip per 32
// chunks) and summed; after the block scan of the totals, the per-chunk bases are written once (from registers
// when there are at most 32 chunks, else from a second pass of loads).
__global__ void __launch_bounds__(1024) k_permute_scan(int32_t* __restrict__ chunk_cnt, int nchunks, int n, int E,
                                                       int32_t* __restrict__ offsets, int32_t* __restrict__ active) {
    constexpr int G = 32;
    __shared__ int tot[1024];
    __shared__ int flag[1024];
    __shared__ int warp_tot[33];
    const int tid = threadIdx.x;
    int has = 0;
    int v[G];
    if (tid < E) {
        int run = 0;
        for (int c0 = 0; c0 < nchunks; c0 += G) {
#pragma unroll
            for (int u = 0; u < G; ++u) v[u] = (c0 + u < nchunks) ? chunk_cnt[(int64_t)(c0 + u) * E + tid] : 0;
#pragma unroll
            for (int u = 0; u < G; ++u) run += v[u];
        }
        tot[tid] = run;
        has = run > 0;
        flag[tid] = has;
    }
    __syncthreads();
    block_exclusive_scan(tot, E, warp_tot);
    if (tid < E) {
        int base = tot[tid];
        offsets[tid] = base;
        if (nchunks <= G) {
#pragma unroll
            for (int u = 0; u < G; ++u)
                if (u < nchunks) {
                    chunk_cnt[(int64_t)u * E + tid] = base;
                    base += v[u];
                }
        } else {
            for (int c0 = 0; c0 < nchunks; c0 += G) {
#pragma unroll
                for (int u = 0; u < G; ++u) v[u] = (c0 + u < nchunks) ? chunk_cnt[(int64_t)(c0 + u) * E + tid] : 0;
#pragma unroll
                for (int u = 0; u < G; ++u)
                    if (c0 + u < nchunks) {
                        chunk_cnt[(int64_t)(c0 + u) * E + tid] = base;
                        base += v[u];
                    }
            }
        }
    }
    if (tid == 0) offsets[E] = n;
    if (active) {
        const int nact = block_exclusive_scan(flag, E, warp_tot);
        if (tid < E && has) active[1 + flag[tid]] = tid;
        if (tid == 0) active[0] = nact;
    }
}

// Rank of a slot within its chunk: lanes of a warp holding the same expert are
// ranked by __match_any_sync, and each warp's count per expert (leader lane) is
// scanned over the chunk's 32 warps in shared memory ([32][E] ints, dynamic).
__global__ void __launch_bounds__(1024) k_permute_place(const int32_t* __restrict__ ids, int n, int E,
                                                        const int32_t* __restrict__ chunk_base,
                                                        int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    extern __shared__ int wcnt[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    const int64_t f = (int64_t)blockIdx.x * kPermChunk + tid;
    int e = -1;
    if (f < n) {
        e = ids[f];
        if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    __syncthreads();
    if (e >= 0 && lrank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {  // exclusive scan over the warps
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) {
            const int v = wcnt[w * E + x];
            wcnt[w * E + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int p = chunk_base[(int64_t)blockIdx.x * E + e] + wcnt[warp * E + e] + lrank;
        perm[p] = (int32_t)f;
        inv[f] = p;
    }
}

// The scan and the placement in one kernel, for at most 32 chunks: every block reads all the chunk counts
// (one independent load per chunk and expert thread), forms the expert totals and its own chunk's bases, scans the
// totals over the experts, and places its chunk as k_permute_place does.  Block 0 also writes offsets and the
// active list.  The same arithmetic as k_permute_scan followed by k_permute_place, without the launch between.
constexpr int kPermFusedMaxChunks = 32;

__global__ void __launch_bounds__(1024) k_permute_scan_place(const int32_t* __restrict__ ids, int n, int E,
                                                             const int32_t* __restrict__ chunk_cnt, int nchunks,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ active, int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv) {
    extern __shared__ int wcnt[];
    __shared__ int tot[1024];
    __shared__ int flag[1024];
    __shared__ int cbase[1024];
    __shared__ int warp_tot[33];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x;
    int base = 0, total = 0;
    if (tid < E) {
#pragma unroll
        for (int c = 0; c < kPermFusedMaxChunks; ++c)
            if (c < nchunks) {
                const int v = __ldg(chunk_cnt + (int64_t)c * E + tid);
                total += v;
                if (c < b) base += v;
            }
        tot[tid] = total;
        flag[tid] = total > 0;
    }
    for (int i = tid; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    const int64_t f = (int64_t)b * kPermChunk + tid;
    int e = -1;
    if (f < n) {
        e = ids[f];
        if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    __syncthreads();
    block_exclusive_scan(tot, E, warp_tot);  // tot[e] <- first permuted row of expert e
    if (tid < E) cbase[tid] = tot[tid] + base;
    if (b == 0) {
        if (tid < E) offsets[tid] = tot[tid];
        if (tid == 0) offsets[E] = n;
        if (active) {
            const int nact = block_exclusive_scan(flag, E, warp_tot);
            if (tid < E && total > 0) active[1 + flag[tid]] = tid;
            if (tid == 0) active[0] = nact;
        }
    }
    if (e >= 0 && lrank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {  // exclusive scan over the warps
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) {
            const int v = wcnt[w * E + x];
            wcnt[w * E + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int p = cbase[e] + wcnt[warp * E + e] + lrank;
        perm[p] = (int32_t)f;
        inv[f] = p;
    }
}

// ----------------------------------------------------------------------------
// combine
// ----------------------------------------------------------------------------

// out[t][n] = bf16(sum_j w[t][j] * y[inv[t*k+j]][n]); 4 columns per thread.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y, const int32_t* __restrict__ inv,
                                                 const float* __restrict__ w, int T, int k, int H,
                                                 uint16_t* __restrict__ out) {
    const int t = blockIdx.x;  // tokens on x: its limit is 2^31 - 1, y's only 65535
    const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (t >= T || n >= H) return;
    const int64_t P = (int64_t)T * k;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const float wj = w[(int64_t)t * k + j];
        const int p = inv[(int64_t)t * k + j];
        if (p < 0 || p >= P) {  // not a row of y: reported, contributes nothing
            if (n == 0) raise_dev_error(FT_DEVERR_BAD_INDEX);
            continue;
        }
        const float4 v = *reinterpret_cast<const float4*>(y + (int64_t)p * H + n);
        acc.x = fmaf(wj, v.x, acc.x);
        acc.y = fmaf(wj, v.y, acc.y);
        acc.z = fmaf(wj, v.z, acc.z);
        acc.w = fmaf(wj, v.w, acc.w);
    }
    uint2 o;
    o.x = (uint32_t)bf16_bits(acc.x) | ((uint32_t)bf16_bits(acc.y) << 16);
    o.y = (uint32_t)bf16_bits(acc.z) | ((uint32_t)bf16_bits(acc.w) << 16);
    *reinterpret_cast<uint2*>(out + (int64_t)t * H + n) = o;
}

}  // namespace ft

using namespace ft;

extern "C" {

ft_status ft_moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, ft_stream_t stream) {
    if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > E || k > 32)
        return fail(FT_ERR_INVALID_ARG, "ft_moe_route: need T >= 0, 1 <= k <= min(E, 32), E <= 1024");
    if (T == 0) return FT_OK;
    if (!logits || !ids || !w) return fail(FT_ERR_INVALID_ARG, "ft_moe_route: null pointer");
    const int threads = 256, per_block = threads / 32;
    const dim3 grid((T + per_block - 1) / per_block);
    const int epl = (E + 31) / 32;
    cudaStream_t s = cu(stream);
    if (epl <= 1) k_route<1><<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (epl <= 2) k_route<2><<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (epl <= 4) k_route<4><<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (epl <= 8) k_route_sorted<<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (epl <= 16) k_route<16><<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    else k_route<32><<<grid, threads, 0, s>>>(logits, T, E, k, ids, w);
    return check_launch("ft_moe_route");
}

size_t ft_moe_permute_workspace_size(int T, int E, int k) {
    if (T <= 0 || E <= 0 || k <= 0) return 0;
    const int64_t n = (int64_t)T * k;
    if (n <= kPermChunk) return 0;
    const int64_t nchunks = (n + kPermChunk - 1) / kPermChunk;
    return (size_t)(nchunks * E * sizeof(int32_t) + 255) / 256 * 256;
}

ft_status ft_moe_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* perm, int32_t* inv,
                         int32_t* active, void* ws, size_t ws_bytes, ft_stream_t stream) {
    if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > E)
        return fail(FT_ERR_INVALID_ARG, "ft_moe_permute: need T >= 0, 1 <= k <= E <= 1024");
    if (!offsets) return fail(FT_ERR_INVALID_ARG, "ft_moe_permute: offsets is null");
    const int64_t n64 = (int64_t)T * k;
    if (n64 > INT_MAX / 2) return fail(FT_ERR_INVALID_ARG, "ft_moe_permute: T*k too large");
    const int n = (int)n64;
    if (n > 0 && (!ids || !perm || !inv)) return fail(FT_ERR_INVALID_ARG, "ft_moe_permute: null pointer");
    cudaStream_t s = cu(stream);
    if (n <= kPermChunk) {
        k_permute_small<<<1, 1024, 0, s>>>(ids, n, E, offsets, perm, inv, active);
        return check_launch("ft_moe_permute");
    }
    const size_t need = ft_moe_permute_workspace_size(T, E, k);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(FT_ERR_INVALID_ARG, "ft_moe_permute: workspace missing, too small or not 256-byte aligned");
    const int nchunks = (n + kPermChunk - 1) / kPermChunk;
    int32_t* chunk_cnt = static_cast<int32_t*>(ws);
    k_permute_hist<<<nchunks, 1024, 0, s>>>(ids, n, E, chunk_cnt);
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(k_permute_place, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024 * 4);
        cudaFuncSetAttribute(k_permute_scan_place, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024 * 4);
    });
    if (nchunks <= kPermFusedMaxChunks) {
        k_permute_scan_place<<<nchunks, 1024, (size_t)32 * E * 4, s>>>(ids, n, E, chunk_cnt, nchunks, offsets, active,
                                                                       perm, inv);
    } else {
        k_permute_scan<<<1, 1024, 0, s>>>(chunk_cnt, nchunks, n, E, offsets, active);
        k_permute_place<<<nchunks, 1024, (size_t)32 * E * 4, s>>>(ids, n, E, chunk_cnt, perm, inv);
    }
    return check_launch("ft_moe_permute");
}

ft_status ft_moe_combine(const float* y, const int32_t* inv, const float* w, int T, int k, int H, uint16_t* out,
                         ft_stream_t stream) {
    if (T < 0 || k <= 0 || H <= 0 || H % 4)
        return fail(FT_ERR_INVALID_ARG, "ft_moe_combine: need T >= 0, k >= 1, H a positive multiple of 4");
    if (T == 0) return FT_OK;
    if (!y || !inv || !w || !out) return fail(FT_ERR_INVALID_ARG, "ft_moe_combine: null pointer");
    if (!aligned(y, 16) || !aligned(out, 8)) return fail(FT_ERR_INVALID_ARG, "ft_moe_combine: misaligned y or out");
    const dim3 grid(T, (H / 4 + 255) / 256);
    k_combine<<<grid, 256, 0, cu(stream)>>>(y, inv, w, T, k, H, out);
    return check_launch("ft_moe_combine");
}

}  // extern "C"
