// expert_cache.cu -- VRAM expert-slot cache with an LRU replacement policy,
// filled from pinned host memory by asynchronous copies on a side stream.
//
// Page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier MoE 拉回本地",
// section 设计核心 (second principle): a global LRU cache of experts in VRAM
// catches the locality of adjacent tokens, so only misses travel from host
// memory.  Page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", paragraph on
// bandwidth-aware storage: hot experts stay in VRAM and cudaMemcpyAsync on CUDA
// streams overlaps transfers with compute.
//
// The policy details the pages leave open are fixed here:
//  * one cache per layer with S slots, initially empty;
//  * a token's k experts are visited in ascending expert id;
//  * a hit sets the expert's last-use stamp to the current step;
//  * a miss takes the lowest free slot, else evicts the slot with the oldest
//    stamp among experts the current token does not select (lower slot wins a
//    tie); the new expert's stamp is the current step.
//
// Elastic resize (same page, section 设计核心, third mechanism: the cache is
// resized and rebuilt from free VRAM at safe points, with no restart and no
// reload): the resident experts move device to device into the new pool (or
// are compacted in place when it shrinks); the ones that no longer fit go,
// least recently used first.
//
// Everything here is host bookkeeping plus cudaMemcpyAsync: the caller owns the
// pinned host pool, the device slot pool and the device slot tables.
#include "common.cuh"

#include <algorithm>
#include <mutex>
#include <vector>

struct ft_expert_cache {
    int L = 0, E = 0, S = 0;
    size_t expert_bytes = 0, slot_stride = 0;
    std::vector<const void*> host;  // [L*E] pinned host source of each expert
    uint8_t* slots = nullptr;       // device slot pool
    int32_t* tables = nullptr;      // device [L][E] expert -> slot or -1
    // per layer
    std::vector<std::vector<int32_t>> expert_of;  // [L][S] slot -> expert (-1 free)
    std::vector<std::vector<int64_t>> stamp;      // [L][S] step of last use
    std::vector<std::vector<int32_t>> slot_of;    // [L][E] expert -> slot (-1 absent)
    std::vector<std::vector<uint8_t>> fetched;    // [L][S] put there by a prefetch and not used since
    // pinned staging of the published tables: a ring per layer, each entry guarded by an event
    static constexpr int kRing = 4;
    int32_t* pinned = nullptr;  // [L][kRing][E]
    std::vector<cudaEvent_t> ring_ev;  // [L][kRing]
    std::vector<int> ring_pos;         // [L]
    // statistics and the host-side fault hook
    int64_t hits = 0, misses = 0, fills = 0, bytes_filled = 0;
    int64_t prefetched = 0, prefetch_used = 0;  // experts installed by a prefetch; of those, later used
    int64_t fail_at_fill = -1;  // the slot copy (fill or resize move) with this 0-based index fails instead
    std::mutex mu;
};

namespace {

ft_status cache_fail(ft_status s, const std::string& msg) { return ft::fail(s, msg); }

}  // namespace

extern "C" {

ft_status ft_expert_cache_create(int L, int E, int S, size_t expert_bytes, const void* const* host_experts, void* slots,
                                 size_t slot_stride, int32_t* tables, ft_expert_cache** out) {
    const char* fn = "ft_expert_cache_create";
    if (!out) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": out is null");
    *out = nullptr;
    if (L <= 0 || E <= 0 || E > 1024 || S <= 0 || S > E || expert_bytes == 0)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need L > 0, 1 <= S <= E <= 1024, expert_bytes > 0");
    if (!host_experts || !slots || !tables) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (slot_stride < expert_bytes || slot_stride % 256 || reinterpret_cast<uintptr_t>(slots) % 256)
        return cache_fail(FT_ERR_INVALID_ARG,
                          std::string(fn) + ": slot_stride must be >= expert_bytes and both it and slots 256-byte aligned");
    for (int i = 0; i < L * E; ++i)
        if (!host_experts[i]) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null host expert pointer");
    auto* c = new (std::nothrow) ft_expert_cache();
    if (!c) return cache_fail(FT_ERR_OOM, std::string(fn) + ": host allocation failed");
    c->L = L;
    c->E = E;
    c->S = S;
    c->expert_bytes = expert_bytes;
    c->slot_stride = slot_stride;
    c->host.assign(host_experts, host_experts + (size_t)L * E);
    c->slots = static_cast<uint8_t*>(slots);
    c->tables = tables;
    c->expert_of.assign(L, std::vector<int32_t>(S, -1));
    c->stamp.assign(L, std::vector<int64_t>(S, -1));
    c->slot_of.assign(L, std::vector<int32_t>(E, -1));
    c->fetched.assign(L, std::vector<uint8_t>(S, 0));
    c->ring_pos.assign(L, 0);
    *out = c;
    return FT_OK;
}

}  // extern "C"

namespace {

// Pinned staging of the published tables and their events, made on the first publish
// (so that creating a cache and looking experts up need no device).
ft_status ensure_staging(ft_expert_cache* c, const char* fn) {
    if (c->pinned) return FT_OK;
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&c->pinned),
                                  sizeof(int32_t) * (size_t)c->L * c->kRing * c->E, cudaHostAllocDefault);
    if (e != cudaSuccess) {
        c->pinned = nullptr;
        return cache_fail(FT_ERR_OOM, std::string(fn) + ": pinned table staging: " + cudaGetErrorString(e));
    }
    std::fill(c->pinned, c->pinned + (size_t)c->L * c->kRing * c->E, -1);
    c->ring_ev.assign((size_t)c->L * c->kRing, nullptr);
    for (auto& ev : c->ring_ev) {
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) {  // undo it all, so that the next publish tries again from scratch
            ev = nullptr;
            for (auto& made : c->ring_ev)
                if (made) cudaEventDestroy(made);
            c->ring_ev.clear();
            cudaFreeHost(c->pinned);
            c->pinned = nullptr;
            return cache_fail(FT_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
        }
    }
    return FT_OK;
}

// Plan of one layer for a resize to new_S slots: moves[i] = the old slot whose
// expert goes to new slot i, or -1.  The occupied slots are always a prefix
// (misses take the lowest free slot; evictions reuse the victim's slot).  When
// they fit, all are kept; otherwise the new_S with the newest stamps (the lower
// old slot on a tie).  The kept experts take new slots 0.. in ascending old-slot
// order, which a compaction in place relies on.
void plan_layer(const ft_expert_cache* c, int layer, int new_S, int32_t* moves) {
    const auto& expert_of = c->expert_of[layer];
    const auto& stamp = c->stamp[layer];
    std::vector<int32_t> occ;
    for (int q = 0; q < c->S; ++q)
        if (expert_of[q] >= 0) occ.push_back(q);
    if ((int)occ.size() > new_S) {
        std::stable_sort(occ.begin(), occ.end(), [&](int32_t a, int32_t b) { return stamp[a] > stamp[b]; });
        occ.resize(new_S);
        std::sort(occ.begin(), occ.end());
    }
    for (int i = 0; i < new_S; ++i) moves[i] = i < (int)occ.size() ? occ[i] : -1;
}

// Device-to-device moves of whole slots between two disjoint pools, passed by
// value (up to kMovesPerLaunch per launch): block (c, m) copies bytes
// [c*kMoveChunk, min(bytes, (c+1)*kMoveChunk)) of move m, 16 bytes per thread
// and step (slot starts are 256-byte aligned), the last bytes singly.
constexpr int kMovesPerLaunch = 256;
constexpr size_t kMoveChunk = 64 * 1024;
struct SlotMoves {
    int32_t src[kMovesPerLaunch];  // global slot index in the old pool (layer*S + slot)
    int32_t dst[kMovesPerLaunch];  // global slot index in the new pool (layer*new_S + slot)
};

__global__ void __launch_bounds__(256) k_slot_moves(const uint8_t* __restrict__ old_base, size_t old_stride,
                                                    uint8_t* __restrict__ new_base, size_t new_stride, size_t bytes,
                                                    SlotMoves mv) {
    const int m = blockIdx.y;
    const size_t c0 = (size_t)blockIdx.x * kMoveChunk;
    if (c0 >= bytes) return;
    const size_t c1 = c0 + kMoveChunk < bytes ? c0 + kMoveChunk : bytes;
    const uint8_t* src = old_base + (size_t)mv.src[m] * old_stride;
    uint8_t* dst = new_base + (size_t)mv.dst[m] * new_stride;
    const size_t v1 = c0 + ((c1 - c0) & ~(size_t)15);  // c0 is a multiple of 16
    for (size_t o = c0 + 16 * (size_t)threadIdx.x; o < v1; o += 16 * (size_t)blockDim.x)
        *reinterpret_cast<uint4*>(dst + o) = __ldg(reinterpret_cast<const uint4*>(src + o));
    for (size_t o = v1 + threadIdx.x; o < c1; o += blockDim.x) dst[o] = src[o];
}

// Copy of layer `layer`'s expert -> slot table to the device, through the pinned ring (caller holds the lock).
ft_status publish_locked(ft_expert_cache* c, int layer, cudaStream_t stream, const char* fn) {
    ft_status st = ensure_staging(c, fn);
    if (st != FT_OK) return st;
    const int pos = c->ring_pos[layer];
    c->ring_pos[layer] = (pos + 1) % c->kRing;
    cudaEvent_t ev = c->ring_ev[(size_t)layer * c->kRing + pos];
    // the staging entry may still feed a copy issued kRing publishes ago
    cudaError_t e = cudaEventSynchronize(ev);
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
    int32_t* stage = c->pinned + ((size_t)layer * c->kRing + pos) * c->E;
    std::copy(c->slot_of[layer].begin(), c->slot_of[layer].end(), stage);
    e = cudaMemcpyAsync(c->tables + (size_t)layer * c->E, stage, sizeof(int32_t) * c->E, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaMemcpyAsync: " + cudaGetErrorString(e));
    e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaEventRecord: " + cudaGetErrorString(e));
    return FT_OK;
}

}  // namespace

extern "C" {

ft_status ft_expert_cache_destroy(ft_expert_cache* c) {
    if (!c) return FT_OK;
    for (auto ev : c->ring_ev)
        if (ev) {
            cudaEventSynchronize(ev);
            cudaEventDestroy(ev);
        }
    if (c->pinned) cudaFreeHost(c->pinned);
    delete c;
    return FT_OK;
}

ft_status ft_expert_cache_lookup(ft_expert_cache* c, int layer, int64_t step, const int32_t* ids, int n,
                                 int32_t* slots_out, int32_t* miss_experts, int32_t* miss_slots, int* n_miss) {
    const char* fn = "ft_expert_cache_lookup";
    if (!c || !ids || !slots_out || !miss_experts || !miss_slots || !n_miss)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (layer < 0 || layer >= c->L || n < 0 || n > c->S)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 0 <= layer < L and 0 <= n <= S");
    std::lock_guard<std::mutex> lock(c->mu);
    std::vector<int32_t> order(ids, ids + n);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= c->E) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": expert id out of range");
    std::sort(order.begin(), order.end());
    for (int i = 1; i < n; ++i)
        if (order[i] == order[i - 1]) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": repeated expert id");
    auto& expert_of = c->expert_of[layer];
    auto& stamp = c->stamp[layer];
    auto& slot_of = c->slot_of[layer];
    int nm = 0;
    auto& fetched = c->fetched[layer];
    for (int e : order) {
        int s = slot_of[e];
        if (s >= 0) {
            stamp[s] = step;
            ++c->hits;
            if (fetched[s]) {
                fetched[s] = 0;
                ++c->prefetch_used;
            }
            continue;
        }
        s = -1;
        for (int q = 0; q < c->S; ++q)
            if (expert_of[q] < 0) {
                s = q;
                break;
            }
        if (s < 0) {  // evict the oldest stamp among experts the token does not select (lower slot on a tie)
            for (int q = 0; q < c->S; ++q) {
                if (std::binary_search(order.begin(), order.end(), expert_of[q])) continue;
                if (s < 0 || stamp[q] < stamp[s]) s = q;
            }
            if (s < 0) return cache_fail(FT_ERR_NO_SLOT, std::string(fn) + ": no evictable slot");
            slot_of[expert_of[s]] = -1;
        }
        expert_of[s] = e;
        stamp[s] = step;
        slot_of[e] = s;
        fetched[s] = 0;
        miss_experts[nm] = e;
        miss_slots[nm] = s;
        ++nm;
        ++c->misses;
    }
    for (int i = 0; i < n; ++i) slots_out[i] = slot_of[ids[i]];
    *n_miss = nm;
    return FT_OK;
}

ft_status ft_expert_cache_prefetch(ft_expert_cache* c, int layer, int64_t step, const int32_t* ids, int n,
                                   int32_t* fill_experts, int32_t* fill_slots, int* n_fill) {
    const char* fn = "ft_expert_cache_prefetch";
    if (!c || (n > 0 && (!ids || !fill_experts || !fill_slots)) || !n_fill)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (layer < 0 || layer >= c->L || n < 0 || n > c->E)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 0 <= layer < L and 0 <= n <= E");
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= c->E) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": expert id out of range");
    std::lock_guard<std::mutex> lock(c->mu);
    std::vector<int32_t> order(ids, ids + n);
    std::sort(order.begin(), order.end());
    order.erase(std::unique(order.begin(), order.end()), order.end());
    auto& expert_of = c->expert_of[layer];
    auto& stamp = c->stamp[layer];
    auto& slot_of = c->slot_of[layer];
    auto& fetched = c->fetched[layer];
    int nf = 0;
    for (int e : order) {
        if (slot_of[e] >= 0) continue;  // resident: left as it is (a prediction is not a use)
        int s = -1;
        for (int q = 0; q < c->S; ++q)
            if (expert_of[q] < 0) {
                s = q;
                break;
            }
        if (s < 0) {  // the oldest stamp before `step` (lower slot on a tie) among experts not predicted now;
                      // this step's experts stay
            for (int q = 0; q < c->S; ++q)
                if (stamp[q] < step && !std::binary_search(order.begin(), order.end(), expert_of[q]) &&
                    (s < 0 || stamp[q] < stamp[s]))
                    s = q;
            if (s < 0) continue;
            slot_of[expert_of[s]] = -1;
        }
        expert_of[s] = e;
        stamp[s] = step - 1;
        slot_of[e] = s;
        fetched[s] = 1;
        fill_experts[nf] = e;
        fill_slots[nf] = s;
        ++nf;
        ++c->prefetched;
    }
    *n_fill = nf;
    return FT_OK;
}

ft_status ft_expert_cache_prefetch_stats(ft_expert_cache* c, int64_t* prefetched, int64_t* used) {
    if (!c || !prefetched || !used) return cache_fail(FT_ERR_INVALID_ARG, "ft_expert_cache_prefetch_stats: null pointer");
    std::lock_guard<std::mutex> lock(c->mu);
    *prefetched = c->prefetched;
    *used = c->prefetch_used;
    return FT_OK;
}

ft_status ft_expert_cache_fill(ft_expert_cache* c, int layer, int expert, int slot, ft_stream_t copy_stream,
                               ft_event_t done) {
    const char* fn = "ft_expert_cache_fill";
    if (!c) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null cache");
    // the whole call holds the lock: a resize changes the pool, its slot count and its stride
    std::lock_guard<std::mutex> lock(c->mu);
    if (layer < 0 || layer >= c->L || expert < 0 || expert >= c->E || slot < 0 || slot >= c->S)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": layer, expert or slot out of range");
    if (c->fills++ == c->fail_at_fill) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": injected copy failure");
    uint8_t* dst = c->slots + ((size_t)layer * c->S + slot) * c->slot_stride;
    cudaError_t e = cudaMemcpyAsync(dst, c->host[(size_t)layer * c->E + expert], c->expert_bytes, cudaMemcpyHostToDevice,
                                    ft::cu(copy_stream));
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaMemcpyAsync: " + cudaGetErrorString(e));
    if (done) {
        e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(done), ft::cu(copy_stream));
        if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaEventRecord: " + cudaGetErrorString(e));
    }
    c->bytes_filled += (int64_t)c->expert_bytes;
    return FT_OK;
}

ft_status ft_expert_cache_publish(ft_expert_cache* c, int layer, ft_stream_t stream) {
    const char* fn = "ft_expert_cache_publish";
    if (!c) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null cache");
    if (layer < 0 || layer >= c->L) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": layer out of range");
    std::lock_guard<std::mutex> lock(c->mu);
    return publish_locked(c, layer, ft::cu(stream), fn);
}

ft_status ft_expert_cache_resize_plan(ft_expert_cache* c, int new_S, int32_t* moves) {
    const char* fn = "ft_expert_cache_resize_plan";
    if (!c || !moves) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (new_S <= 0 || new_S > c->E) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= new_S <= E");
    std::lock_guard<std::mutex> lock(c->mu);
    for (int l = 0; l < c->L; ++l) plan_layer(c, l, new_S, moves + (size_t)l * new_S);
    return FT_OK;
}

ft_status ft_expert_cache_resize(ft_expert_cache* c, int new_S, void* new_slots, size_t new_slot_stride,
                                 ft_stream_t stream) {
    const char* fn = "ft_expert_cache_resize";
    if (!c || !new_slots) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (new_S <= 0 || new_S > c->E) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= new_S <= E");
    if (new_slot_stride < c->expert_bytes || new_slot_stride % 256 || reinterpret_cast<uintptr_t>(new_slots) % 256)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) +
                                                  ": new_slot_stride must be >= expert_bytes and both it and new_slots "
                                                  "256-byte aligned");
    std::lock_guard<std::mutex> lock(c->mu);
    uint8_t* nb = static_cast<uint8_t*>(new_slots);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(c->slots), o1 = o0 + (size_t)c->L * c->S * c->slot_stride;
    const uintptr_t n0 = reinterpret_cast<uintptr_t>(nb), n1 = n0 + (size_t)c->L * new_S * new_slot_stride;
    const bool overlap = n0 < o1 && o0 < n1;
    const bool in_place = nb == c->slots && new_slot_stride == c->slot_stride && new_S <= c->S;
    if (overlap && !in_place)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) +
                                                  ": the new pool overlaps the old one (only a shrink in place, same "
                                                  "base and stride, may)");
    std::vector<int32_t> moves((size_t)c->L * new_S);
    for (int l = 0; l < c->L; ++l) plan_layer(c, l, new_S, moves.data() + (size_t)l * new_S);
    ft_status st = FT_OK;
    std::string err;
    if (in_place) {
        // Moves in ascending (layer, new slot) order on one stream, one slot per copy: new index l*new_S + i is
        // never above the source l*S + q (i <= q, new_S <= S) and sources only grow, so no copy overwrites a
        // source still unread, and same-stride slots never partly overlap.
        for (int l = 0; l < c->L && st == FT_OK; ++l)
            for (int i = 0; i < new_S && st == FT_OK; ++i) {
                const int q = moves[(size_t)l * new_S + i];
                if (q < 0) continue;
                const uint8_t* src = c->slots + ((size_t)l * c->S + q) * c->slot_stride;
                uint8_t* dst = nb + ((size_t)l * new_S + i) * new_slot_stride;
                if (src == dst) continue;
                if (c->fills++ == c->fail_at_fill) {
                    st = FT_ERR_CUDA;
                    err = "injected copy failure";
                    break;
                }
                const cudaError_t e =
                    cudaMemcpyAsync(dst, src, c->expert_bytes, cudaMemcpyDeviceToDevice, ft::cu(stream));
                if (e != cudaSuccess) {
                    st = FT_ERR_CUDA;
                    err = std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e);
                }
            }
    } else {
        // Disjoint pools: all moves are independent, so one copy kernel per kMovesPerLaunch of them (a
        // cudaMemcpyAsync per expert pays a fixed cost of several microseconds, about what its bytes take).
        SlotMoves mv;
        int n = 0;
        const unsigned chunks = (unsigned)((c->expert_bytes + kMoveChunk - 1) / kMoveChunk);
        auto flush = [&]() {
            if (n == 0) return;
            if (c->fills++ == c->fail_at_fill) {
                st = FT_ERR_CUDA;
                err = "injected copy failure";
                return;
            }
            k_slot_moves<<<dim3(chunks, (unsigned)n), 256, 0, ft::cu(stream)>>>(c->slots, c->slot_stride, nb,
                                                                               new_slot_stride, c->expert_bytes, mv);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) {
                st = FT_ERR_CUDA;
                err = std::string("slot move kernel: ") + cudaGetErrorString(e);
            }
            n = 0;
        };
        for (int l = 0; l < c->L && st == FT_OK; ++l)
            for (int i = 0; i < new_S && st == FT_OK; ++i) {
                const int q = moves[(size_t)l * new_S + i];
                if (q < 0) continue;
                mv.src[n] = l * c->S + q;
                mv.dst[n] = l * new_S + i;
                if (++n == kMovesPerLaunch) flush();
            }
        if (st == FT_OK) flush();
    }
    // the new geometry in either case; after a failed move no slot is trusted and every access refills from host
    for (int l = 0; l < c->L; ++l) {
        std::vector<int32_t> eo(new_S, -1);
        std::vector<int64_t> sp(new_S, -1);
        std::vector<uint8_t> fe(new_S, 0);
        if (st == FT_OK)
            for (int i = 0; i < new_S; ++i) {
                const int q = moves[(size_t)l * new_S + i];
                if (q < 0) continue;
                eo[i] = c->expert_of[l][q];
                sp[i] = c->stamp[l][q];
                fe[i] = c->fetched[l][q];
            }
        std::fill(c->slot_of[l].begin(), c->slot_of[l].end(), -1);
        for (int i = 0; i < new_S; ++i)
            if (eo[i] >= 0) c->slot_of[l][eo[i]] = i;
        c->expert_of[l].swap(eo);
        c->stamp[l].swap(sp);
        c->fetched[l].swap(fe);
    }
    c->S = new_S;
    c->slots = nb;
    c->slot_stride = new_slot_stride;
    if (st != FT_OK) return cache_fail(st, std::string(fn) + ": " + err + " (the cache is now empty)");
    for (int l = 0; l < c->L; ++l) {
        st = publish_locked(c, l, ft::cu(stream), fn);
        if (st != FT_OK) return st;
    }
    return FT_OK;
}

ft_status ft_expert_cache_stats(ft_expert_cache* c, int64_t* hits, int64_t* misses, int64_t* bytes_filled) {
    if (!c || !hits || !misses || !bytes_filled)
        return cache_fail(FT_ERR_INVALID_ARG, "ft_expert_cache_stats: null pointer");
    std::lock_guard<std::mutex> lock(c->mu);
    *hits = c->hits;
    *misses = c->misses;
    *bytes_filled = c->bytes_filled;
    return FT_OK;
}

ft_status ft_expert_cache_inject_fill_failure(ft_expert_cache* c, int64_t fill_index) {
    if (!c) return cache_fail(FT_ERR_INVALID_ARG, "ft_expert_cache_inject_fill_failure: null cache");
    std::lock_guard<std::mutex> lock(c->mu);
    c->fail_at_fill = fill_index;
    return FT_OK;
}

}  // extern "C"
