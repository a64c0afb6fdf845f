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
    // pinned staging of the published tables: a ring per layer, each entry guarded by an event
    static constexpr int kRing = 4;
    int32_t* pinned = nullptr;  // [L][kRing][E]
    std::vector<cudaEvent_t> ring_ev;  // [L][kRing]
    std::vector<int> ring_pos;         // [L]
    // statistics and the host-side fault hook
    int64_t hits = 0, misses = 0, fills = 0, bytes_filled = 0;
    int64_t fail_at_fill = -1;  // the fill with this index (0-based) reports a failure instead of copying
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
        if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
    }
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
    for (int e : order) {
        int s = slot_of[e];
        if (s >= 0) {
            stamp[s] = step;
            ++c->hits;
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
        miss_experts[nm] = e;
        miss_slots[nm] = s;
        ++nm;
        ++c->misses;
    }
    for (int i = 0; i < n; ++i) slots_out[i] = slot_of[ids[i]];
    *n_miss = nm;
    return FT_OK;
}

ft_status ft_expert_cache_fill(ft_expert_cache* c, int layer, int expert, int slot, ft_stream_t copy_stream,
                               ft_event_t done) {
    const char* fn = "ft_expert_cache_fill";
    if (!c) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null cache");
    if (layer < 0 || layer >= c->L || expert < 0 || expert >= c->E || slot < 0 || slot >= c->S)
        return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": layer, expert or slot out of range");
    int64_t idx;
    {
        std::lock_guard<std::mutex> lock(c->mu);
        idx = c->fills++;
    }
    if (idx == c->fail_at_fill) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": injected copy failure");
    uint8_t* dst = c->slots + ((size_t)layer * c->S + slot) * c->slot_stride;
    cudaError_t e = cudaMemcpyAsync(dst, c->host[(size_t)layer * c->E + expert], c->expert_bytes, cudaMemcpyHostToDevice,
                                    ft::cu(copy_stream));
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaMemcpyAsync: " + cudaGetErrorString(e));
    if (done) {
        e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(done), ft::cu(copy_stream));
        if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaEventRecord: " + cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lock(c->mu);
    c->bytes_filled += (int64_t)c->expert_bytes;
    return FT_OK;
}

ft_status ft_expert_cache_publish(ft_expert_cache* c, int layer, ft_stream_t stream) {
    const char* fn = "ft_expert_cache_publish";
    if (!c) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null cache");
    if (layer < 0 || layer >= c->L) return cache_fail(FT_ERR_INVALID_ARG, std::string(fn) + ": layer out of range");
    std::lock_guard<std::mutex> lock(c->mu);
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
    e = cudaMemcpyAsync(c->tables + (size_t)layer * c->E, stage, sizeof(int32_t) * c->E, cudaMemcpyHostToDevice,
                        ft::cu(stream));
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaMemcpyAsync: " + cudaGetErrorString(e));
    e = cudaEventRecord(ev, ft::cu(stream));
    if (e != cudaSuccess) return cache_fail(FT_ERR_CUDA, std::string(fn) + ": cudaEventRecord: " + cudaGetErrorString(e));
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
