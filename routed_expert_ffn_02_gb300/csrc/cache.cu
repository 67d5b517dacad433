// cache.cu -- an HBM-resident expert cache with a host-memory cold tier.
//
// The GB300 analogue of the pages' elastic VRAM expert cache (dsv41-flash-
// offload wiki, overview and file map: a VRAM expert cache in front of the
// experts kept in host RAM), for models whose experts do not all fit in HBM.
// The cache owns n_slots expert slots in one caller-allocated device block;
// an expert of any layer, once copied in, stays resident across calls until
// it is the least recently used one and its slot is needed.  A call runs
// n_layers layers:
//
//   1. compute stream: route every layer and mark its touched experts in a
//      pinned host flag array written by the GPU; synchronise once.
//   2. for layer l: each touched expert is a hit (already in a slot) or a
//      miss; a miss takes the least recently used slot not needed by layer l
//      and is copied in on the copy stream (W_gate, W_up, W_down rows of that
//      expert), after the compute of the last layer that read the slot; one
//      copy kernel per layer moves all of its misses (SM loads over the host
//      link, see expert_copy.cu).  The
//      layer's expert -> slot table goes to the device on the compute stream,
//      which waits for the layer's copies and runs the layer on the slots.
//
// Every event a copy waits on was recorded for an earlier layer's compute,
// so the two streams never wait on each other in a cycle.
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "moe_internal.cuh"

namespace {

size_t expert_bytes(const moe_shape* sh) { return (size_t)sh->I * sh->H * sizeof(moe_bf16); }

size_t table_bytes(const moe_shape* sh, int max_layers) {
    return moe::align_up((size_t)max_layers * sh->E * sizeof(int32_t), 256);
}

moe_status cache_fail(moe_status st, const char* msg) {
    moe::set_last_error("%s", msg);
    return st;
}

moe_status cuda_fail(const char* where, cudaError_t e) {
    moe::set_last_error("%s: %s", where, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

}  // namespace

struct moe_cache {
    int E, H, I;
    int n_slots, max_layers;
    uint8_t* wg;                 // [n_slots, I, H] bf16
    uint8_t* wu;                 // [n_slots, I, H]
    uint8_t* wd;                 // [n_slots, H, I]
    int32_t* tables_d;           // [max_layers, E] expert -> slot, one row per layer of a call
    int32_t* tables_h;           // pinned staging of the same
    uint8_t* flags_h = nullptr;  // [max_layers, E] touched flags, pinned and mapped
    uint8_t* flags_d = nullptr;
    moe::ExpertCopyList list;         // the misses of the layer being enqueued
    std::vector<int64_t> key;         // per slot: layer_id << 32 | expert, -1 when empty
    std::vector<int64_t> last_use;    // per slot: tick of the last layer that needed it
    std::vector<int> reader;          // per slot: done[] index of that layer, -1 if none
    std::unordered_map<int64_t, int> where;
    std::vector<cudaEvent_t> done;    // ring of per-layer "compute finished" events
    std::vector<cudaEvent_t> copied;  // ring of per-layer "copies landed" events
    int64_t tick = 0, hits = 0, misses = 0;
    int ring = 0;
};

extern "C" size_t moe_cache_bytes(const moe_shape* shape, int32_t n_slots, int32_t max_layers) {
    if (moe::check_shape_status(shape) != MOE_OK || n_slots < 1 || max_layers < 1) return 0;
    return 3 * (size_t)n_slots * expert_bytes(shape) + table_bytes(shape, max_layers);
}

extern "C" moe_status moe_cache_create(const moe_shape* shape, int32_t n_slots,
                                       int32_t max_layers, void* mem, size_t mem_bytes,
                                       moe_cache** out) {
    if (!out) return cache_fail(MOE_ERR_INVALID_ARG, "moe_cache_create: out is NULL");
    *out = nullptr;
    const size_t need = moe_cache_bytes(shape, n_slots, max_layers);
    if (need == 0) return cache_fail(MOE_ERR_INVALID_ARG, "moe_cache_create: bad shape or sizes");
    if (!mem || (reinterpret_cast<uintptr_t>(mem) % 256) || mem_bytes < need)
        return cache_fail(MOE_ERR_INVALID_ARG,
                          "moe_cache_create: memory NULL, misaligned or below moe_cache_bytes");
    moe_cache* c = new (std::nothrow) moe_cache();
    if (!c) return cache_fail(MOE_ERR_CUDA, "moe_cache_create: out of host memory");
    c->E = shape->E;
    c->H = shape->H;
    c->I = shape->I;
    c->n_slots = n_slots;
    c->max_layers = max_layers;
    const size_t slab = (size_t)n_slots * expert_bytes(shape);
    c->wg = static_cast<uint8_t*>(mem);
    c->wu = c->wg + slab;
    c->wd = c->wu + slab;
    c->tables_d = reinterpret_cast<int32_t*>(c->wd + slab);
    c->key.assign(n_slots, -1);
    c->last_use.assign(n_slots, -1);
    c->reader.assign(n_slots, -1);
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&c->tables_h),
                                  (size_t)max_layers * shape->E * sizeof(int32_t),
                                  cudaHostAllocDefault);
    void* fh = nullptr;
    void* fd = nullptr;
    if (e == cudaSuccess) e = cudaHostAlloc(&fh, (size_t)max_layers * shape->E, cudaHostAllocMapped);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&fd, fh, 0);
    c->flags_h = static_cast<uint8_t*>(fh);
    c->flags_d = static_cast<uint8_t*>(fd);
    for (int i = 0; e == cudaSuccess && i < max_layers; ++i) {
        cudaEvent_t a = nullptr, b = nullptr;
        e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
        if (a) c->done.push_back(a);
        if (b) c->copied.push_back(b);
    }
    if (e != cudaSuccess) {
        moe_cache_destroy(c);
        return cuda_fail("moe_cache_create", e);
    }
    *out = c;
    moe::set_last_error("");
    return MOE_OK;
}

extern "C" moe_status moe_cache_destroy(moe_cache* c) {
    if (!c) return MOE_OK;
    for (cudaEvent_t ev : c->done) cudaEventDestroy(ev);
    for (cudaEvent_t ev : c->copied) cudaEventDestroy(ev);
    if (c->tables_h) cudaFreeHost(c->tables_h);
    if (c->flags_h) cudaFreeHost(c->flags_h);
    delete c;
    return MOE_OK;
}

extern "C" moe_status moe_cache_stats(const moe_cache* c, int64_t* hits, int64_t* misses) {
    if (!c || !hits || !misses) return cache_fail(MOE_ERR_INVALID_ARG, "moe_cache_stats: NULL");
    *hits = c->hits;
    *misses = c->misses;
    return MOE_OK;
}

extern "C" moe_status moe_forward_cached(moe_cache* c, const moe_shape* shape, int32_t n_layers,
                                         const int32_t* layer_ids, const float* const* logits,
                                         const moe_bf16* x, const void* const* host_weights,
                                         moe_bf16* const* out, void* ws, size_t ws_bytes,
                                         moe_stream_t compute, moe_stream_t copy) {
    if (!c) return cache_fail(MOE_ERR_INVALID_ARG, "moe_forward_cached: cache is NULL");
    moe_status st = moe::check_shape_status(shape);
    if (st != MOE_OK) return st;
    if (shape->E != c->E || shape->H != c->H || shape->I != c->I)
        return cache_fail(MOE_ERR_INVALID_ARG, "moe_forward_cached: shape differs from the cache's");
    if (n_layers < 0 || n_layers > c->max_layers ||
        (n_layers > 0 && (!layer_ids || !logits || !host_weights || !out)))
        return cache_fail(MOE_ERR_INVALID_ARG, "moe_forward_cached: bad layer arguments");
    if (compute == copy)
        return cache_fail(MOE_ERR_INVALID_ARG,
                          "moe_forward_cached: the copy stream must differ from the compute stream");
    for (int l = 0; l < n_layers; ++l) {
        if (layer_ids[l] < 0 || !logits[l] || !host_weights[l] || !out[l])
            return cache_fail(MOE_ERR_INVALID_ARG, "moe_forward_cached: bad layer pointer or id");
        const void* view = nullptr;
        if (moe::device_view_of_host(host_weights[l], &view) != cudaSuccess ||
            reinterpret_cast<uintptr_t>(view) % 16)
            return cache_fail(MOE_ERR_INVALID_ARG,
                              "moe_forward_cached: host weights must be 16-byte aligned pinned "
                              "host memory");
    }
    if (n_layers == 0 || shape->T == 0) {
        moe::set_last_error("");
        return MOE_OK;
    }
    cudaStream_t cs = (cudaStream_t)compute, ks = (cudaStream_t)copy;
    const int E = c->E;
    const size_t eb = expert_bytes(shape);
    cudaError_t e;

    // 1. touched experts of every layer (the previous call synchronised).
    memset(c->flags_h, 0, (size_t)n_layers * E);
    for (int l = 0; l < n_layers; ++l) {
        st = moe::mark_touched_experts(shape, logits[l], ws, ws_bytes, c->flags_d + (size_t)l * E,
                                       cs);
        if (st != MOE_OK) return st;
    }
    if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail("moe_forward_cached", e);

    // 2. per layer: hits, misses into least recently used slots, the layer.
    std::vector<int> need;
    for (int l = 0; l < n_layers; ++l) {
        const uint8_t* touched = c->flags_h + (size_t)l * E;
        need.clear();
        for (int ex = 0; ex < E; ++ex)
            if (touched[ex]) need.push_back(ex);
        if ((int)need.size() > c->n_slots)
            return cache_fail(MOE_ERR_INVALID_ARG,
                              "moe_forward_cached: a layer touches more experts than the cache has slots");
        const int64_t now = ++c->tick;
        const int ev = c->ring;
        c->ring = (c->ring + 1) % c->max_layers;
        int32_t* table = c->tables_h + (size_t)l * E;
        for (int ex = 0; ex < E; ++ex) table[ex] = 0;     // untouched: never read
        // hits first, so that misses cannot evict an expert this layer needs
        std::vector<int> miss;
        for (int ex : need) {
            const int64_t k = ((int64_t)layer_ids[l] << 32) | (uint32_t)ex;
            auto it = c->where.find(k);
            if (it != c->where.end()) {
                table[ex] = it->second;
                c->last_use[it->second] = now;
                c->reader[it->second] = ev;
                ++c->hits;
            } else {
                miss.push_back(ex);
            }
        }
        c->list.n = 0;
        for (int ex : miss) {
            int victim = -1;
            for (int s = 0; s < c->n_slots; ++s)
                if (c->last_use[s] != now && (victim < 0 || c->last_use[s] < c->last_use[victim]))
                    victim = s;
            // a victim exists: this layer needs at most n_slots slots
            if (c->key[victim] >= 0) c->where.erase(c->key[victim]);
            if (c->reader[victim] >= 0 &&
                (e = cudaStreamWaitEvent(ks, c->done[c->reader[victim]], 0)) != cudaSuccess)
                return cuda_fail("moe_forward_cached", e);
            c->list.src_e[c->list.n] = ex;
            c->list.dst_e[c->list.n] = victim;
            ++c->list.n;
            const int64_t k = ((int64_t)layer_ids[l] << 32) | (uint32_t)ex;
            c->key[victim] = k;
            c->where[k] = victim;
            c->last_use[victim] = now;
            c->reader[victim] = ev;
            table[ex] = victim;
            ++c->misses;
        }
        const void* src = nullptr;
        if ((e = moe::device_view_of_host(host_weights[l], &src)) != cudaSuccess)   // checked above
            return cuda_fail("moe_forward_cached", e);
        const size_t mat = (size_t)E * eb;   // bytes of one matrix for all experts
        const void* srcs[3] = {src, static_cast<const uint8_t*>(src) + mat,
                               static_cast<const uint8_t*>(src) + 2 * mat};
        void* dsts[3] = {c->wg, c->wu, c->wd};
        if ((e = moe::launch_expert_copy(c->list, srcs, dsts, eb, ks)) != cudaSuccess)
            return cuda_fail("moe_forward_cached", e);
        int32_t* table_d = c->tables_d + (size_t)l * E;
        if ((e = cudaEventRecord(c->copied[ev], ks)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs, c->copied[ev], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(table_d, table, (size_t)E * sizeof(int32_t),
                                 cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return cuda_fail("moe_forward_cached", e);
        st = moe::forward_blocks(shape, logits[l], x, reinterpret_cast<const moe_bf16*>(c->wg),
                                 reinterpret_cast<const moe_bf16*>(c->wu),
                                 reinterpret_cast<const moe_bf16*>(c->wd), table_d, c->n_slots,
                                 out[l], ws, ws_bytes, compute);
        if (st != MOE_OK) return st;
        if ((e = cudaEventRecord(c->done[ev], cs)) != cudaSuccess)
            return cuda_fail("moe_forward_cached", e);
    }
    moe::set_last_error("");
    return MOE_OK;
}
