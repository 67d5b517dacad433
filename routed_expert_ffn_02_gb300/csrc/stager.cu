// stager.cu -- expert weights streamed from pinned host memory into HBM
// staging slots on a side copy stream, overlapped with the layers' compute.
//
// All routed experts are kept in pinned host memory and copied into a ring
// of device staging slots in batches, overlapped with compute, with the next
// layers' copies issued while the current layer runs (dsv41-flash-offload
// wiki, overview and its notes on 8 staging slots and cross-layer DMA
// prefetch).  The wiki's batches go through the copy engine; here one copy
// kernel per layer moves them with SM loads, which keep the host link at its
// full rate where the copy engine's many separate copies do not (see
// expert_copy.cu).  Here one slot has room for one layer's whole
// expert set (W_gate | W_up | W_down, the layout moe_forward takes), but only
// the experts the layer's tokens are routed to are copied (the wiki's file
// map: one weight copy per batch for the experts with positive counts).
//
//   1. compute stream: route every layer and mark its touched experts in a
//      pinned host flag array (written by the GPU); synchronise once.
//   2. for layer l (slot s = l mod n_slots):
//      copy stream:    wait for the compute that last used slot s (layer
//                      l - n), one copy kernel for the touched experts'
//                      three matrices into the same offsets of slot s,
//                      record copied[s]
//      compute stream: wait copied[s], moe_forward on the slot, record
//                      freed[s]
//
// Untouched experts' regions of a slot keep stale bytes and are never read:
// no token is routed to them.  Every copy for all layers is enqueued up front,
// so the copies run up to n_slots layers ahead of the compute.  The
// caller owns the slot memory; the stager holds its events and the flag
// array (pinned host memory, grown on demand).
#include <cstdlib>
#include <cstring>
#include <new>

#include "moe_internal.cuh"

struct moe_stager {
    uint8_t* slots;
    int n_slots;
    size_t slot_bytes;
    cudaEvent_t* copied;
    cudaEvent_t* freed;
    uint8_t* flags_h;      // [n_layers x E] touched flags, pinned and mapped
    uint8_t* flags_d;      // the device's view of flags_h
    size_t flags_cap;
    moe::ExpertCopyList list;   // the layer being enqueued
};

namespace {

moe_status stager_fail(moe_status st, const char* msg) {
    moe::set_last_error("%s", msg);
    return st;
}

}  // namespace

extern "C" moe_status moe_stager_create(void* slots, int32_t n_slots, size_t slot_bytes,
                                        moe_stager** out) {
    if (!out) return stager_fail(MOE_ERR_INVALID_ARG, "moe_stager_create: out is NULL");
    *out = nullptr;
    if (!slots || n_slots < 1 || slot_bytes == 0 || (reinterpret_cast<uintptr_t>(slots) % 256) ||
        slot_bytes % 256)
        return stager_fail(MOE_ERR_INVALID_ARG,
                           "moe_stager_create: need n_slots >= 1 and 256-byte aligned slots");
    moe_stager* st = new (std::nothrow) moe_stager;
    if (!st) return stager_fail(MOE_ERR_CUDA, "moe_stager_create: out of host memory");
    st->slots = static_cast<uint8_t*>(slots);
    st->n_slots = n_slots;
    st->slot_bytes = slot_bytes;
    st->flags_h = nullptr;
    st->flags_d = nullptr;
    st->flags_cap = 0;
    st->copied = new (std::nothrow) cudaEvent_t[n_slots]();
    st->freed = new (std::nothrow) cudaEvent_t[n_slots]();
    if (!st->copied || !st->freed) {
        delete[] st->copied;
        delete[] st->freed;
        delete st;
        return stager_fail(MOE_ERR_CUDA, "moe_stager_create: out of host memory");
    }
    for (int i = 0; i < n_slots; ++i) {
        if (cudaEventCreateWithFlags(&st->copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&st->freed[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j <= i; ++j) {
                if (st->copied[j]) cudaEventDestroy(st->copied[j]);
                if (st->freed[j]) cudaEventDestroy(st->freed[j]);
            }
            delete[] st->copied;
            delete[] st->freed;
            delete st;
            return stager_fail(MOE_ERR_CUDA, "moe_stager_create: cudaEventCreate failed");
        }
    }
    *out = st;
    moe::set_last_error("");
    return MOE_OK;
}

extern "C" moe_status moe_stager_destroy(moe_stager* st) {
    if (!st) return MOE_OK;
    for (int i = 0; i < st->n_slots; ++i) {
        cudaEventDestroy(st->copied[i]);
        cudaEventDestroy(st->freed[i]);
    }
    delete[] st->copied;
    delete[] st->freed;
    if (st->flags_h) cudaFreeHost(st->flags_h);
    delete st;
    return MOE_OK;
}

extern "C" size_t moe_layer_weight_bytes(const moe_shape* shape) {
    if (!shape || shape->E < 1 || shape->H < 1 || shape->I < 1) return 0;
    return (size_t)3 * shape->E * shape->H * shape->I * sizeof(moe_bf16);
}

extern "C" moe_status moe_forward_offload(moe_stager* st, const moe_shape* shape,
                                          int32_t n_layers, const float* const* logits,
                                          const moe_bf16* x, const void* const* host_weights,
                                          moe_bf16* const* out, void* ws, size_t ws_bytes,
                                          moe_stream_t compute, moe_stream_t copy) {
    if (!st) return stager_fail(MOE_ERR_INVALID_ARG, "moe_forward_offload: stager is NULL");
    if (!shape || n_layers < 0 || (n_layers > 0 && (!logits || !host_weights || !out)))
        return stager_fail(MOE_ERR_INVALID_ARG, "moe_forward_offload: bad arguments");
    const size_t wbytes = moe_layer_weight_bytes(shape);
    if (wbytes == 0 || wbytes > st->slot_bytes)
        return stager_fail(MOE_ERR_INVALID_ARG,
                           "moe_forward_offload: a layer's weights do not fit a slot");
    if (compute == copy)
        return stager_fail(MOE_ERR_INVALID_ARG,
                           "moe_forward_offload: the copy stream must differ from the compute stream");
    cudaStream_t cs = (cudaStream_t)compute, ks = (cudaStream_t)copy;
    const int E = shape->E;
    const size_t per = (size_t)E * shape->I * shape->H;            // elements per matrix
    const size_t per_expert = (size_t)shape->I * shape->H * sizeof(moe_bf16);
    for (int l = 0; l < n_layers; ++l) {
        if (!host_weights[l] || !logits[l] || !out[l])
            return stager_fail(MOE_ERR_INVALID_ARG, "moe_forward_offload: NULL layer pointer");
        const void* view = nullptr;
        if (moe::device_view_of_host(host_weights[l], &view) != cudaSuccess ||
            reinterpret_cast<uintptr_t>(view) % 16)
            return stager_fail(MOE_ERR_INVALID_ARG,
                               "moe_forward_offload: host weights must be 16-byte aligned pinned "
                               "host memory");
    }
    if (n_layers == 0 || shape->T == 0) {
        moe::set_last_error("");
        return MOE_OK;
    }
    cudaError_t e = cudaSuccess;
    // 1. touched experts of every layer, written by the GPU into pinned
    // host flags (the previous call's readers are done: it synchronised).
    const size_t need = (size_t)n_layers * E;
    if (need > st->flags_cap) {
        if (st->flags_h) cudaFreeHost(st->flags_h);
        st->flags_h = nullptr;
        st->flags_d = nullptr;
        st->flags_cap = 0;
        void* h = nullptr;
        void* d = nullptr;
        if ((e = cudaHostAlloc(&h, need, cudaHostAllocMapped)) != cudaSuccess ||
            (e = cudaHostGetDevicePointer(&d, h, 0)) != cudaSuccess) {
            if (h) cudaFreeHost(h);
            moe::set_last_error("moe_forward_offload: %s", cudaGetErrorString(e));
            return MOE_ERR_CUDA;
        }
        st->flags_h = static_cast<uint8_t*>(h);
        st->flags_d = static_cast<uint8_t*>(d);
        st->flags_cap = need;
    }
    memset(st->flags_h, 0, need);
    for (int l = 0; l < n_layers; ++l) {
        const moe_status ms = moe::mark_touched_experts(shape, logits[l], ws, ws_bytes,
                                                        st->flags_d + (size_t)l * E, cs);
        if (ms != MOE_OK) return ms;
    }
    if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) {
        moe::set_last_error("moe_forward_offload: %s", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    // 2. copies of the touched experts and the layers' compute.
    for (int l = 0; l < n_layers; ++l) {
        const int s = l % st->n_slots;
        uint8_t* slot = st->slots + (size_t)s * st->slot_bytes;
        const uint8_t* touched = st->flags_h + (size_t)l * E;
        st->list.n = 0;
        for (int x = 0; x < E; ++x)
            if (touched[x]) {
                st->list.src_e[st->list.n] = x;
                st->list.dst_e[st->list.n] = x;
                ++st->list.n;
            }
        const void* src = nullptr;
        if (e == cudaSuccess) e = moe::device_view_of_host(host_weights[l], &src);   // checked above
        const size_t mat = per * sizeof(moe_bf16);
        const void* srcs[3] = {src, static_cast<const uint8_t*>(src) + mat,
                               static_cast<const uint8_t*>(src) + 2 * mat};
        void* dsts[3] = {slot, slot + mat, slot + 2 * mat};
        // The slot may be refilled only once the compute of its last layer
        // has finished (that event was recorded in an earlier iteration).
        if (e == cudaSuccess && l >= st->n_slots) e = cudaStreamWaitEvent(ks, st->freed[s], 0);
        if (e == cudaSuccess) e = moe::launch_expert_copy(st->list, srcs, dsts, per_expert, ks);
        if (e == cudaSuccess) e = cudaEventRecord(st->copied[s], ks);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, st->copied[s], 0);
        if (e != cudaSuccess) {
            moe::set_last_error("moe_forward_offload: %s", cudaGetErrorString(e));
            return MOE_ERR_CUDA;
        }
        const moe_bf16* Wg = reinterpret_cast<const moe_bf16*>(slot);
        const moe_status fs = moe_forward(shape, logits[l], x, Wg, Wg + per, Wg + 2 * per, out[l],
                                          nullptr, nullptr, ws, ws_bytes, compute);
        if (fs != MOE_OK) return fs;
        if ((e = cudaEventRecord(st->freed[s], cs)) != cudaSuccess) {
            moe::set_last_error("moe_forward_offload: %s", cudaGetErrorString(e));
            return MOE_ERR_CUDA;
        }
    }
    moe::set_last_error("");
    return MOE_OK;
}
