// permute_noalloc.cu -- moe_permute_noalloc: the route-list kernels with
// their scratch in a fixed device array owned by the library, for callers
// that cannot allocate device memory.
//
// Who needs it: a serving process that hands every byte of HBM to the expert
// weights and the KV cache up front and keeps no pool to carve a workspace
// from, and host code that must not call cudaMalloc on its hot path because
// cudaMalloc can synchronise the whole device and stall the other streams.
// Such callers pass only inputs and outputs; the histogram and scan scratch
// lives in `g_permute_scratch` below.
//
// Costs and rules of the shared array:
//   * Every GPU that loads libmoe holds the array (kScratchBytes, about
//     1 MiB) until the process exits.
//   * All calls on a device share it and it keeps the previous call's
//     contents; each call clears the status word before its kernels run, and
//     the kernels overwrite every other byte they read.
//   * Calls whose kernels overlap on the GPU (different streams without
//     ordering between them) race on the array and give wrong results.
//   * Host code cannot use the array's name as a device address (on the host
//     it names a host-side shadow).  The device address is looked up once per
//     device with cudaGetSymbolAddress, with that device current, by the
//     first call made on it; make that first call before any stream capture.
//     A device reset (cudaDeviceReset) ends the context that address belongs
//     to: the next call on that device sees a new context and looks the
//     address up again (the lookup is keyed by the context's unique id).
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"

using namespace moe;

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if there is none).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

constexpr int64_t kNoallocMaxSlots = 262144;   // T * k
constexpr int64_t kNoallocMaxChunks = kNoallocMaxSlots / kPermChunk;
constexpr size_t kScratchInts = (size_t)2 * kNoallocMaxChunks * kMaxE;
constexpr size_t kScratchBytes = sizeof(WsHeader) + kScratchInts * sizeof(int32_t);

// [WsHeader | chunk_hist | chunk_base]
static __device__ __align__(256) unsigned char g_permute_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // context id of the address

}  // namespace

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_idx, int32_t T, int32_t E,
                                          int32_t k, int32_t* counts, int32_t* offsets,
                                          int32_t* perm, int32_t* inv_perm,
                                          int32_t* device_status, moe_stream_t stream) {
    auto fail = [](moe_status st, const char* msg) {
        set_last_error("moe_permute_noalloc: %s", msg);
        return st;
    };
    set_last_error("");
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E)
        return fail(MOE_ERR_INVALID_ARG, "T, E or k outside the limits of moe_permute");
    const int64_t P = (int64_t)T * k;
    if (P > kNoallocMaxSlots)
        return fail(MOE_ERR_UNSUPPORTED,
                    "T*k exceeds the 262144 slots its fixed scratch holds; use moe_permute");
    if (!counts || !offsets || (P > 0 && (!topk_idx || !perm || !inv_perm)))
        return fail(MOE_ERR_INVALID_ARG, "NULL pointer");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ERR_UNSUPPORTED, "device ordinal beyond the 64 devices it keeps scratch "
                                         "addresses for");
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const unsigned long long ctx = current_context_id();
        if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
            if (e != cudaSuccess || !p) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
            g_scratch_addr[dev] = p;
            // the lookup made the device's context current if it was not yet
            g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
        }
        base = g_scratch_addr[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    WsHeader* hdr = static_cast<WsHeader*>(base);
    int32_t* chunk_hist = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(base) +
                                                     sizeof(WsHeader));
    const int64_t nch = (P + kPermChunk - 1) / kPermChunk;
    int32_t* chunk_base = chunk_hist + nch * E;

    // The status word must start at zero; everything else is overwritten.
    if (cudaMemsetAsync(&hdr->status, 0, sizeof(int32_t), s) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    cudaError_t e = launch_permute(topk_idx, T, E, k, counts, offsets, perm, inv_perm,
                                   chunk_hist, chunk_base, hdr, nullptr, s);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    if (device_status &&
        cudaMemcpyAsync(device_status, &hdr->status, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        s) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "cudaMemcpyAsync of the status word failed");
    return MOE_OK;
}
