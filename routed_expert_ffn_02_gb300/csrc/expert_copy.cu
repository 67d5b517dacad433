// expert_copy.cu -- expert weights from pinned host memory into device
// blocks by SM loads over the host link, one launch for a whole layer's list
// of experts.
//
// The offload design moves the experts a layer touches from host RAM into
// VRAM before the layer runs (dsv41-flash-offload wiki, overview: experts
// pinned in host RAM, copied into staging slots, one weight copy per batch
// for the experts with positive counts).  Measured on a GB300 with a Grace
// host: one large pinned copy crosses the host link at 211 GB/s whether the
// copy engine or SM loads drive it, but the copy engine reaches only
// ~170 GB/s over a layer's ~280 separate copies (one per run of touched
// experts and matrix).  A kernel whose CTAs keep ~2 MB of 16-byte loads in
// flight holds the link at its full rate for the whole list, needs one
// launch per layer, and shares the SMs with the layer compute at little
// cost: its CTAs take no shared memory and ~10K registers, so they fit
// beside a GEMM CTA on the same SM.
//
// Work items are 256 KB pieces of one expert's matrix, ordered (list entry,
// matrix, piece); CTA b takes items b, b + grid, ...  Each thread keeps 8
// loads in flight before storing them.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyCtas = 64;
constexpr int kCopyUnroll = 8;
constexpr int64_t kPieceVec = 16384;   // 16-byte vectors per work item (256 KB)

__global__ void __launch_bounds__(kCopyThreads)
expert_copy_kernel(const __grid_constant__ ExpertCopyList list, const uint4* __restrict__ src0,
                   const uint4* __restrict__ src1, const uint4* __restrict__ src2,
                   uint4* __restrict__ dst0, uint4* __restrict__ dst1, uint4* __restrict__ dst2,
                   int64_t vec) {
    const int64_t pieces = (vec + kPieceVec - 1) / kPieceVec;
    const int64_t items = (int64_t)list.n * 3 * pieces;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t p = it % pieces;
        const int64_t em = it / pieces;
        const int m = (int)(em % 3);
        const int j = (int)(em / 3);
        const uint4* s = (m == 0 ? src0 : m == 1 ? src1 : src2) + (int64_t)list.src_e[j] * vec;
        uint4* d = (m == 0 ? dst0 : m == 1 ? dst1 : dst2) + (int64_t)list.dst_e[j] * vec;
        const int64_t end = min(p * kPieceVec + kPieceVec, vec);
        int64_t i = p * kPieceVec + threadIdx.x;
        for (; i + (kCopyUnroll - 1) * kCopyThreads < end; i += kCopyUnroll * kCopyThreads) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) v[u] = __ldg(s + i + u * kCopyThreads);
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) d[i + u * kCopyThreads] = v[u];
        }
        for (; i < end; i += kCopyThreads) d[i] = __ldg(s + i);
    }
}

}  // namespace

cudaError_t device_view_of_host(const void* host, const void** dev) {
    *dev = nullptr;
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, host);
    if (e != cudaSuccess) return e;
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return cudaErrorInvalidValue;
    *dev = a.devicePointer;
    return cudaSuccess;
}

cudaError_t launch_expert_copy(const ExpertCopyList& list, const void* const src[3],
                               void* const dst[3], size_t expert_bytes, cudaStream_t s) {
    if (list.n < 0 || list.n > kMaxE || expert_bytes % 16) return cudaErrorInvalidValue;
    for (int m = 0; m < 3; ++m)
        if ((reinterpret_cast<uintptr_t>(src[m]) | reinterpret_cast<uintptr_t>(dst[m])) % 16)
            return cudaErrorInvalidValue;
    if (list.n == 0) return cudaSuccess;
    const int64_t vec = (int64_t)(expert_bytes / 16);
    const int64_t items = (int64_t)list.n * 3 * ((vec + kPieceVec - 1) / kPieceVec);
    const int grid = (int)std::min<int64_t>(kCopyCtas, items);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, expert_copy_kernel, list,
                              static_cast<const uint4*>(src[0]), static_cast<const uint4*>(src[1]),
                              static_cast<const uint4*>(src[2]), static_cast<uint4*>(dst[0]),
                              static_cast<uint4*>(dst[1]), static_cast<uint4*>(dst[2]), vec);
}

}  // namespace moe
