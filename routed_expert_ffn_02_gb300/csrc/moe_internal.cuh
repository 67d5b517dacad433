// moe_internal.cuh -- shared definitions of libmoe's CUDA translation units:
// limits, the workspace header, and the launchers each stage exports to the
// C ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe.h"

namespace moe {

constexpr int kMaxK = 8;             // experts per token
constexpr int kMaxE = 1024;          // experts per layer
constexpr int kThinMaxTokens = 32;   // slots one weight-streaming expert may hold
constexpr int kPermChunk = 2048;     // slots per block in the route-list kernels
constexpr int kTileM = 128;          // rows (slots) per grouped-GEMM tile

// First 256 bytes of every workspace.
struct WsHeader {
    int32_t status;        // moe_status recorded by kernels (sticky)
    int32_t n_fat_tiles;   // grouped-GEMM row tiles built by the planner
    int32_t n_thin;        // experts on the weight-streaming path
    int32_t reserved[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// One grouped-GEMM row tile: rows [row0, row0 + rows) of expert `expert`
// in sorted-slot order.
struct FatTile {
    int32_t expert;
    int32_t row0;
    int32_t rows;
    int32_t pad;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Planner outputs (the split of experts between the two expert paths).
struct Plan {
    FatTile* tiles;     // [max_fat_tiles(P, E)]
    int32_t* thin;      // [E] experts on the weight-streaming path, ascending
    WsHeader* hdr;
    int32_t fat_threshold;
};

inline int64_t max_fat_tiles(int64_t P, int E) { return P / kTileM + E + 1; }

// Launchers (all asynchronous on `s`; they return the launch's cudaError_t).
cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int32_t* idx, float* gates, cudaStream_t s);

// Route lists; when plan != nullptr the planner runs in the same kernels.
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, int32_t* chunk_hist,
                           int32_t* chunk_base, WsHeader* hdr,
                           const Plan* plan, cudaStream_t s);
size_t permute_scratch_ints(int64_t P, int E);   // chunk_hist + chunk_base

cudaError_t launch_plan(const int32_t* counts, const int32_t* offsets, int E,
                        const Plan& plan, cudaStream_t s);

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* perm, int k,
                          int H, const Plan& plan, __nv_bfloat16* x_sorted,
                          int num_sms, cudaStream_t s);

cudaError_t launch_thin_gate_up(const __nv_bfloat16* x, const int32_t* perm,
                                const int32_t* offsets, const int32_t* counts,
                                int k, int H, int I, const __nv_bfloat16* Wg,
                                const __nv_bfloat16* Wu, const Plan& plan,
                                __nv_bfloat16* h, int num_sms, cudaStream_t s);

cudaError_t launch_thin_down(const __nv_bfloat16* h, const int32_t* offsets,
                             const int32_t* counts, int H, int I,
                             const __nv_bfloat16* Wd, const Plan& plan,
                             __nv_bfloat16* y_sorted, int num_sms,
                             cudaStream_t s);

// Grouped GEMMs on tcgen05.  gate_up: h = silu(A Wg^T) * (A Wu^T) for the
// fat tiles, A = x_sorted [rows_alloc, H].  down: y = h Wd^T, A = h.
cudaError_t launch_gemm_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                                int E, int H, int I, const Plan& plan,
                                __nv_bfloat16* h, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_down(const __nv_bfloat16* h, int64_t rows_alloc,
                             const __nv_bfloat16* Wd, int E, int H, int I,
                             const Plan& plan, __nv_bfloat16* y_sorted,
                             int num_sms, cudaStream_t s);

cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* inv_perm,
                           const float* gates, int T, int k, int H,
                           __nv_bfloat16* out, int num_sms, cudaStream_t s);

// Sets the calling thread's moe_last_error() message (printf format).
void set_last_error(const char* fmt, ...);

// Records a device-side condition in the workspace status word (first one wins).
__device__ __forceinline__ void set_status(WsHeader* hdr, int code) {
    atomicCAS(&hdr->status, 0, code);
}

}  // namespace moe
