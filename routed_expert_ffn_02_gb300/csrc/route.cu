// route.cu -- top-k router kernel (one warp per token; the per-token
// selection and softmax are in route_dev.cuh) and the touched-expert marker
// used by the offload stager.
#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

template <int EPL>   // candidates per lane
__global__ void __launch_bounds__(256)
route_kernel(const float* __restrict__ logits, int T, int E, int k,
             int32_t* __restrict__ idx, float* __restrict__ gates) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    routing::route_row<EPL>(logits + t * (int64_t)E, E, k, idx + t * k, gates + t * k);
}

template <int EPL>
cudaError_t launch_epl(const float* logits, int T, int E, int k, int32_t* idx,
                       float* gates, cudaStream_t s) {
    const int warps_per_block = 8;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    return launch_pdl(route_kernel<EPL>, dim3(blocks), dim3(32 * warps_per_block), 0, s, logits,
                      T, E, k, idx, gates);
}

// flags[idx[s]] = 1 for every routed slot (every writer stores the same
// value, so the races are benign); indices outside [0, E) are skipped.
__global__ void __launch_bounds__(256)
mark_touched_kernel(const int32_t* __restrict__ idx, int64_t P, int E, uint8_t* flags) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < P;
         s += (int64_t)gridDim.x * blockDim.x) {
        const int e = idx[s];
        if ((unsigned)e < (unsigned)E) flags[e] = 1;
    }
}

}  // namespace

cudaError_t launch_mark_touched(const int32_t* idx, int64_t P, int E, uint8_t* flags,
                                cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((P + 255) / 256, 1024);
    return launch_pdl(mark_touched_kernel, dim3((unsigned)blocks), dim3(256), 0, s, idx, P, E,
                      flags);
}

cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int32_t* idx, float* gates, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    switch (routing::candidates_per_lane(E)) {
        case 1: return launch_epl<1>(logits, T, E, k, idx, gates, s);
        case 2: return launch_epl<2>(logits, T, E, k, idx, gates, s);
        case 4: return launch_epl<4>(logits, T, E, k, idx, gates, s);
        case 8: return launch_epl<8>(logits, T, E, k, idx, gates, s);
        case 12: return launch_epl<12>(logits, T, E, k, idx, gates, s);
        case 16: return launch_epl<16>(logits, T, E, k, idx, gates, s);
        case 24: return launch_epl<24>(logits, T, E, k, idx, gates, s);
        default: return launch_epl<32>(logits, T, E, k, idx, gates, s);
    }
}

}  // namespace moe
