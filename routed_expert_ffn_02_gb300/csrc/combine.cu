// combine.cu -- gate-weighted un-permute ("split/combine on GPU",
// dsv41-flash-offload wiki, file map):
//   out[t] = bf16( sum_{j<k} gates[t,j] * y_sorted[inv_perm[t*k + j]] )
// fp32 accumulation in ascending j, no atomics, so repeated runs are
// bit-identical (combine_dev.cuh).  One block per token row (grid-stride),
// 16-byte vectors.
#include "moe_internal.cuh"
#include "combine_dev.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ inv_perm,
               const float* __restrict__ gates, int T, int k, int H,
               uint4* __restrict__ out) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int vec = H / 8;
    auto load = [&](int64_t i) { return __ldg(y + i); };
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        int64_t src[kMaxK];
        float g[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            src[j] = (j < k) ? (int64_t)inv_perm[t * k + j] * vec : 0;
            g[j] = (j < k) ? gates[t * k + j] : 0.f;
        }
        for (int v = threadIdx.x; v < vec; v += blockDim.x)
            out[t * vec + v] = combine_vec(load, src, g, k, v);
    }
}

}  // namespace

cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* inv_perm,
                           const float* gates, int T, int k, int H,
                           __nv_bfloat16* out, int num_sms, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>(T, (int64_t)num_sms * 8);
    return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, s,
                      reinterpret_cast<const uint4*>(y_sorted), inv_perm, gates, T, k, H,
                      reinterpret_cast<uint4*>(out));
}

}  // namespace moe
