// route.cu -- top-k router: one warp per token.
//
// Each token is routed to k of the layer's E experts (dsv41-flash-offload
// wiki, overview).  Selection compares raw fp32 logits under the total order
// (value descending, index ascending), so it is exact and needs no
// arithmetic; gates are a softmax over the k selected logits in fp32.
//
// Each lane holds ceil(E/32) candidates as 64-bit keys
//   key = order(value) << 32 | ~index
// where order() maps fp32 to an unsigned integer with the same ordering
// (-0.0 folded onto +0.0, since they compare equal).  The largest key is the
// next expert to select; k rounds of a warp max-reduction pick the top k in
// output order.  Key 0 marks an empty or already-taken candidate and sorts
// below every real logit, including -inf.
#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t float_order(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u & 0x7fffffffu) == 0u) u = 0u;                 // -0.0 == +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_to_float(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

template <int EPL>   // candidates per lane
__global__ void __launch_bounds__(256)
route_kernel(const float* __restrict__ logits, int T, int E, int k,
             int32_t* __restrict__ idx, float* __restrict__ gates) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + t * (int64_t)E;

    uint64_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? ((uint64_t)float_order(__ldg(row + e)) << 32) |
                               (uint64_t)(~(uint32_t)e)
                         : 0ull;
    }

    float sel_val[kMaxK];
    int sel_idx[kMaxK];
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
        sel_val[r] = 0.f;
        sel_idx[r] = 0;
        if (r < k) {
            uint64_t best = 0ull;
#pragma unroll
            for (int j = 0; j < EPL; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
                best = o > best ? o : best;
            }
            // The owner retires the winner (keys are unique: indices differ).
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (key[j] == best) key[j] = 0ull;
            sel_val[r] = order_to_float((uint32_t)(best >> 32));
            sel_idx[r] = (int)(~(uint32_t)(best & 0xffffffffull));
        }
    }

    // Softmax over the selection, relative to the largest selected logit.
    const float m = sel_val[0];
    float w[kMaxK];
    float denom = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
        w[r] = (r < k) ? expf(sel_val[r] - m) : 0.f;
        denom += w[r];
    }
    // Lane r writes output r (coalesced).
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
        if (r < k && lane == r) {
            idx[t * k + r] = sel_idx[r];
            gates[t * k + r] = w[r] / denom;
        }
    }
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
    const int epl = (E + 31) / 32;
    if (epl <= 1) return launch_epl<1>(logits, T, E, k, idx, gates, s);
    if (epl <= 2) return launch_epl<2>(logits, T, E, k, idx, gates, s);
    if (epl <= 4) return launch_epl<4>(logits, T, E, k, idx, gates, s);
    if (epl <= 8) return launch_epl<8>(logits, T, E, k, idx, gates, s);
    if (epl <= 12) return launch_epl<12>(logits, T, E, k, idx, gates, s);
    if (epl <= 16) return launch_epl<16>(logits, T, E, k, idx, gates, s);
    if (epl <= 24) return launch_epl<24>(logits, T, E, k, idx, gates, s);
    return launch_epl<32>(logits, T, E, k, idx, gates, s);
}

}  // namespace moe
