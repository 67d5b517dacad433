// route_dev.cuh -- the per-token top-k router, shared by the router kernel
// and the streaming kernels that route small batches themselves.
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
// next expert to select: each round takes every lane's largest key (a
// pairwise tree), the warp maximum of their high halves, then the maximum low
// half among the lanes that hold that high half (two redux.sync warp
// reductions), and the owner retires it; k rounds give the top k in output
// order.  Key 0 marks an empty or already-taken candidate and sorts below
// every real logit, including -inf.
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace routing {

__device__ __forceinline__ uint32_t float_order(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u & 0x7fffffffu) == 0u) u = 0u;                 // -0.0 == +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_to_float(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// One warp routes one token: writes idx[0, k) (experts in selection order)
// and gates[0, k).  All 32 lanes call it together.  The selection rounds are
// a loop (lane r keeps the r-th winner), so the routine stays a few hundred
// instructions long: it runs once per launch inside much larger kernels,
// where an unrolled copy cost more in instruction fetch than in arithmetic;
// and each round is two warp reductions deep rather than a five-step
// shuffle tree of 64-bit keys.
template <int EPL>   // candidates per lane
__device__ __forceinline__ void route_row(const float* __restrict__ row, int E, int k,
                                          int32_t* __restrict__ idx, float* __restrict__ gates) {
    const int lane = threadIdx.x & 31;
    uint64_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? ((uint64_t)float_order(__ldg(row + e)) << 32) |
                               (uint64_t)(~(uint32_t)e)
                         : 0ull;
    }

    float sel_val = 0.f;   // lane r < k: the r-th selected logit and its expert
    int sel_idx = 0;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        uint64_t t[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) t[j] = key[j];
#pragma unroll
        for (int span = 1; span < EPL; span *= 2)
#pragma unroll
            for (int j = 0; j + span < EPL; j += 2 * span) t[j] = t[j + span] > t[j] ? t[j + span] : t[j];
        const uint32_t hi = (uint32_t)(t[0] >> 32), lo = (uint32_t)t[0];
        const uint32_t best_hi = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t best_lo = __reduce_max_sync(0xffffffffu, hi == best_hi ? lo : 0u);
        const uint64_t best = ((uint64_t)best_hi << 32) | best_lo;
        // The owner retires the winner (keys are unique: indices differ).
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (key[j] == best) key[j] = 0ull;
        if (lane == r) {
            sel_val = order_to_float(best_hi);
            sel_idx = (int)(~best_lo);
        }
    }

    // Softmax over the selection, relative to the largest selected logit; the
    // denominator sums the k weights in selection order.
    const float m = __shfl_sync(0xffffffffu, sel_val, 0);
    const float w = (lane < k) ? expf(sel_val - m) : 0.f;
    float denom = 0.f;
#pragma unroll 1
    for (int r = 0; r < k; ++r) denom += __shfl_sync(0xffffffffu, w, r);
    // Lane r writes output r (coalesced).
    if (lane < k) {
        idx[lane] = sel_idx;
        gates[lane] = w / denom;
    }
}

// Candidates per lane for E experts: the smallest of 1, 2, 4, 8, 12, 16, 24,
// 32 that covers E (E <= 1024).
inline int candidates_per_lane(int E) {
    const int epl = (E + 31) / 32;
    const int steps[] = {1, 2, 4, 8, 12, 16, 24, 32};
    for (int v : steps)
        if (epl <= v) return v;
    return 32;
}

}  // namespace routing
}  // namespace moe
