// combine_dev.cuh -- one 16-byte output vector of the gate-weighted
// un-permute ("split/combine on GPU", dsv41-flash-offload wiki, file map):
//   out[t][8v .. 8v+7] = bf16( sum_{j<k} g[j] * y_sorted[src[j] + v] )
// fp32 fmaf in ascending j from 0, round to nearest even at the end.  Shared
// by the combine kernel and the fused combine of the small-batch streaming
// down kernel, so both give the same bits.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// r[j]: the 16-byte vector of slot j's y row (j < k); g[j]: its gate.
__device__ __forceinline__ uint4 combine_vals(const uint4 (&r)[kMaxK], const float (&g)[kMaxK],
                                              int k) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&r[j]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(p[q]);
                acc[2 * q] = fmaf(g[j], f.x, acc[2 * q]);
                acc[2 * q + 1] = fmaf(g[j], f.y, acc[2 * q + 1]);
            }
        }
    }
    uint4 o;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) po[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    return o;
}

// load(i): 16-byte vector i of y_sorted; src[j]: first vector of slot j's row.
template <typename Load>
__device__ __forceinline__ uint4 combine_vec(Load load, const int64_t (&src)[kMaxK],
                                             const float (&g)[kMaxK], int k, int64_t v) {
    uint4 r[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
        if (j < k) r[j] = load(src[j] + v);
    return combine_vals(r, g, k);
}

}  // namespace moe
