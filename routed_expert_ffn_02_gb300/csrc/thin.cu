// thin.cu -- weight-streaming expert path for experts holding fewer slots
// than the fat threshold (all experts in decode).
//
// In decode only a handful of experts per layer are touched per token
// (dsv41-flash-offload wiki, PCIe paragraph); each touched expert's weights
// are read from HBM once and applied to all (<= 32) of its slots.  The work is
// memory-bound: one warp owns one weight row, streams it with 16-byte
// coalesced loads, keeps one fp32 accumulator per slot in registers and
// finishes with warp-shuffle reductions.
//
//   gate/up: h[p, i] = bf16( silu(Wg[e,i,:] . x_t) * (Wu[e,i,:] . x_t) )
//   down:    y[p, r] = bf16( Wd[e,r,:] . h[p, :] )
// for every sorted position p of expert e (token t = perm[p] / k).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// One row i of expert e for its n (<= NT) slots.  xrow[t] = token row offsets
// (in uint4 units), held in shared memory by the calling warp.
template <int NT>
__device__ __forceinline__ void gate_up_row(const uint4* __restrict__ wg,
                                            const uint4* __restrict__ wu,
                                            const uint4* __restrict__ x,
                                            const int64_t* xrow, int n, int vec,
                                            float (&g)[NT], float (&u)[NT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < NT; ++t) { g[t] = 0.f; u[t] = 0.f; }
#pragma unroll 2
    for (int v = lane; v < vec; v += 32) {
        float fg[8], fu[8];
        bf16x8_to_f32(ldg_stream(wg + v), fg);
        bf16x8_to_f32(ldg_stream(wu + v), fu);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < n) {
                float fx[8];
                bf16x8_to_f32(__ldg(x + xrow[t] + v), fx);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    g[t] = fmaf(fg[q], fx[q], g[t]);
                    u[t] = fmaf(fu[q], fx[q], u[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < n) {
            g[t] = warp_sum(g[t]);
            u[t] = warp_sum(u[t]);
        }
    }
}

template <int NT>
__device__ __forceinline__ void down_row(const uint4* __restrict__ wd,
                                         const uint4* __restrict__ h,
                                         int64_t hrow0, int n, int vec,
                                         float (&acc)[NT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 2
    for (int v = lane; v < vec; v += 32) {
        float fw[8];
        bf16x8_to_f32(ldg_stream(wd + v), fw);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < n) {
                float fh[8];
                bf16x8_to_f32(__ldg(h + (hrow0 + t) * vec + v), fh);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[t] = fmaf(fw[q], fh[q], acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
        if (t < n) acc[t] = warp_sum(acc[t]);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

template <int NT>
__device__ __forceinline__ void gate_up_item(const uint4* wg, const uint4* wu,
                                             const uint4* x, const int64_t* xrow,
                                             int n, int vec, __nv_bfloat16* hcol,
                                             int64_t ldh) {
    float g[NT], u[NT];
    gate_up_row<NT>(wg, wu, x, xrow, n, vec, g, u);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < NT; ++t)
        if (t < n && lane == t) hcol[t * ldh] = __float2bfloat16_rn(silu_mul(g[t], u[t]));
}

template <int NT>
__device__ __forceinline__ void down_item(const uint4* wd, const uint4* h,
                                          int64_t hrow0, int n, int vec,
                                          __nv_bfloat16* ycol, int64_t ldy) {
    float acc[NT];
    down_row<NT>(wd, h, hrow0, n, vec, acc);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < NT; ++t)
        if (t < n && lane == t) ycol[t * ldy] = __float2bfloat16_rn(acc[t]);
}

// Work item = (thin expert q, weight row i); items are spread over all warps
// of a persistent grid so every SM streams weights.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
thin_gate_up_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                    const int32_t* __restrict__ offsets,
                    const int32_t* __restrict__ counts, int k, int H, int I,
                    const uint4* __restrict__ Wg, const uint4* __restrict__ Wu,
                    const int32_t* __restrict__ thin, const WsHeader* __restrict__ hdr,
                    __nv_bfloat16* __restrict__ h) {
    __shared__ int64_t xrow_s[kWarpsPerBlock][kThinMaxTokens];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t warp = (int64_t)blockIdx.x * kWarpsPerBlock + wib;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    const int64_t items = (int64_t)hdr->n_thin * I;
    const int vec = H / 8;
    int cur_q = -1;
    int e = 0, n = 0, row0 = 0;
    for (int64_t it = warp; it < items; it += nwarps) {
        const int q = (int)(it / I);
        const int i = (int)(it % I);
        if (q != cur_q) {
            cur_q = q;
            e = thin[q];
            n = min(counts[e], kThinMaxTokens);
            row0 = offsets[e];
            __syncwarp();
            if (lane < n) xrow_s[wib][lane] = (int64_t)(perm[row0 + lane] / k) * vec;
            __syncwarp();
        }
        const uint4* wg = Wg + ((int64_t)e * I + i) * vec;
        const uint4* wu = Wu + ((int64_t)e * I + i) * vec;
        __nv_bfloat16* hcol = h + (int64_t)row0 * I + i;
        const int64_t* xr = xrow_s[wib];
        if (n <= 1) gate_up_item<1>(wg, wu, x, xr, n, vec, hcol, I);
        else if (n <= 2) gate_up_item<2>(wg, wu, x, xr, n, vec, hcol, I);
        else if (n <= 4) gate_up_item<4>(wg, wu, x, xr, n, vec, hcol, I);
        else if (n <= 8) gate_up_item<8>(wg, wu, x, xr, n, vec, hcol, I);
        else if (n <= 16) gate_up_item<16>(wg, wu, x, xr, n, vec, hcol, I);
        else gate_up_item<32>(wg, wu, x, xr, n, vec, hcol, I);
    }
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
thin_down_kernel(const uint4* __restrict__ h, const int32_t* __restrict__ offsets,
                 const int32_t* __restrict__ counts, int H, int I,
                 const uint4* __restrict__ Wd, const int32_t* __restrict__ thin,
                 const WsHeader* __restrict__ hdr, __nv_bfloat16* __restrict__ y) {
    const int wib = threadIdx.x >> 5;
    const int64_t warp = (int64_t)blockIdx.x * kWarpsPerBlock + wib;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    const int64_t items = (int64_t)hdr->n_thin * H;
    const int vec = I / 8;
    for (int64_t it = warp; it < items; it += nwarps) {
        const int q = (int)(it / H);
        const int r = (int)(it % H);
        const int e = thin[q];
        const int n = min(counts[e], kThinMaxTokens);
        const int row0 = offsets[e];
        const uint4* wd = Wd + ((int64_t)e * H + r) * vec;
        __nv_bfloat16* ycol = y + (int64_t)row0 * H + r;
        if (n <= 1) down_item<1>(wd, h, row0, n, vec, ycol, H);
        else if (n <= 2) down_item<2>(wd, h, row0, n, vec, ycol, H);
        else if (n <= 4) down_item<4>(wd, h, row0, n, vec, ycol, H);
        else if (n <= 8) down_item<8>(wd, h, row0, n, vec, ycol, H);
        else if (n <= 16) down_item<16>(wd, h, row0, n, vec, ycol, H);
        else down_item<32>(wd, h, row0, n, vec, ycol, H);
    }
}

}  // namespace

cudaError_t launch_thin_gate_up(const __nv_bfloat16* x, const int32_t* perm,
                                const int32_t* offsets, const int32_t* counts,
                                int k, int H, int I, const __nv_bfloat16* Wg,
                                const __nv_bfloat16* Wu, const Plan& plan,
                                __nv_bfloat16* h, int num_sms, cudaStream_t s) {
    thin_gate_up_kernel<<<num_sms * 4, 32 * kWarpsPerBlock, 0, s>>>(
        reinterpret_cast<const uint4*>(x), perm, offsets, counts, k, H, I,
        reinterpret_cast<const uint4*>(Wg), reinterpret_cast<const uint4*>(Wu),
        plan.thin, plan.hdr, h);
    return cudaGetLastError();
}

cudaError_t launch_thin_down(const __nv_bfloat16* h, const int32_t* offsets,
                             const int32_t* counts, int H, int I,
                             const __nv_bfloat16* Wd, const Plan& plan,
                             __nv_bfloat16* y_sorted, int num_sms,
                             cudaStream_t s) {
    thin_down_kernel<<<num_sms * 4, 32 * kWarpsPerBlock, 0, s>>>(
        reinterpret_cast<const uint4*>(h), offsets, counts, H, I,
        reinterpret_cast<const uint4*>(Wd), plan.thin, plan.hdr, y_sorted);
    return cudaGetLastError();
}

}  // namespace moe
