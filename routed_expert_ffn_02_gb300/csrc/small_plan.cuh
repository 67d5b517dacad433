// small_plan.cuh -- routing, route lists and weight-streaming units of a
// small batch (at most kSelfRouteSlots token slots), computed by every CTA of
// a streaming kernel in its own shared memory (see SelfRoute).
//
// The results are those of the router, route-list and planner kernels for
// the same batch: the top-k and gates come from the same per-token routine
// (route_dev.cuh); the route lists are the stable counting sort of the slots
// s = t*k + j by expert (position of a slot = number of slots with a smaller
// (expert, s) key, the keys being distinct); each touched expert is one unit
// of all its slots, in ascending expert order, priced by thin_unit_cost.
#pragma once

#include "combine_dev.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_dev.cuh"

namespace moe {

struct SmallPlan {
    int32_t idx[kSelfRouteSlots];       // slot -> expert
    float gates[kSelfRouteSlots];       // slot -> gate
    int32_t perm[kSelfRouteSlots];      // sorted position -> slot
    int32_t inv_perm[kSelfRouteSlots];  // slot -> sorted position
    ThinUnit units[kSelfRouteSlots];    // one per touched expert
    int32_t n_units;
    int32_t weight;                     // sum of thin_unit_cost over the units
};

// One warp routes one token row (all 32 lanes call it), with the candidates
// per lane the router kernel uses for E.
static __device__ __noinline__ void route_token(const float* row, int E, int k, int32_t* idx,
                                                float* gates) {
    const int epl = (E + 31) / 32;
    if (epl <= 1) routing::route_row<1>(row, E, k, idx, gates);
    else if (epl <= 2) routing::route_row<2>(row, E, k, idx, gates);
    else if (epl <= 4) routing::route_row<4>(row, E, k, idx, gates);
    else if (epl <= 8) routing::route_row<8>(row, E, k, idx, gates);
    else if (epl <= 12) routing::route_row<12>(row, E, k, idx, gates);
    else if (epl <= 16) routing::route_row<16>(row, E, k, idx, gates);
    else if (epl <= 24) routing::route_row<24>(row, E, k, idx, gates);
    else routing::route_row<32>(row, E, k, idx, gates);
}

// Called by every thread of the block.  Warp w routes tokens w, w + warps,
// ...; then warp 0 (lane = slot, later lane = sorted position) builds the
// route lists and the units.  Requires T * k <= kSelfRouteSlots and E <= 1024.
__device__ inline void build_small_plan(const SelfRoute& sr, SmallPlan& sp) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_warps = blockDim.x >> 5;
    for (int t = warp; t < sr.T; t += n_warps)
        route_token(sr.logits + (int64_t)t * sr.E, sr.E, sr.k, sp.idx + t * sr.k,
                    sp.gates + t * sr.k);
    __syncthreads();
    if (warp == 0) {
        const int P = sr.T * sr.k;
        const bool live = lane < P;
        // key = expert * 32 + slot: distinct, ordered by (expert, slot)
        const uint32_t key = live ? ((uint32_t)sp.idx[lane] << 5) | (uint32_t)lane : 0xffffffffu;
        int pos = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) pos += __shfl_sync(0xffffffffu, key, j) < key ? 1 : 0;
        if (live) {
            sp.perm[pos] = lane;
            sp.inv_perm[lane] = pos;
        }
        __syncwarp();
        // lane p: sorted position p; a unit starts where the expert changes
        const int e = live ? sp.idx[sp.perm[lane]] : -1;
        const int e_prev = __shfl_up_sync(0xffffffffu, e, 1);
        const bool head = live && (lane == 0 || e_prev != e);
        const unsigned heads = __ballot_sync(0xffffffffu, head);
        const unsigned later = lane < 31 ? heads & ~((2u << lane) - 1u) : 0u;
        const int n = (later ? __ffs(later) - 1 : P) - lane;
        const int cost = head ? thin_unit_cost(n) : 0;
        int incl = cost;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (head) {
            ThinUnit u;
            u.expert = e;
            u.row0 = lane;
            u.n = n;
            u.cost_before = incl - cost;
            sp.units[__popc(heads & ((1u << lane) - 1u))] = u;
        }
        if (lane == 31) {
            sp.n_units = __popc(heads);
            sp.weight = incl;
        }
    }
    __syncthreads();
}

// Called by every thread of one block: writes the batch's router outputs,
// route lists, units and planner counts where the router, route-list and
// planner kernels would have written them (on_mma: the units are the
// tensor-core streaming kernel's tiles, one per expert with all its slots).
__device__ inline void write_small_plan(const SelfRoute& sr, const SmallPlan& sp, WsHeader* hdr,
                                        bool on_mma = false) {
    const int P = sr.T * sr.k;
    for (int s = threadIdx.x; s < P; s += blockDim.x) {
        sr.idx[s] = sp.idx[s];
        sr.gates[s] = sp.gates[s];
        sr.perm[s] = sp.perm[s];
        sr.inv_perm[s] = sp.inv_perm[s];
    }
    for (int u = threadIdx.x; u < sp.n_units; u += blockDim.x) sr.units[u] = sp.units[u];
    for (int e = threadIdx.x; e <= sr.E; e += blockDim.x) {
        int c = 0, before = 0;
        for (int s = 0; s < P; ++s) {
            c += sp.idx[s] == e ? 1 : 0;
            before += sp.idx[s] < e ? 1 : 0;
        }
        if (e < sr.E) sr.counts[e] = c;
        sr.offsets[e] = before;   // offsets[E] = P
    }
    if (threadIdx.x == 0) {
        hdr->ticket = 0;   // the down kernel's fused combine counts CTAs on it
        hdr->n_fat_tiles = 0;
        hdr->n_thin = on_mma ? 0 : sp.n_units;
        hdr->thin_weight = on_mma ? 0 : sp.weight;
        hdr->n_thin_mma = on_mma ? sp.n_units : 0;
        hdr->n_solo = 0;
    }
}

// Called by every thread of the block, after the kernel that ran
// write_small_plan has completed: the batch's units, gates and route lists
// back into shared memory (only what the streaming down kernel and its fused
// combine read).  The unit list holds at least min(E, T*k) entries.
__device__ inline void load_small_plan(const SelfRoute& sr, const WsHeader* hdr, SmallPlan& sp) {
    const int P = sr.T * sr.k;
    const int nu = P < sr.E ? P : sr.E;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        sp.gates[i] = sr.gates[i];
        sp.inv_perm[i] = sr.inv_perm[i];
        if (i < nu) sp.units[i] = sr.units[i];
    }
    if (threadIdx.x == 0) {
        sp.n_units = hdr->n_thin > 0 ? hdr->n_thin : hdr->n_thin_mma;
        sp.weight = hdr->thin_weight;
    }
    __syncthreads();
}

// The last CTA of a streaming down kernel to finish combines the batch.
// Called by every thread of the block once its y rows are stored: each
// thread fences its stores, the CTA takes a ticket from the workspace header
// (zeroed by the gate/up kernel, and again by the CTA that takes the last
// ticket), and the CTA with the last ticket reads every CTA's rows (through
// L2) and writes out.  No thread waits on another CTA.
__device__ inline void combine_if_last(const SelfRoute& sr, const SmallPlan& sp, WsHeader* hdr,
                                       const __nv_bfloat16* y_sorted, int H);

// Called by every thread of one block: out[t] for every token of the batch,
// from y_sorted rows written by other CTAs of the same kernel (read through
// L2) and the batch's gates and route lists in sp.  The batch's T * H / 8
// output vectors are taken two per thread per pass, with the 2k row loads of
// both issued before either is summed (combine_vals: the combine kernel's
// arithmetic).
__device__ inline void combine_small(const SelfRoute& sr, const SmallPlan& sp,
                                     const __nv_bfloat16* y_sorted, int H) {
    const int vec = H / 8, k = sr.k;
    const int n = sr.T * vec;
    const uint4* y = reinterpret_cast<const uint4*>(y_sorted);
    uint4* out = reinterpret_cast<uint4*>(sr.out);
    for (int i0 = threadIdx.x; i0 < n; i0 += 2 * (int)blockDim.x) {
        const int i1 = i0 + (int)blockDim.x;
        const bool two = i1 < n;
        const int t0 = i0 / vec, v0 = i0 - t0 * vec;
        const int t1 = two ? i1 / vec : t0, v1 = two ? i1 - t1 * vec : v0;
        uint4 r0[kMaxK], r1[kMaxK];
        float g0[kMaxK], g1[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                r0[j] = __ldcg(y + (int64_t)sp.inv_perm[t0 * k + j] * vec + v0);
                r1[j] = __ldcg(y + (int64_t)sp.inv_perm[t1 * k + j] * vec + v1);
                g0[j] = sp.gates[t0 * k + j];
                g1[j] = sp.gates[t1 * k + j];
            } else {
                g0[j] = g1[j] = 0.f;
            }
        }
        out[i0] = combine_vals(r0, g0, k);
        if (two) out[i1] = combine_vals(r1, g1, k);
    }
}

__device__ inline void combine_if_last(const SelfRoute& sr, const SmallPlan& sp, WsHeader* hdr,
                                       const __nv_bfloat16* y_sorted, int H) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        s_last = atomicAdd(&hdr->ticket, 1) == (int)gridDim.x - 1;
        // Every CTA has taken its ticket: the last one sets the counter back
        // to zero at once, so a step never leaves a count behind for the
        // next one (whose gate/up kernel zeroes it as well).
        if (s_last) atomicExch(&hdr->ticket, 0);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        combine_small(sr, sp, y_sorted, H);
    }
}

// The combine of a cooperative launch (every CTA resident): each CTA fences
// its y rows and arrives on the workspace's layer_sync counter (monotonic,
// like the one-launch layer's first grid-wide wait); thread 0 waits, bounded,
// for the whole grid, and then the CTA combines its own share of the batch's
// T*H/8 output vectors with the combine kernel's arithmetic (combine_vals).
// Each CTA loads a few vectors once, instead of one CTA loading all of them.
// inv_perm / gates: [T*k], shared (the batch's own plan) or global memory.
__device__ inline void combine_spread(const SelfRoute& sr, const int32_t* inv_perm,
                                      const float* gates, WsHeader* hdr,
                                      const __nv_bfloat16* y_sorted, int H,
                                      long long wait_cycles) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t seen = atomicAdd(&hdr->layer_sync, 1u);
        const uint32_t target = (seen / gridDim.x + 1) * gridDim.x;
        const long long t0 = clock64();
        while ((int32_t)(ptx::ld_acquire_gpu(&hdr->layer_sync) - target) < 0) {
            if (clock64() - t0 > wait_cycles) {
                set_status(hdr, MOE_ERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
    }
    __syncthreads();
    const int vec = H / 8, k = sr.k;
    const int n = sr.T * vec;
    const int i_end = (int)((int64_t)n * (blockIdx.x + 1) / gridDim.x);
    const uint4* y = reinterpret_cast<const uint4*>(y_sorted);
    uint4* out = reinterpret_cast<uint4*>(sr.out);
    for (int i = (int)((int64_t)n * blockIdx.x / gridDim.x) + (int)threadIdx.x; i < i_end;
         i += (int)blockDim.x) {
        const int t = i / vec, v = i - t * vec;
        uint4 r[kMaxK];
        float g[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                r[j] = __ldcg(y + (int64_t)inv_perm[t * k + j] * vec + v);
                g[j] = gates[t * k + j];
            } else {
                g[j] = 0.f;
            }
        }
        out[i] = combine_vals(r, g, k);
    }
}

}  // namespace moe
