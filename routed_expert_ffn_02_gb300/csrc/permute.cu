// permute.cu -- per-expert route lists: histogram, exclusive scan and a
// stable counting-sort scatter of the T*k token slots (slot s = t*k + j),
// plus the planner that splits experts between the grouped GEMM ("busy"
// experts, >= fat threshold slots) and the weight-streaming path, and the
// row gather that feeds the GEMM.
//
// Route lists with positive counts come from the dsv41-flash-offload wiki
// (file map); the busy/fat split with threshold 32 from the model page's
// launch flags.  Stability (slots ascending within an expert) makes the
// result unique, so it is bit-exact against a textbook counting sort.
//
// Large inputs (P = T*k > kPermChunk) take three kernels:
//   hist    one block per chunk of kPermChunk slots -> chunk_hist[c][e]
//   scan    one block: chunk_base[c][e] = sum_{c'<c} chunk_hist[c'][e],
//           counts, offsets (+ planner)
//   scatter one block per chunk; warp w owns a contiguous sub-chunk; ranks
//           inside a warp come from __match_any_sync, so the order of slots
//           of one expert is kept.
// Small inputs (decode) take one single-block kernel doing all of it.
#include "gather_dev.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kScatterWarps = 8;
constexpr int kSlotsPerWarp = kPermChunk / kScatterWarps;   // 256

// Exclusive scan, in place, of a[0, n) held in shared memory by a block of
// NT threads; returns the total to every thread.  ws: shared int[33].
template <int NT>
__device__ int block_exclusive_scan(int* a, int n, int* ws) {
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
    const int per = (n + NT - 1) / NT;
    const int beg = min(n, (int)threadIdx.x * per);
    const int end = min(n, beg + per);
    int local = 0;
    for (int i = beg; i < end; ++i) local += a[i];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) ws[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int v = (lane < NT / 32) ? ws[lane] : 0;
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += u;
        }
        if (lane < NT / 32) ws[lane] = inc - v;
        if (lane == 31) ws[32] = inc;
    }
    __syncthreads();
    int run = ws[w] + incl - local;
    for (int i = beg; i < end; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    const int total = ws[32];
    __syncthreads();
    return total;
}

// Planner: fat experts (count >= threshold, count > 0) get 2*ceil(count/256)
// row tiles of up to 128 rows; thin experts (0 < count < threshold) with at least thin_mma_min
// slots get one tile for the tensor-core streaming kernel; the other thin
// experts get ceil(count/unit_tokens) CUDA-core streaming units, each with the
// running sum of unit costs before it (thin_unit_cost) so that kernel can
// split rows evenly by cost.
// cnt/off: shared copies of counts/offsets; ta, tb: shared int[E] scratch.
template <int NT>
__device__ void block_plan(const int* cnt, const int* off, int E, const Plan& plan,
                           int* ta, int* tb, int* ws) {
    const int thr = plan.fat_threshold;
    const int nu = plan.unit_tokens;
    const int mma_min = plan.thin_mma_min;
    auto is_fat = [&](int c) { return c > 0 && c >= thr; };
    auto is_mma = [&](int c) { return c > 0 && c < thr && c >= mma_min; };
    auto is_unit = [&](int c) { return c > 0 && c < thr && c < mma_min; };
    // A fat expert's 128-row tiles come in pairs (tiles 2q and 2q+1 cover
    // rows [256q, 256q+128) and [256q+128, 256q+256)), so the grouped GEMM
    // can run each pair on a CTA pair.  An expert with a single tile (at most
    // 128 slots) is a solo tile for the one-CTA GEMM; an expert with an odd
    // number of tiles above one pads its last pair with an empty tile (a solo
    // tile there would read the expert's weights from DRAM a second time).
    auto n_tiles_of = [](int c) { return (c + kTileM - 1) / kTileM; };
    auto is_solo = [&](int c) { return is_fat(c) && n_tiles_of(c) == 1; };
    auto paired_of = [&](int c) { return (is_fat(c) && !is_solo(c)) ? (n_tiles_of(c) + 1) & ~1 : 0; };
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = cnt[e];
        ta[e] = paired_of(c);
        tb[e] = is_mma(c) ? 1 : 0;
    }
    __syncthreads();
    const int n_tiles = block_exclusive_scan<NT>(ta, E, ws);
    const int n_mma = block_exclusive_scan<NT>(tb, E, ws);
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = cnt[e];
        if (paired_of(c) > 0) {
            const int nt = paired_of(c);
            for (int i = 0; i < nt; ++i) {
                FatTile ft;
                ft.expert = e;
                ft.row0 = off[e] + i * kTileM;
                ft.rows = max(0, min(kTileM, c - i * kTileM));
                ft.pad = 0;
                plan.tiles[ta[e] + i] = ft;
            }
        } else if (is_mma(c)) {
            FatTile ft;
            ft.expert = e;
            ft.row0 = off[e];
            ft.rows = c;
            ft.pad = 0;
            plan.mma_tiles[tb[e]] = ft;
        }
    }
    __syncthreads();
    // solo tiles: fat experts with a single tile
    for (int e = threadIdx.x; e < E; e += NT) ta[e] = is_solo(cnt[e]) ? 1 : 0;
    __syncthreads();
    const int n_solo = block_exclusive_scan<NT>(ta, E, ws);
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = cnt[e];
        if (is_solo(c)) {
            FatTile ft;
            ft.expert = e;
            ft.row0 = off[e];
            ft.rows = c;
            ft.pad = 0;
            plan.solo_tiles[ta[e]] = ft;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = cnt[e];
        tb[e] = is_unit(c) ? (c + nu - 1) / nu : 0;
        // unit costs of the expert, scanned below
        int w = 0;
        if (is_unit(c))
            for (int i = 0; i * nu < c; ++i) w += thin_unit_cost(min(nu, c - i * nu));
        ta[e] = w;
    }
    __syncthreads();
    const int n_units = block_exclusive_scan<NT>(tb, E, ws);
    const int weight = block_exclusive_scan<NT>(ta, E, ws);
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = cnt[e];
        if (is_unit(c)) {
            int before = ta[e];
            for (int i = 0; i * nu < c; ++i) {
                ThinUnit u;
                u.expert = e;
                u.row0 = off[e] + i * nu;
                u.n = min(nu, c - i * nu);
                u.cost_before = before;
                before += thin_unit_cost(u.n);
                plan.units[tb[e] + i] = u;
            }
        }
    }
    if (threadIdx.x == 0) {
        plan.hdr->n_fat_tiles = n_tiles;
        plan.hdr->n_thin = n_units;
        plan.hdr->thin_weight = weight;
        plan.hdr->n_thin_mma = n_mma;
        plan.hdr->n_solo = n_solo;
    }
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---- large path -------------------------------------------------------

__global__ void __launch_bounds__(256)
hist_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
            int32_t* __restrict__ chunk_hist, WsHeader* hdr) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int h[kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int64_t beg = (int64_t)blockIdx.x * kPermChunk;
    const int64_t end = min(P, beg + kPermChunk);
    for (int64_t s = beg + threadIdx.x; s < end; s += blockDim.x) {
        const int e = idx[s];
        if ((unsigned)e < (unsigned)E) atomicAdd(&h[e], 1);
        else set_status(hdr, MOE_ERR_BAD_INDEX);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_hist[(int64_t)blockIdx.x * E + e] = h[e];
}

__global__ void __launch_bounds__(1024)
scan_kernel(const int32_t* __restrict__ chunk_hist, int nchunks, int E,
            int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets, int64_t P, Plan plan, int do_plan) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int cnt[kMaxE], off[kMaxE], ta[kMaxE], tb[kMaxE];
    __shared__ int ws[33];
    const int e = threadIdx.x;
    if (e < E) {
        int run = 0;
        int c = 0;
        // Loads are independent of the running sum; unrolling keeps several
        // in flight.
        for (; c + 8 <= nchunks; c += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = chunk_hist[(int64_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                chunk_base[(int64_t)(c + u) * E + e] = run;
                run += v[u];
            }
        }
        for (; c < nchunks; ++c) {
            const int v = chunk_hist[(int64_t)c * E + e];
            chunk_base[(int64_t)c * E + e] = run;
            run += v;
        }
        cnt[e] = run;
        off[e] = run;
    }
    __syncthreads();
    block_exclusive_scan<1024>(off, E, ws);
    if (e < E) {
        counts[e] = cnt[e];
        offsets[e] = off[e];
    }
    if (e == 0) offsets[E] = (int32_t)P;
    if (do_plan) block_plan<1024>(cnt, off, E, plan, ta, tb, ws);
}

__global__ void __launch_bounds__(32 * kScatterWarps)
scatter_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
               const int32_t* __restrict__ chunk_base,
               const int32_t* __restrict__ offsets,
               int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int wc[kScatterWarps][kMaxE];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x)
        wc[i / E][i % E] = 0;
    __syncthreads();
    const int64_t beg = (int64_t)blockIdx.x * kPermChunk + (int64_t)w * kSlotsPerWarp;
    // pass 1: per-warp counts
    for (int it = 0; it < kSlotsPerWarp / 32; ++it) {
        const int64_t s = beg + it * 32 + lane;
        int e = (s < P) ? idx[s] : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wc[w][e] += __popc(peers);
    }
    __syncthreads();
    // per-warp starting positions
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = offsets[e] + chunk_base[(int64_t)blockIdx.x * E + e];
#pragma unroll
        for (int ww = 0; ww < kScatterWarps; ++ww) {
            const int v = wc[ww][e];
            wc[ww][e] = run;
            run += v;
        }
    }
    __syncthreads();
    // pass 2: scatter in slot order
    const unsigned lt = lanemask_lt();
    for (int it = 0; it < kSlotsPerWarp / 32; ++it) {
        const int64_t s = beg + it * 32 + lane;
        int e = (s < P) ? idx[s] : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = wc[w][e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = (int32_t)s;
            inv_perm[s] = pos;
            if (lane == __ffs(peers) - 1) wc[w][e] += __popc(peers);
        }
        __syncwarp();
    }
}

// ---- small path: everything in one block -------------------------------

__global__ void __launch_bounds__(32 * kScatterWarps)
permute_small_kernel(const int32_t* __restrict__ idx, int P, int E,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
                     WsHeader* hdr, Plan plan, int do_plan) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int wc[kScatterWarps][kMaxE];   // reused as planner scratch
    __shared__ int cnt[kMaxE], off[kMaxE];
    __shared__ int ws[33];
    constexpr int NT = 32 * kScatterWarps;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kScatterWarps * E; i += NT) wc[i / E][i % E] = 0;
    __syncthreads();
    const int beg = w * kSlotsPerWarp;
    for (int it = 0; it < kSlotsPerWarp / 32; ++it) {
        const int s = beg + it * 32 + lane;
        int e = (s < P) ? idx[s] : -1;
        if (s < P && (unsigned)e >= (unsigned)E) set_status(hdr, MOE_ERR_BAD_INDEX);
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) wc[w][e] += __popc(peers);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) {
        int c = 0;
#pragma unroll
        for (int ww = 0; ww < kScatterWarps; ++ww) c += wc[ww][e];
        cnt[e] = c;
        off[e] = c;
    }
    __syncthreads();
    block_exclusive_scan<NT>(off, E, ws);
    for (int e = threadIdx.x; e < E; e += NT) {
        int run = off[e];
#pragma unroll
        for (int ww = 0; ww < kScatterWarps; ++ww) {
            const int v = wc[ww][e];
            wc[ww][e] = run;
            run += v;
        }
        counts[e] = cnt[e];
        offsets[e] = off[e];
    }
    if (threadIdx.x == 0) offsets[E] = P;
    __syncthreads();
    const unsigned lt = lanemask_lt();
    for (int it = 0; it < kSlotsPerWarp / 32; ++it) {
        const int s = beg + it * 32 + lane;
        int e = (s < P) ? idx[s] : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = wc[w][e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = s;
            inv_perm[s] = pos;
            if (lane == __ffs(peers) - 1) wc[w][e] += __popc(peers);
        }
        __syncwarp();
    }
    __syncthreads();
    if (do_plan) block_plan<NT>(cnt, off, E, plan, &wc[0][0], &wc[4][0], ws);
}

__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
            int E, Plan plan) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int cnt[kMaxE], off[kMaxE], ta[kMaxE], tb[kMaxE];
    __shared__ int ws[33];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        cnt[e] = counts[e];
        off[e] = offsets[e];
    }
    __syncthreads();
    block_plan<1024>(cnt, off, E, plan, ta, tb, ws);
}

// x_sorted[p] = x[perm[p] / k] for the rows of the fat tiles (paired and
// solo) and of the tensor-core streaming tiles (all of them, or one of the
// two gather parts); one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256)
gather_kernel(GatherRows g, const WsHeader* __restrict__ hdr, int part) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t r_beg, r_end;
    gather_part_rows(hdr, part, &r_beg, &r_end);
    gather_rows(g, hdr, r_beg, r_end, warp, nwarps);
}

}  // namespace

size_t permute_scratch_ints(int64_t P, int E) {
    const int64_t nchunks = (P + kPermChunk - 1) / kPermChunk;
    return (size_t)(2 * nchunks * E);
}

cudaError_t launch_permute(const int32_t* idx, int T, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, int32_t* chunk_hist,
                           int32_t* chunk_base, WsHeader* hdr,
                           const Plan* plan, cudaStream_t s) {
    const int64_t P = (int64_t)T * k;
    Plan pl{};
    if (plan) pl = *plan;
    if (P <= kPermChunk) {
        return launch_pdl(permute_small_kernel, dim3(1), dim3(32 * kScatterWarps), 0, s, idx,
                          (int)P, E, counts, offsets, perm, inv_perm, hdr, pl,
                          (int)(plan != nullptr));
    }
    const int nchunks = (int)((P + kPermChunk - 1) / kPermChunk);
    cudaError_t e = launch_pdl(hist_kernel, dim3(nchunks), dim3(256), 0, s, idx, P, E,
                               chunk_hist, hdr);
    if (e == cudaSuccess)
        e = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, s, chunk_hist, nchunks, E,
                       chunk_base, counts, offsets, P, pl, (int)(plan != nullptr));
    if (e == cudaSuccess)
        e = launch_pdl(scatter_kernel, dim3(nchunks), dim3(32 * kScatterWarps), 0, s, idx, P,
                       E, chunk_base, offsets, perm, inv_perm);
    return e;
}

cudaError_t launch_plan(const int32_t* counts, const int32_t* offsets, int E,
                        const Plan& plan, cudaStream_t s) {
    return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s, counts, offsets, E, plan);
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* perm, int k,
                          int H, const Plan& plan, __nv_bfloat16* x_sorted,
                          int num_sms, cudaStream_t s, int part) {
    GatherRows g;
    g.x = reinterpret_cast<const uint4*>(x);
    g.perm = perm;
    g.k = k;
    g.vec = H / 8;
    g.tiles = plan.tiles;
    g.solo_tiles = plan.solo_tiles;
    g.mma_tiles = plan.mma_tiles;
    g.x_sorted = reinterpret_cast<uint4*>(x_sorted);
    return launch_pdl(gather_kernel, dim3(num_sms * 8), dim3(256), 0, s, g,
                      (const WsHeader*)plan.hdr, part);
}

}  // namespace moe
