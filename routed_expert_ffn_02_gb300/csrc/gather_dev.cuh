// gather_dev.cuh -- the row gather x_sorted[p] = x[perm[p] / k] over the rows
// of the fat tiles (paired and solo) and of the tensor-core streaming tiles,
// shared by the gather kernel and the gate/up grouped GEMM (whose idle warps
// gather the rows of the later pair tiles while it computes the first ones).
#pragma once

#include "moe_internal.cuh"

namespace moe {

struct GatherRows {
    const uint4* x;            // [T, H] as 16-byte vectors
    const int32_t* perm;
    int k;
    int vec;                   // H / 8
    const FatTile* tiles;      // plan.tiles, plan.solo_tiles, plan.mma_tiles
    const FatTile* solo_tiles;
    const FatTile* mma_tiles;
    uint4* x_sorted;
};

// Gathered rows r (over all tiles, in list order) of part 0 (all), 1 (the
// first gather_first_pairs() pair tiles) or 2 (the others).
__device__ __forceinline__ void gather_part_rows(const WsHeader* hdr, int part, int64_t* r_beg,
                                                 int64_t* r_end) {
    const int64_t fat_rows = (int64_t)hdr->n_fat_tiles * kTileM;
    const int64_t rows = fat_rows + (int64_t)hdr->n_solo * kTileM +
                         (int64_t)hdr->n_thin_mma * kThinMaxTokens;
    const int64_t split =
        min(fat_rows, (int64_t)2 * gather_first_pairs(hdr->n_fat_tiles >> 1) * kTileM);
    *r_beg = part == 2 ? split : 0;
    *r_end = part == 1 ? split : rows;
}

// Called by whole warps: warp `worker` of `n_workers` copies rows r_beg +
// worker, r_beg + worker + n_workers, ... below r_end; sixteen 16-byte loads
// per lane (a whole row at H = 4096) are in flight before their stores.
__device__ __forceinline__ void gather_rows(const GatherRows& g, const WsHeader* hdr,
                                            int64_t r_beg, int64_t r_end, int64_t worker,
                                            int64_t n_workers) {
    const int lane = threadIdx.x & 31;
    const int64_t fat_rows = (int64_t)hdr->n_fat_tiles * kTileM;
    const int64_t solo_rows = fat_rows + (int64_t)hdr->n_solo * kTileM;
    for (int64_t r = r_beg + worker; r < r_end; r += n_workers) {
        FatTile ft;
        int i;
        if (r < fat_rows) {
            ft = g.tiles[r / kTileM];
            i = (int)(r % kTileM);
        } else if (r < solo_rows) {
            ft = g.solo_tiles[(r - fat_rows) / kTileM];
            i = (int)((r - fat_rows) % kTileM);
        } else {
            ft = g.mma_tiles[(r - solo_rows) / kThinMaxTokens];
            i = (int)((r - solo_rows) % kThinMaxTokens);
        }
        if (i >= ft.rows) continue;
        const int64_t p = ft.row0 + i;
        const uint4* src = g.x + (int64_t)(g.perm[p] / g.k) * g.vec;
        uint4* dst = g.x_sorted + p * g.vec;
        for (int v0 = lane; v0 < g.vec; v0 += 32 * 16) {
            uint4 buf[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (v0 + 32 * u < g.vec) buf[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (v0 + 32 * u < g.vec) dst[v0 + 32 * u] = buf[u];
        }
    }
}

}  // namespace moe
