// gemm_tc.cu -- grouped expert GEMMs for "busy" experts on the 5th-generation
// tensor cores (tcgen05 + TMEM), fed by TMA, on CTA pairs.
//
// Experts holding at least the fat threshold of slots run as dense GEMMs
// (dsv41-flash-offload wiki, overview: busy experts run as FP16 GEMMs; model
// page launch flags: fat threshold 32).  Here the GEMMs are bf16 with fp32
// accumulation, over variable-size groups, scheduled entirely on the device:
//
//   gate/up:  h[rows, n0:n0+128] = silu(A Wg_e[n0:n0+128]^T) * (A Wu_e[n0:n0+128]^T)
//             A = x_sorted[rows, :H]; one MMA of N = 256 covers the gate and
//             up halves, so SiLU*up is fused into the epilogue.
//   down:     y[rows, n0:n0+256] = h[rows, :I] Wd_e[n0:n0+256]^T
//
// Each work item is a 256 x 256 output tile computed by a cluster of two
// CTAs (tcgen05 cta_group::2, M = 256): CTA r of the pair loads its own
// 128 rows of A (planner tile 2q + r of the expert) and half of the B tile
// (gate rows / up rows for gate/up, the first / second 128 weight rows for
// down), so each SM reads 32 KB from L2 per 64 K instead of the 48 KB a
// one-CTA 128 x 256 tile needs.  A stage holds a 128-wide K block (two
// swizzle atoms per operand, 64 KB per CTA, 3 stages): per-stage handoffs
// (barrier wait, commit) cost the tensor pipe ~100 cycles each, so 128-wide
// stages ran 8% faster than 64-wide ones with the same bytes in flight.
// Both CTAs' copies complete on the even CTA's "full" barrier; the even CTA
// issues the MMAs, whose commits arrive on the "empty" and "accumulator
// full" barriers of both CTAs; each CTA's epilogue reads its own 128 TMEM
// lanes and releases the accumulator on the even CTA's barrier.
//
// Roles per CTA (persistent, one cluster per SM pair):
//   warp 0      TMA producer (one lane);
//   warp 1      MMA issuer (one lane, even CTA only): M=256, N=256, K=16,
//               fp32 accumulators in TMEM, two 256-column buffers so the
//               epilogue of one tile overlaps the main loop of the next;
//   warp 2      TMEM allocator (both CTAs, collectively);
//   warps 2-3   gate/up, first launch of a batch only: the row gather for
//               the second launch (see below);
//   warps 4-7   epilogue: tcgen05.ld -> activation -> bf16 -> a 128-byte-
//               swizzled 32 x 64 shared tile per warp -> one TMA tensor store
//               (coalesced 128-byte rows; per-lane stores of 16 bytes to 32
//               different rows cost the down GEMM 20% of its time, measured
//               by compiling them out); a warp whose rows cross the expert's
//               end stores its valid rows itself.
// Rows of a tile past the expert's end belong to other experts (or are past
// the tensor and zero-filled by TMA); they are computed and discarded.
//
// The gate/up GEMM of a batch runs as two launches (GemmArgs::part): the
// first over the first third of the pair tiles, whose x_sorted rows the
// gather kernel copied, while its otherwise idle warps 2-3 copy the rows of
// the other tiles (gather_dev.cuh); the second over the rest.  So two thirds
// of the gather's HBM traffic run under tensor-bound work (prefill chunk:
// 5.37-5.52 -> 5.28-5.42 ms per step, measured; a first part of a quarter or
// a fifth left the idle warps too little time and stretched the first
// launch).
//
// Every mbarrier wait is bounded (main-loop waits by GemmArgs::wait_cycles).
// On expiry the role records MOE_ERR_TIMEOUT in the workspace status and
// raises the abort flag of both CTAs; every role then stops issuing work, the
// MMA issuer waits for its issued MMAs, and before TMEM is freed the even CTA
// waits for every stage round either CTA filled (see drain_pair): no copy or
// MMA is in flight when the pair exits.
#include <cuda.h>
#include <algorithm>
#include <mutex>

#include "gather_dev.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = kTileM;          // A rows per CTA (M = 2 * BM per pair)
constexpr int KSUB = 2;             // 128-byte swizzle atoms (64 bf16) per K block
constexpr int BK = 64 * KSUB;       // K per stage: fewer, larger stages (see below)
constexpr int BN_MMA = 256;         // MMA N (each CTA holds BN_MMA / 2 rows of B)
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;                // 32 KB
constexpr int B_BYTES = (BN_MMA / 2) * BK * 2;      // 32 KB (this CTA's half)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;      // 64 KB
constexpr int TMEM_COLS = 512;                      // two 256-column accumulators
// Epilogue staging: each epilogue warp writes its 32 rows x 64 columns of
// the output into a 128-byte-swizzled shared tile (two per warp, alternating)
// that one tensor store copies out.
constexpr int OUT_COLS = 64;
constexpr int OUT_BUF_BYTES = 32 * OUT_COLS * 2;            // 4 KB
constexpr int STAGING_BYTES = 4 * 2 * OUT_BUF_BYTES;        // 32 KB
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 256 /*barriers*/;

constexpr uint32_t kIdesc = tc::make_idesc(2 * BM, BN_MMA);
constexpr uint16_t kPairMask = 0x3;

struct GemmArgs {
    const FatTile* tiles;  // pairs: tiles 2q, 2q+1 belong to one expert
    const int32_t* wslot;  // expert -> weight block (nullptr: identity)
    const WsHeader* hdr_ro;
    WsHeader* hdr;
    int n_blocks_n;        // N tiles per expert
    int k_blocks;          // K / BK
    int b_rows_per_expert; // rows of the B tensor(s) per expert (I or H)
    int b_half_rows;       // B row offset of the odd CTA's half (0 gated: own tensor)
    int bn_out;            // output columns per tile (128 gated, 256 down)
    __nv_bfloat16* out;    // [rows, ld_out]
    int64_t ld_out;
    long long wait_cycles; // limit of each main-loop wait (SM cycles)
    int part;              // pair tiles: 0 all, 1 the first gather part (its idle
                           // warps then gather the other rows), 2 the rest
    GatherRows gather;     // part 1 of gate/up: the rows of part 2
};

// Stage rounds filled into stage s by a producer that filled `fills` stages
// in ring order.
__device__ __forceinline__ int rounds_filled(int fills, int s) {
    return fills > s ? (fills - s + STAGES - 1) / STAGES : 0;
}

// After an abort, run by one thread of the even CTA once both CTAs' roles
// have stopped (fills_even / fills_odd: the stages each CTA's producer
// filled).  Every round of a stage that either CTA filled completes on the
// even CTA's full barrier; the two producers differ by at most one round per
// stage (a round needs the previous one consumed, which needs both CTAs'
// bytes).  A round only the odd CTA filled is armed here for its bytes; a
// round only the even CTA filled is credited the odd CTA's missing bytes.
// Then each last round is waited for with the full bound, so every copy of
// both CTAs has landed.
__device__ __forceinline__ void drain_pair(uint32_t full0, int fills_even, int fills_odd,
                                           uint32_t stage_bytes) {
    for (int s = 0; s < STAGES; ++s) {
        const uint32_t bar = full0 + 8u * s;
        const int re = rounds_filled(fills_even, s) - 1, ro = rounds_filled(fills_odd, s) - 1;
        if (re < 0 && ro < 0) continue;
        if (ro == re + 1) {
            if (re >= 0) (void)ptx::mbar_wait(bar, (uint32_t)(re & 1));
            ptx::mbar_expect_tx(bar, stage_bytes);
            (void)ptx::mbar_wait(bar, (uint32_t)(ro & 1));
        } else if (re == ro + 1) {
            ptx::mbar_complete_tx(bar, stage_bytes);
            (void)ptx::mbar_wait(bar, (uint32_t)(re & 1));
        } else {
            (void)ptx::mbar_wait(bar, (uint32_t)(re & 1));
        }
    }
}

// B rows of N tile nt: gated: 128 rows of Wg (even CTA) or Wu (odd CTA);
// down: rows [256 nt, 256 nt + 256) of Wd, the odd CTA taking the upper 128.
template <bool kGated>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmOut, GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t staging = base + STAGES * STAGE_BYTES;
    const uint32_t bars = staging + STAGING_BYTES;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + STAGES * STAGE_BYTES + STAGING_BYTES + 8 * (2 * STAGES + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* fills_out = reinterpret_cast<int*>(tmem_holder + 2);   // stages this CTA filled

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();     // 0: issues the MMAs
    const uint32_t peer_abort = mapa_shared(smem_u32(tmem_holder + 1), rank ^ 1u);
    // A role that gives up stops both CTAs of the pair.
    auto give_up = [&]() {
        *abort_flag = 1;
        st_shared_cluster(peer_abort, 1u);
        set_status(args.hdr, MOE_ERR_TIMEOUT);
    };
    const int cluster = (int)blockIdx.x >> 1;
    const int n_clusters = (int)gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);     // even CTA's producer + both CTAs' bytes
            mbar_init(empty_bar(s), 1);    // the pair's MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 8);   // one lane of 4 epilogue warps x 2 CTAs
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        *fills_out = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmA);
        prefetch_map(&tmB0);
        if (kGated) prefetch_map(&tmB1);
        prefetch_map(&tmOut);
    }
    if (warp == 2) tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
    fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    grid_dep_wait();      // everything above overlaps the previous kernel
    grid_dep_launch();

    const int n_pairs = args.hdr_ro->n_fat_tiles >> 1;
    const int q_split = gather_first_pairs(n_pairs);
    const int w0 = (args.part == 2 ? q_split : 0) * args.n_blocks_n;
    const int total = (args.part == 1 ? q_split : n_pairs) * args.n_blocks_n;
    const int w_first = w0 + cluster;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        const CUtensorMap* tmB = (kGated && rank == 1) ? &tmB1 : &tmB0;
        const uint32_t full0 = mapa_shared(full_bar(0), 0);   // even CTA's barriers
        int stage = 0;
        uint32_t phase = 0;
        int fills = 0;
        bool ok = true;
        // Each item's tile is loaded one item ahead (its latency is hidden).
        FatTile ft_next = {};
        if (w_first < total) ft_next = args.tiles[2 * (w_first / args.n_blocks_n) + (int)rank];
        for (int w = w_first; ok && w < total; w += n_clusters) {
            const int nt = w % args.n_blocks_n;
            const FatTile ft = ft_next;
            if (w + n_clusters < total)
                ft_next = args.tiles[2 * ((w + n_clusters) / args.n_blocks_n) + (int)rank];
            const int brow = weight_block(args.wslot, ft.expert) * args.b_rows_per_expert +
                             nt * (kGated ? BM : BN_MMA) +
                             (int)rank * args.b_half_rows;
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(empty_bar(stage), phase ^ 1u, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = base + stage * STAGE_BYTES;
                const uint32_t fb = full0 + 8u * stage;
                if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * STAGE_BYTES);
#pragma unroll
                for (int a = 0; a < KSUB; ++a) {
                    tma_load_2d_pair(sa + a * (A_BYTES / KSUB), &tmA, fb, kb * BK + 64 * a, ft.row0);
                    tma_load_2d_pair(sa + A_BYTES + a * (B_BYTES / KSUB), tmB, fb, kb * BK + 64 * a, brow);
                }
                ++fills;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && !*abort_flag) give_up();
        // Without an abort every filled stage is read by the pair's MMAs,
        // which complete before the epilogues finish; after one, drain_pair
        // waits for the copies.
        *fills_out = fills;
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------- MMA issuer (even CTA) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        bool issued = false;
        for (int w = w_first; ok && w < total; w += n_clusters, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait_for(tempty_bar(acc), acc_phase ^ 1u, args.wait_cycles, abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN_MMA);
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(full_bar(stage), phase, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t sa = base + stage * STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // +32 bytes per 16-element K step inside a swizzle row
                    const int a = kk / 4;
                    const uint64_t ad = sw128_desc(sa + a * (A_BYTES / KSUB));
                    const uint64_t bd = sw128_desc(sa + A_BYTES + a * (B_BYTES / KSUB));
                    mma_bf16_pair(d_tmem, ad + (uint64_t)((kk % 4) * 2), bd + (uint64_t)((kk % 4) * 2),
                                  kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                issued = true;
                commit_pair_multicast(empty_bar(stage), kPairMask);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            commit_pair_multicast(tfull_bar(acc), kPairMask);
        }
        if (!ok) {
            if (!*abort_flag) give_up();
            if (issued) {
                // Wait for every MMA issued so far before TMEM is freed.
                commit_pair_multicast(done_bar, 0x1);
                (void)mbar_wait(done_bar, 0);
            }
        }
    } else if (kGated && args.part == 1 && (warp == 2 || warp == 3)) {
        // ---------------- gather of the later pair tiles' rows ----------------
        // (the next launch's A rows; this launch's tiles were gathered before)
        int64_t r_beg, r_end;
        gather_part_rows(args.hdr_ro, 2, &r_beg, &r_end);
        gather_rows(args.gather, args.hdr_ro, r_beg, r_end,
                    (int64_t)blockIdx.x * 2 + (warp - 2), (int64_t)gridDim.x * 2);
    } else if (warp >= 4) {
        // ---------------- epilogue (both CTAs) ----------------
        const int ew = warp - 4;              // TMEM lanes 32*ew .. 32*ew+31
        const int row = ew * 32 + lane;
        const uint32_t out_buf = staging + (uint32_t)ew * 2u * OUT_BUF_BYTES;
        int n_out = 0;                        // tensor stores this warp issued
        const uint32_t tempty0 = mapa_shared(tempty_bar(0), 0);
        int it = 0;
        FatTile ft_next = {};
        if (w_first < total) ft_next = args.tiles[2 * (w_first / args.n_blocks_n) + (int)rank];
        for (int w = w_first; w < total; w += n_clusters, ++it) {
            const FatTile ft = ft_next;
            if (w + n_clusters < total)
                ft_next = args.tiles[2 * ((w + n_clusters) / args.n_blocks_n) + (int)rank];
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)((it >> 1) & 1);
            // the whole warp decides together (tcgen05.ld below is warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait_for(tfull_bar(acc), acc_phase, args.wait_cycles, abort_flag))) {
                if (!*abort_flag) give_up();
                break;
            }
            fence_after();
            const int nt = w % args.n_blocks_n;
            const bool valid = row < ft.rows;
            // all 32 rows of this warp belong to the tile's expert: tensor
            // stores of whole 32 x 64 boxes; else each valid lane stores its row
            const bool whole = ew * 32 + 32 <= ft.rows;
            __nv_bfloat16* dst = args.out + (int64_t)(ft.row0 + row) * args.ld_out +
                                 (int64_t)nt * args.bn_out;
            const uint32_t taddr = tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * BN_MMA);
#pragma unroll 1
            for (int c = 0; c < args.bn_out; c += OUT_COLS) {
                uint32_t packed[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int cc = c + 32 * half;
                    if (kGated) {
                        uint32_t g[32], u[32];
                        tmem_ld32(taddr + cc, g);
                        tmem_ld32(taddr + 128 + cc, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            packed[16 * half + q] = pack_bf16(
                                swiglu(__uint_as_float(g[2 * q]), __uint_as_float(u[2 * q])),
                                swiglu(__uint_as_float(g[2 * q + 1]), __uint_as_float(u[2 * q + 1])));
                    } else {
                        uint32_t v[32];
                        tmem_ld32(taddr + cc, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            packed[16 * half + q] =
                                pack_bf16(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                    }
                }
                if (whole) {
                    const uint32_t buf = out_buf + (uint32_t)(n_out & 1) * OUT_BUF_BYTES;
                    // the store that used this buffer two boxes ago has read it
                    if (lane == 0 && n_out >= 2) bulk_wait_read<1>();
                    __syncwarp();
                    // row `lane`, 16-byte chunk j at chunk j ^ (row mod 8) (128-byte swizzle)
                    const uint32_t rb = buf + (uint32_t)lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(rb + ((uint32_t)(j ^ (lane & 7)) << 4), packed[4 * j],
                                     packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOut, buf, nt * args.bn_out + c, ft.row0 + ew * 32);
                        bulk_commit();
                    }
                    ++n_out;
                } else if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                           packed[4 * q + 3]);
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * acc);
        }
        // every tensor store of this warp has completed before the CTA leaves
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' roles have stopped
    // Both CTAs read the same two flags here, so they agree on the drain.
    if (*abort_flag || ld_shared_cluster(peer_abort) != 0) {
        if (rank == 0 && threadIdx.x == 0)
            drain_pair(full_bar(0), *fills_out,
                       (int)ld_shared_cluster(mapa_shared(smem_u32(fills_out), 1)),
                       (uint32_t)STAGE_BYTES);
        cluster_sync();
    }
    // the pair is done with each other's barriers, shared memory and TMEM
    if (warp == 2) {
        fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---- host side -----------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

template <bool kGated>
cudaError_t set_smem_attr() {
    static std::atomic<int> done[kMaxDevices];
    return smem_limit_once(grouped_gemm_kernel<kGated>, SMEM_BYTES, done);
}

// CTAs to launch: two per co-resident cluster (an SM pair whose partner is
// busy or absent cannot host a cluster, so this can be below the SM count).
template <bool kGated>
cudaError_t pair_grid(int num_sms, int* grid) {
    constexpr int kMaxDev = kMaxDevices;
    static int cached[kMaxDev] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (!cached[dev]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<kGated>, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        cached[dev] = 2 * std::min(clusters, num_sms / 2);
    }
    *grid = cached[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t make_tma_map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                              uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H, int I,
                                const Plan& plan, __nv_bfloat16* h, int num_sms,
                                cudaStream_t s, int part, const __nv_bfloat16* x,
                                const int32_t* perm, int k) {
    CUtensorMap mA, mG, mU;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mA, x_sorted, (uint64_t)rows_alloc, (uint64_t)H, BM)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mG, Wg, (uint64_t)plan.n_wblocks * I, (uint64_t)H, 128)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mU, Wu, (uint64_t)plan.n_wblocks * I, (uint64_t)H, 128)) != cudaSuccess) return e;
    CUtensorMap mO;
    if ((e = make_tma_map_bf16(&mO, h, (uint64_t)rows_alloc, (uint64_t)I, 32)) != cudaSuccess) return e;
    if ((e = set_smem_attr<true>()) != cudaSuccess) return e;
    int grid = 0;
    if ((e = pair_grid<true>(num_sms, &grid)) != cudaSuccess) return e;
    GemmArgs a;
    a.tiles = plan.tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks_n = I / 128;
    a.k_blocks = H / BK;
    a.b_rows_per_expert = I;
    a.b_half_rows = 0;        // the odd CTA reads the same rows of Wu
    a.bn_out = 128;
    a.out = h;
    a.ld_out = I;
    a.wait_cycles = main_wait_cycles();
    a.part = part;
    a.gather.x = reinterpret_cast<const uint4*>(x);
    a.gather.perm = perm;
    a.gather.k = k;
    a.gather.vec = H / 8;
    a.gather.tiles = plan.tiles;
    a.gather.solo_tiles = plan.solo_tiles;
    a.gather.mma_tiles = plan.mma_tiles;
    a.gather.x_sorted = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(x_sorted));
    return launch_pdl(grouped_gemm_kernel<true>, dim3(grid), dim3(256), SMEM_BYTES, s, mA, mG, mU,
                      mO, a);
}

cudaError_t launch_gemm_down(const __nv_bfloat16* h, int64_t rows_alloc,
                             const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                             __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s) {
    CUtensorMap mA, mD;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mA, h, (uint64_t)rows_alloc, (uint64_t)I, BM)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mD, Wd, (uint64_t)plan.n_wblocks * H, (uint64_t)I, 128)) != cudaSuccess) return e;
    CUtensorMap mO;
    if ((e = make_tma_map_bf16(&mO, y_sorted, (uint64_t)rows_alloc, (uint64_t)H, 32)) != cudaSuccess) return e;
    if ((e = set_smem_attr<false>()) != cudaSuccess) return e;
    int grid = 0;
    if ((e = pair_grid<false>(num_sms, &grid)) != cudaSuccess) return e;
    GemmArgs a;
    a.tiles = plan.tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks_n = H / 256;
    a.k_blocks = I / BK;
    a.b_rows_per_expert = H;
    a.b_half_rows = 128;      // the odd CTA reads the upper half of the 256 rows
    a.bn_out = 256;
    a.out = y_sorted;
    a.ld_out = H;
    a.wait_cycles = main_wait_cycles();
    a.part = 0;
    a.gather = GatherRows{};
    return launch_pdl(grouped_gemm_kernel<false>, dim3(grid), dim3(256), SMEM_BYTES, s, mA, mD,
                      mD, mO, a);
}

}  // namespace moe
