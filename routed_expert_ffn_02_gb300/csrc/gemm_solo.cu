// gemm_solo.cu -- one-CTA grouped GEMMs for the fat experts' solo tiles.
//
// The grouped GEMM runs a fat expert's 128-row tiles in pairs on CTA pairs
// (gemm_tc.cu).  When an expert has an odd number of tiles its last tile
// would pair with an empty one and waste the partner CTA's MMA work; the
// planner lists it as a solo tile instead, and this kernel runs the solo
// tiles with tcgen05 cta_group::1 (tcgen05 instructions of both group sizes
// cannot share a kernel).  Same products as the pair GEMMs:
//
//   gate/up:  h[rows, n0:n0+128] = silu(A Wg_e[n0:n0+128]^T) * (A Wu_e[n0:n0+128]^T),
//             A = x_sorted[rows, :H]; the gate and up rows of the same 128
//             intermediate columns land back to back, one N = 256 MMA.
//   down:     y[rows, n0:n0+256] = h[rows, :I] Wd_e[n0:n0+256]^T
//
// Persistent CTAs (one per SM), warp-specialised: warp 0 TMA producer (one
// lane), warp 1 MMA issuer (M = 128, N = 256, K = 16), warp 2 TMEM
// allocator, warps 4-7 epilogue; 4-stage ring of 64-wide K blocks (48 KB),
// two 256-column TMEM accumulators.  Every wait is bounded; on expiry the
// kernel records MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM
// and returns.
#include <cuda.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = kTileM;                      // 128 rows per tile
constexpr int BK = 64;                          // one 128-byte swizzle row
constexpr int BN = 256;                         // MMA N
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int TMEM_COLS = 512;                  // two 256-column accumulators
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kIdesc = make_idesc(BM, BN);

struct SoloArgs {
    const FatTile* tiles;  // plan.solo_tiles
    const int32_t* wslot;  // expert -> weight block (nullptr: identity)
    const WsHeader* hdr_ro;
    WsHeader* hdr;
    int n_blocks_n;        // N tiles per expert
    int k_blocks;          // K / 64
    int b_rows_per_expert; // rows of the B tensor(s) per expert (I or H)
    int bn_out;            // output columns per tile (128 gated, 256 down)
    __nv_bfloat16* out;    // [rows, ld_out]
    int64_t ld_out;
    long long wait_cycles;     // limit of each main-loop wait (SM cycles)
};

template <bool kGated>
__global__ void __launch_bounds__(256, 1)
grouped_gemm_solo_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmB1, SoloArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + STAGES * STAGE_BYTES;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Nothing to do for most launches (solo tiles are few): leave before
    // allocating anything.  Uniform per CTA.
    grid_dep_wait();
    grid_dep_launch();
    const int total = args.hdr_ro->n_solo * args.n_blocks_n;
    // Items go round-robin to the first `active` CTAs, as many as keep every
    // wave full: a last wave of a few items (8 of 464 at the prefill chunk)
    // would stream alone at one SM's copy rate, well below its share of HBM.
    const int waves = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int active = waves > 0 ? (total + waves - 1) / waves : 0;
    if ((int)blockIdx.x >= active) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 128);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmA);
        prefetch_map(&tmB0);
        if (kGated) prefetch_map(&tmB1);
    }
    if (warp == 2) tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int b_tile_rows = kGated ? 128 : 256;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int pending[STAGES];
        for (int s = 0; s < STAGES; ++s) pending[s] = -1;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total; t += active) {
            const FatTile ft = args.tiles[t / args.n_blocks_n];
            const int brow = weight_block(args.wslot, ft.expert) * args.b_rows_per_expert +
                             (t % args.n_blocks_n) * b_tile_rows;
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(empty_bar(stage), phase ^ 1u, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = base + stage * STAGE_BYTES;
                const uint32_t sb = sa + A_BYTES;
                mbar_expect_tx(full_bar(stage), STAGE_BYTES);
                tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, ft.row0);
                if (kGated) {
                    tma_load_2d(sb, &tmB0, full_bar(stage), kb * BK, brow);
                    tma_load_2d(sb + B_BYTES / 2, &tmB1, full_bar(stage), kb * BK, brow);
                } else {
                    tma_load_2d(sb, &tmB0, full_bar(stage), kb * BK, brow);
                }
                pending[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            set_status(args.hdr, MOE_ERR_TIMEOUT);
            for (int s = 0; s < STAGES; ++s)
                if (pending[s] >= 0) (void)mbar_wait(full_bar(s), (uint32_t)pending[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        bool issued = false;
        for (int t = blockIdx.x; ok && t < total; t += active, ++it) {
            const int acc = it & 1;
            if (!mbar_wait_for(tempty_bar(acc), (uint32_t)((it >> 1) & 1) ^ 1u, args.wait_cycles, abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(full_bar(stage), phase, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t sa = base + stage * STAGE_BYTES;
                const uint64_t ad = sw128_desc(sa);
                const uint64_t bd = sw128_desc(sa + A_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)   // +32 bytes per 16-element K step
                    mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), kIdesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
                issued = true;
                commit(empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            commit(tfull_bar(acc));
        }
        if (!ok) {
            *abort_flag = 1;
            set_status(args.hdr, MOE_ERR_TIMEOUT);
            if (issued) {
                commit(done_bar);
                (void)mbar_wait(done_bar, 0);
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue ----------------
        const int ew = warp - 4;   // TMEM lanes 32*ew .. 32*ew+31
        const int row = ew * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += active, ++it) {
            const int acc = it & 1;
            // the whole warp decides together (tcgen05.ld below is warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait_for(tfull_bar(acc), (uint32_t)((it >> 1) & 1), args.wait_cycles, abort_flag))) {
                *abort_flag = 1;
                set_status(args.hdr, MOE_ERR_TIMEOUT);
                break;
            }
            fence_after();
            const FatTile ft = args.tiles[t / args.n_blocks_n];
            const int nt = t % args.n_blocks_n;
            const bool valid = row < ft.rows;
            __nv_bfloat16* dst =
                args.out + (int64_t)(ft.row0 + row) * args.ld_out + (int64_t)nt * args.bn_out;
            const uint32_t taddr = tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * BN);
            if (kGated) {
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(taddr + c, g);
                    tmem_ld32(taddr + 128 + c, u);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        packed[q] = pack_bf16(
                            swiglu(__uint_as_float(g[2 * q]), __uint_as_float(u[2 * q])),
                            swiglu(__uint_as_float(g[2 * q + 1]), __uint_as_float(u[2 * q + 1])));
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                               packed[4 * q + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(taddr + c, v);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        packed[q] = pack_bf16(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                               packed[4 * q + 3]);
                    }
                }
            }
            fence_before();
            mbar_arrive(tempty_bar(acc));
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 2) {
        fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool kGated>
cudaError_t set_smem_attr() {
    static std::atomic<int> done[kMaxDevices];
    return smem_limit_once(grouped_gemm_solo_kernel<kGated>, SMEM_BYTES, done);
}

}  // namespace

cudaError_t launch_gemm_solo_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                     const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H,
                                     int I, const Plan& plan, __nv_bfloat16* h, int num_sms,
                                     cudaStream_t s) {
    CUtensorMap mA, mG, mU;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mA, x_sorted, (uint64_t)rows_alloc, (uint64_t)H, BM)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mG, Wg, (uint64_t)plan.n_wblocks * I, (uint64_t)H, 128)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mU, Wu, (uint64_t)plan.n_wblocks * I, (uint64_t)H, 128)) != cudaSuccess) return e;
    if ((e = set_smem_attr<true>()) != cudaSuccess) return e;
    SoloArgs a;
    a.tiles = plan.solo_tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks_n = I / 128;
    a.k_blocks = H / BK;
    a.b_rows_per_expert = I;
    a.bn_out = 128;
    a.out = h;
    a.ld_out = I;
    a.wait_cycles = main_wait_cycles();
    return launch_pdl(grouped_gemm_solo_kernel<true>, dim3(num_sms), dim3(256), SMEM_BYTES, s,
                      mA, mG, mU, a);
}

cudaError_t launch_gemm_solo_down(const __nv_bfloat16* h, int64_t rows_alloc,
                                  const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                                  __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s) {
    CUtensorMap mA, mD;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mA, h, (uint64_t)rows_alloc, (uint64_t)I, BM)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mD, Wd, (uint64_t)plan.n_wblocks * H, (uint64_t)I, 256)) != cudaSuccess) return e;
    if ((e = set_smem_attr<false>()) != cudaSuccess) return e;
    SoloArgs a;
    a.tiles = plan.solo_tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks_n = H / 256;
    a.k_blocks = I / BK;
    a.b_rows_per_expert = H;
    a.bn_out = 256;
    a.out = y_sorted;
    a.ld_out = H;
    a.wait_cycles = main_wait_cycles();
    return launch_pdl(grouped_gemm_solo_kernel<false>, dim3(num_sms), dim3(256), SMEM_BYTES, s,
                      mA, mD, mD, a);
}

}  // namespace moe
