// thin_mma.cu -- weight streaming on the tensor cores for thin experts.
//
// A thin expert (fewer slots than the fat threshold; dsv41-flash-offload
// wiki, overview: the group/thin kernel for experts that are not busy) must
// stream all of its weights from HBM once, reused over at most
// kThinMaxTokens slots.  On CUDA cores the bf16 FMAs of a weight element
// cost more than its HBM read beyond ~5 slots; here the product runs on
// tcgen05 instead so the kernel stays bound by the weight stream at any slot
// count.  The roles of the grouped GEMM are swapped ("swap AB"):
//
//   MMA A (M = 128)  a 128-row block of one weight matrix, K-major
//                    (Wg/Wu rows i of [I, H]; Wd rows of [H, I]);
//   MMA B (N = 32)   the expert's slots, K-major (x_sorted or h rows);
//   D (TMEM)         D[i][j] = weight row i . slot j, fp32.
//
// A work item is (thin expert, 128-row block); consecutive CTAs take
// consecutive blocks of one expert so its slot rows are shared in L2.
// gate/up: one item covers 128 rows of Wg and of Wu (two MMAs into two TMEM
// accumulators) and writes h[row0 + j][i] = bf16(silu(g) * u) for j < n.
// down: y[row0 + j][i] = bf16(D[i][j]).  Columns j >= n read other experts'
// rows (or TMA's zero fill past the tensor); each output column depends only
// on its own slot row, so they are computed and discarded.
//
// Small batches routed inside the kernels (SelfRoute, small_plan.cuh): every
// gate/up CTA builds the batch's plan in shared memory, one tile per touched
// expert, and loads each tile's activation rows straight from x with one-row
// TMA boxes (the 128-byte swizzle follows the shared-memory address, so a row
// lands where a 32-row box would put it), so no gather runs; the down kernel
// reads the plan back and, launched cooperatively, every CTA combines its
// share of the batch after a bounded grid-wide wait (combine_spread).
//
// Persistent, one CTA per SM, warp-specialised like the grouped GEMM:
// warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM allocator, warps 4-7
// epilogue; two TMEM accumulator buffers so an item's epilogue overlaps the
// next item's stream.  Every wait is bounded; on expiry the kernel records
// MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "small_plan.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int BM = 128;              // weight rows per item (MMA M)
constexpr int BN = kThinMaxTokens;   // slot columns (MMA N)
constexpr int BK = 64;               // 128-byte swizzle row
constexpr int W_BYTES = BM * BK * 2;   // 16 KB
constexpr int X_BYTES = BN * BK * 2;   // 4 KB
constexpr uint32_t kIdesc = make_idesc(BM, BN);

template <bool kGated>
struct Cfg {
    static constexpr int kMats = kGated ? 2 : 1;
    static constexpr int kStageBytes = kMats * W_BYTES + X_BYTES;   // 36 / 20 KB
    static constexpr int kStages = kGated ? 6 : 10;
    static constexpr int kAccCols = kMats * BN;                     // per buffer
    static constexpr int kTmemCols = kGated ? 128 : 64;             // two buffers
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
};

struct ThinMmaArgs {
    const FatTile* tiles;     // thin experts on this kernel: (expert, row0, n)
    const int32_t* wslot;     // expert -> weight block (nullptr: identity)
    const WsHeader* hdr_ro;
    WsHeader* hdr;
    int n_blocks;             // 128-row weight blocks per expert
    int k_blocks;             // reduction length / 64
    int w_rows_per_expert;    // rows of the weight tensor per expert
    __nv_bfloat16* out;       // [rows_alloc, ld_out]
    int64_t ld_out;
    SelfRoute sr;             // logits != nullptr: the batch routes itself
    long long wait_cycles;     // limit of each main-loop wait (SM cycles)
};

template <bool kGated>
__global__ void __launch_bounds__(256, 1)
thin_mma_kernel(const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmW0,
                const __grid_constant__ CUtensorMap tmW1,
                const __grid_constant__ CUtensorMap tmXrow, ThinMmaArgs args) {
    using C = Cfg<kGated>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ SmallPlan sp;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + C::kStages * C::kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * C::kStages + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * C::kStages + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * C::kStages + 4);
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(base_ptr + C::kStages * C::kStageBytes + 8 * (2 * C::kStages + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
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
        prefetch_map(&tmX);
        prefetch_map(&tmW0);
        if (kGated) prefetch_map(&tmW1);
    }
    if (warp == 2) tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    grid_dep_wait();      // everything above overlaps the previous kernel
    grid_dep_launch();
    const bool self = args.sr.logits != nullptr;
    if (self) {
        if (kGated) {
            build_small_plan(args.sr, sp);
            if (blockIdx.x == 0) write_small_plan(args.sr, sp, args.hdr, true);
        } else {
            load_small_plan(args.sr, args.hdr, sp);
        }
    }
    const int n_tiles = self ? sp.n_units : args.hdr_ro->n_thin_mma;
    const int total = n_tiles * args.n_blocks;
    // Items go round-robin to the first `active` CTAs, as many as keep every
    // wave full: one SM streams well below its share of HBM bandwidth when
    // few others run, so a last wave of a few items (8 of 616 at decode batch
    // 24) would run alone at that rate.  The other CTAs take no item.
    const int waves = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int active = waves > 0 ? (total + waves - 1) / waves : 1;
    const int first = (int)blockIdx.x < active ? (int)blockIdx.x : total;
    auto tile_at = [&](int i) {
        if (!self) return args.tiles[i];
        const ThinUnit u = sp.units[i];
        FatTile f;
        f.expert = u.expert;
        f.row0 = u.row0;
        f.rows = u.n;
        f.pad = 0;
        return f;
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int pending[C::kStages];
        for (int s = 0; s < C::kStages; ++s) pending[s] = -1;
        bool ok = true;
        // Each item's tile is loaded one item ahead (its latency is hidden).
        FatTile ft_next = {};
        if (first < total) ft_next = tile_at(first / args.n_blocks);
        for (int t = first; ok && t < total; t += active) {
            const FatTile ft = ft_next;
            if (t + active < total) ft_next = tile_at((t + active) / args.n_blocks);
            const int wrow = weight_block(args.wslot, ft.expert) * args.w_rows_per_expert +
                             (t % args.n_blocks) * BM;
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(empty_bar(stage), phase ^ 1u, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sw = base + stage * C::kStageBytes;
                const bool rows = kGated && self;   // x rows by token, one box each
                mbar_expect_tx(full_bar(stage), rows ? (uint32_t)(C::kMats * W_BYTES + ft.rows * BK * 2)
                                                     : (uint32_t)C::kStageBytes);
                tma_load_2d(sw, &tmW0, full_bar(stage), kb * BK, wrow);
                if (kGated) tma_load_2d(sw + W_BYTES, &tmW1, full_bar(stage), kb * BK, wrow);
                if (rows) {
                    for (int j = 0; j < ft.rows; ++j)
                        tma_load_2d(sw + C::kMats * W_BYTES + (uint32_t)(j * BK * 2), &tmXrow,
                                    full_bar(stage), kb * BK, sp.perm[ft.row0 + j] / args.sr.k);
                } else {
                    tma_load_2d(sw + C::kMats * W_BYTES, &tmX, full_bar(stage), kb * BK, ft.row0);
                }
                pending[stage] = (int)phase;
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            set_status(args.hdr, MOE_ERR_TIMEOUT);
            for (int s = 0; s < C::kStages; ++s)
                if (pending[s] >= 0) (void)mbar_wait(full_bar(s), (uint32_t)pending[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        bool issued = false;
        for (int t = first; ok && t < total; t += active, ++it) {
            const int acc = it & 1;
            if (!mbar_wait_for(tempty_bar(acc), (uint32_t)((it >> 1) & 1) ^ 1u, args.wait_cycles, abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t d0 = tmem_base + (uint32_t)(acc * C::kAccCols);
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_for(full_bar(stage), phase, args.wait_cycles, abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t sw = base + stage * C::kStageBytes;
                const uint64_t a0 = sw128_desc(sw);
                const uint64_t bx = sw128_desc(sw + C::kMats * W_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16(d0, a0 + (uint64_t)(kk * 2), bx + (uint64_t)(kk * 2), kIdesc, accum);
                    if (kGated)
                        mma_bf16(d0 + BN, sw128_desc(sw + W_BYTES) + (uint64_t)(kk * 2),
                                 bx + (uint64_t)(kk * 2), kIdesc, accum);
                }
                issued = true;
                commit(empty_bar(stage));
                if (++stage == C::kStages) {
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
        const int ew = warp - 4;   // TMEM lanes (weight rows) 32*ew .. 32*ew+31
        int it = 0;
        FatTile ft_next = {};
        if (first < total) ft_next = tile_at(first / args.n_blocks);
        for (int t = first; t < total; t += active, ++it) {
            const FatTile ft = ft_next;
            if (t + active < total) ft_next = tile_at((t + active) / args.n_blocks);
            const int acc = it & 1;
            // the whole warp decides together (tcgen05.ld below is warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait_for(tfull_bar(acc), (uint32_t)((it >> 1) & 1), args.wait_cycles, abort_flag))) {
                *abort_flag = 1;
                set_status(args.hdr, MOE_ERR_TIMEOUT);
                break;
            }
            fence_after();
            const int col = (t % args.n_blocks) * BM + ew * 32 + lane;
            __nv_bfloat16* dst = args.out + (int64_t)ft.row0 * args.ld_out + col;
            const uint32_t taddr =
                tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(acc * C::kAccCols);
            uint32_t v[32];
            tmem_ld32(taddr, v);
            if (kGated) {
                uint32_t u[32];
                tmem_ld32(taddr + BN, u);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < BN; ++j)
                    if (j < ft.rows)
                        dst[(int64_t)j * args.ld_out] = __float2bfloat16_rn(
                            swiglu(__uint_as_float(v[j]), __uint_as_float(u[j])));
            } else {
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < BN; ++j)
                    if (j < ft.rows)
                        dst[(int64_t)j * args.ld_out] = __float2bfloat16_rn(__uint_as_float(v[j]));
            }
            fence_before();
            mbar_arrive(tempty_bar(acc));
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 2) {
        fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    // a fused combine (a cooperative launch): every CTA combines its share,
    // by the batch's own plan or the planned route lists
    if (!kGated && args.sr.out)
        combine_spread(args.sr, self ? sp.inv_perm : args.sr.inv_perm,
                       self ? sp.gates : args.sr.gates, args.hdr, args.out, (int)args.ld_out,
                       args.wait_cycles);
}

template <bool kGated>
cudaError_t set_smem_attr() {
    static std::atomic<int> done[kMaxDevices];
    return smem_limit_once(thin_mma_kernel<kGated>, Cfg<kGated>::kSmemBytes, done);
}

}  // namespace

cudaError_t launch_thin_mma_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                    const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H,
                                    int I, const Plan& plan, __nv_bfloat16* h, int num_sms,
                                    cudaStream_t s, const SelfRoute* sr, const __nv_bfloat16* x) {
    CUtensorMap mX, mG, mU, mXr;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mX, x_sorted, (uint64_t)rows_alloc, (uint64_t)H, BN)) != cudaSuccess) return e;
    mXr = mX;
    if (sr && (e = make_tma_map_bf16(&mXr, x, (uint64_t)sr->T, (uint64_t)H, 1)) != cudaSuccess)
        return e;
    if ((e = make_tma_map_bf16(&mG, Wg, (uint64_t)plan.n_wblocks * I, (uint64_t)H, BM)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mU, Wu, (uint64_t)plan.n_wblocks * I, (uint64_t)H, BM)) != cudaSuccess) return e;
    if ((e = set_smem_attr<true>()) != cudaSuccess) return e;
    ThinMmaArgs a;
    a.tiles = plan.mma_tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks = I / BM;
    a.k_blocks = H / BK;
    a.w_rows_per_expert = I;
    a.out = h;
    a.ld_out = I;
    a.wait_cycles = main_wait_cycles();
    a.sr = sr ? *sr : SelfRoute{};
    return launch_pdl(thin_mma_kernel<true>, dim3(num_sms), dim3(256), Cfg<true>::kSmemBytes, s,
                      mX, mG, mU, mXr, a);
}

cudaError_t launch_thin_mma_down(const __nv_bfloat16* h, int64_t rows_alloc,
                                 const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                                 __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s,
                                 const SelfRoute* sr) {
    CUtensorMap mX, mD;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mX, h, (uint64_t)rows_alloc, (uint64_t)I, BN)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mD, Wd, (uint64_t)plan.n_wblocks * H, (uint64_t)I, BM)) != cudaSuccess) return e;
    if ((e = set_smem_attr<false>()) != cudaSuccess) return e;
    ThinMmaArgs a;
    a.tiles = plan.mma_tiles;
    a.wslot = plan.wslot;
    a.hdr_ro = plan.hdr;
    a.hdr = plan.hdr;
    a.n_blocks = H / BM;
    a.k_blocks = I / BK;
    a.w_rows_per_expert = H;
    a.out = y_sorted;
    a.ld_out = H;
    a.wait_cycles = main_wait_cycles();
    a.sr = sr ? *sr : SelfRoute{};
    // with the combine fused the CTAs wait for one another before it: every
    // CTA resident at once
    return launch_pdl_coop(sr != nullptr && sr->out != nullptr, thin_mma_kernel<false>, dim3(num_sms), dim3(256),
                           Cfg<false>::kSmemBytes, s, mX, mD, mD, mX, a);
}

}  // namespace moe
