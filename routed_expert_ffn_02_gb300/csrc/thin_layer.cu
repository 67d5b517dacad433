// thin_layer.cu -- the one-launch decode layer on the CUDA-core weight-
// streaming path (the path and its ring: thin_dev.cuh).
#include "thin_dev.cuh"

namespace moe {
namespace {

// One decode layer of a self-routed batch in one cooperative launch (every
// CTA resident at once, one per SM):
//   1. gate/up: routing, route lists and units in every CTA (CTA 0 stores
//      them), then the gate/up stream of thin_gate_up_kernel;
//   2. each CTA fences its h rows and arrives on the workspace's layer_sync
//      counter (monotonic: this launch waits for the next multiple of the
//      grid size after the count it found);
//   3. down: the ring is set up again for W_down; the producer copies its
//      first ring of weight rows, waits (bounded) until every CTA has
//      arrived, and then stages h rows and streams the rest, as
//      thin_down_kernel;
//   4. after a second grid-wide wait, every CTA combines its share of the
//      batch (combine_spread).
// Compared with the two launches it saves the second kernel's start, and a
// CTA that finishes its gate/up share early streams W_down while the others
// finish theirs.  VG / VD: the register-cached row paths of the two kernels.
constexpr int kPreIssueOneToken = 4;

// kBufs: activation buffers of the two rings (2 from two tokens on: a CTA
// whose range reaches into the next unit has that unit's rows staged while
// it finishes the current one; a single token keeps one buffer).
template <int VG, int VD, int kBufs>
__global__ void __launch_bounds__(kThreads, 1)
thin_layer_kernel(const __nv_bfloat16* __restrict__ x, int k, int H, int I, int Rg, int Rd,
                  const __nv_bfloat16* __restrict__ Wg, const __nv_bfloat16* __restrict__ Wu,
                  const __nv_bfloat16* __restrict__ Wd, const int32_t* __restrict__ wslot,
                  WsHeader* hdr, __nv_bfloat16* __restrict__ h, __nv_bfloat16* __restrict__ y,
                  int stage_g, int slots_g, int act_g, int stage_d, int slots_d, int act_d,
                  SelfRoute sr, long long wait_cycles) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SmallPlan sp;
    __shared__ uint32_t s_target;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_warps = blockDim.x >> 5;

    int failed;
    {   // ---------------- gate/up ----------------
        constexpr int kProducers = 2;   // warp 0 issues the gate rows, warp 1 the up rows
        const int nc = min(n_warps - kProducers, slots_g - 1);
        const Smem m = smem_setup(smem, stage_g, slots_g, act_g, kProducers, nc, kBufs);
        grid_dep_wait();      // the logits may come from the previous kernel
        grid_dep_launch();
        build_small_plan(sr, sp);
        if (blockIdx.x == 0) write_small_plan(sr, sp, hdr);
        const int vec = H / 8, ipe = I / Rg;
        const Range rg = cta_range(sp.units, sp.n_units, sp.weight, ipe);
        const uint32_t half = (uint32_t)Rg * H * 2, xrow = (uint32_t)H * 2;
        bool ok = true;
        if (warp < kProducers) {
            if (lane == 0) {
                const uint64_t policy = policy_evict_first();
                const __nv_bfloat16* W = warp == 0 ? Wg : Wu;
                const uint32_t part = warp == 0 ? 0u : half;
                ok = produce<kBufs>(
                    m, warp, rg, warp == 0,
                    [&](int it, uint32_t dst, uint32_t bar) {
                        const ThinUnit un = sp.units[it / ipe];
                        const size_t off = ((size_t)weight_block(wslot, un.expert) * I +
                                            (size_t)(it % ipe) * Rg) * H;
                        mbar_expect_tx(bar, half);
                        bulk_g2s_evict_first(dst + part, W + off, half, bar, policy);
                    },
                    [&](int u, uint32_t dst, uint32_t bar) {
                        const ThinUnit un = sp.units[u];
                        mbar_expect_tx(bar, (uint32_t)un.n * xrow);
                        for (int t = 0; t < un.n; ++t)
                            bulk_g2s(dst + t * xrow, x + (size_t)(sp.perm[un.row0 + t] / k) * H,
                                     xrow, bar);
                    },
                    wait_cycles);
            }
        } else if (warp - kProducers < nc) {
            ok = consume<16, kBufs>(m, rg, ipe, sp.units, warp - kProducers, nc, wait_cycles,
                                    [&]<int N>(int it, int slot, const Smem& mu) {
                const ThinUnit un = sp.units[it / ipe];
                __nv_bfloat16* hcol = h + (int64_t)un.row0 * I + (it % ipe) * Rg;
                gate_up_slot<N, VG>(mu, slot, Rg, vec, un.n, hcol, I);
            });
        }
        if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
        // this CTA's h rows, for other CTAs' bulk copies
        fence_proxy_async_global();
        __threadfence();
        failed = __syncthreads_or(!ok);
        // after a timeout the ring may still have copies in flight: the CTA
        // then skips the down phase (the status already records the error)
        if (!failed) smem_teardown(m);
    }
    if (threadIdx.x == 0) {   // arrive; the down producer waits for the whole grid
        const uint32_t seen = atomicAdd(&hdr->layer_sync, 1u);
        s_target = (seen / gridDim.x + 1) * gridDim.x;
    }
    if (!failed) {   // ---------------- down ----------------
        constexpr int kProducers = 1;
        const int nc = min(n_warps - kProducers, slots_d - 1);
        const Smem m = smem_setup(smem, stage_d, slots_d, act_d, kProducers, nc, kBufs);
        const int vec = I / 8, ipe = H / Rd;
        const Range rg = cta_range(sp.units, sp.n_units, sp.weight, ipe);
        const uint32_t bytes = (uint32_t)Rd * I * 2, hrow = (uint32_t)I * 2;
        bool ok = true;
        if (warp == 0) {
            if (lane == 0) {
                const uint64_t policy = policy_evict_first();
                auto copy_item = [&](int it, uint32_t dst, uint32_t bar) {
                    const ThinUnit un = sp.units[it / ipe];
                    mbar_expect_tx(bar, bytes);
                    bulk_g2s_evict_first(dst, Wd + ((size_t)weight_block(wslot, un.expert) * H +
                                                    (size_t)(it % ipe) * Rd) * I,
                                         bytes, bar, policy);
                };
                // W_down copies issued before the grid-wide wait: a full ring,
                // except for a single token, whose gate/up shares end close
                // together and whose wait returns sooner with fewer copies
                // queued (measured: batch 1 gains with 4, batch 2 loses).
                const int cap = sr.T == 1 ? min(kPreIssueOneToken, m.slots) : m.slots;
                const int pre = rg.cnt < cap ? (rg.cnt > 0 ? rg.cnt : 0) : cap;
                for (int i = 0; i < pre; ++i) copy_item(rg.beg + i, m.buf(i), m.full(i));
                // every CTA's h rows are stored (bounded wait)
                const uint32_t target = s_target;
                const long long t0 = clock64();
                while ((int32_t)(ld_acquire_gpu(&hdr->layer_sync) - target) < 0) {
                    if (clock64() - t0 > wait_cycles) {
                        set_status(hdr, MOE_ERR_TIMEOUT);
                        break;
                    }
                    __nanosleep(32);
                }
                fence_proxy_async_global();
                ok = produce<kBufs>(
                    m, 0, rg, true, copy_item,
                    [&](int u, uint32_t dst, uint32_t bar) {
                        const ThinUnit un = sp.units[u];
                        // the unit's h rows are consecutive sorted positions
                        mbar_expect_tx(bar, (uint32_t)un.n * hrow);
                        bulk_g2s(dst, h + (size_t)un.row0 * I, (uint32_t)un.n * hrow, bar);
                    },
                    wait_cycles, pre);
            }
        } else if (warp - kProducers < nc) {
            constexpr int kExact =
                (VD > 0 && DownRegSlots<VD>::value > 0) ? DownRegSlots<VD>::value : 16;
            ok = consume<kExact, kBufs>(m, rg, ipe, sp.units, warp - kProducers, nc,
                                        wait_cycles, [&]<int N>(int it, int slot, const Smem& mu) {
                const ThinUnit un = sp.units[it / ipe];
                __nv_bfloat16* ycol = y + (int64_t)un.row0 * H + (it % ipe) * Rd;
                down_slot<N, VD>(mu, slot, Rd, vec, un.n, ycol, H);
            });
        }
        if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
    }
    combine_spread(sr, sp.inv_perm, sp.gates, hdr, y, H, wait_cycles);
}

template <int VG, int VD, int kBufs>
cudaError_t launch_layer(const __nv_bfloat16* x, int k, int H, int I, const __nv_bfloat16* Wg,
                         const __nv_bfloat16* Wu, const __nv_bfloat16* Wd, const Plan& plan,
                         const Geometry& g1, const Geometry& g2, __nv_bfloat16* h,
                         __nv_bfloat16* y, int num_sms, cudaStream_t s, const SelfRoute& sr) {
    static std::atomic<int> done[kMaxDevices];
    cudaError_t e = smem_limit_once(thin_layer_kernel<VG, VD, kBufs>, kSmemBudget + 1024, done);
    if (e != cudaSuccess) return e;
    // every CTA resident at once (the down phase waits for all of them), and
    // allowed to start while the previous kernel on s finishes
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = std::max(g1.smem, g2.smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = t_pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, thin_layer_kernel<VG, VD, kBufs>, x, k, H, I, g1.R, g2.R, Wg, Wu,
                              Wd, plan.wslot, plan.hdr, h, y, g1.stage, g1.slots, g1.act,
                              g2.stage, g2.slots, g2.act, sr, main_wait_cycles());
}

}  // namespace

bool thin_layer_fused(int H, int I) {
    return (H == 4096 && I == 2048) || (H == 2048 && I == 1024) || (H == 512 && I == 256);
}

cudaError_t launch_thin_layer(const __nv_bfloat16* x, int k, int H, int I,
                              const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                              const __nv_bfloat16* Wd, const Plan& plan, int64_t max_slots,
                              __nv_bfloat16* h, __nv_bfloat16* y_sorted, int num_sms,
                              cudaStream_t s, const SelfRoute& sr) {
    const int act_tokens =
        (int)std::min<int64_t>(plan.unit_tokens, std::max<int64_t>(max_slots, 1));
    const int bufs = sr.T >= 2 ? 2 : 1;
    const Geometry g1 = geometry(2 * H * 2, H * 2, act_tokens, false, bufs);
    const Geometry g2 = geometry(I * 2, I * 2, act_tokens, true, bufs);
    if (g1.stage != kStageTarget || g2.stage != kStageTarget)
        return cudaErrorInvalidConfiguration;
#define MOE_LAYER(VG, VD)                                                                     \
    return bufs == 2 ? launch_layer<VG, VD, 2>(x, k, H, I, Wg, Wu, Wd, plan, g1, g2, h, y_sorted, \
                                               num_sms, s, sr)                                \
                     : launch_layer<VG, VD, 1>(x, k, H, I, Wg, Wu, Wd, plan, g1, g2, h, y_sorted, \
                                               num_sms, s, sr)
    if (H == 4096 && I == 2048) MOE_LAYER(16, 8);
    if (H == 2048 && I == 1024) MOE_LAYER(8, 4);
    if (H == 512 && I == 256) MOE_LAYER(2, 1);
#undef MOE_LAYER
    return cudaErrorInvalidConfiguration;
}

}  // namespace moe
