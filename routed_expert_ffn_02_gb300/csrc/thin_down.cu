// thin_down.cu -- the down kernel of the CUDA-core weight-streaming path and
// its launcher (the path and its ring: thin_dev.cuh).
#include "thin_dev.cuh"

namespace moe {
namespace {

// ---- kernels -------------------------------------------------------------------

// VPL = I / 256 when a 16 KB slot holds 32 / VPL whole rows of W_down
// (I = 256 ... 8192): register-cached path; 0: any I.
template <int VPL>
__global__ void __launch_bounds__(kThreads, 1)
thin_down_kernel(const __nv_bfloat16* __restrict__ h, int H, int I, int R,
                 const __nv_bfloat16* __restrict__ Wd, const ThinUnit* __restrict__ units,
                 const int32_t* __restrict__ wslot, WsHeader* hdr,
                 __nv_bfloat16* __restrict__ y, int stage_bytes, int slots, int act_bytes,
                 SelfRoute sr, long long wait_cycles) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SmallPlan sp;
    constexpr int kProducers = 1;
    const int nc = (blockDim.x >> 5) - kProducers;
    const Smem m = smem_setup(smem, stage_bytes, slots, act_bytes, kProducers, nc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int vec = I / 8;
    const int ipe = H / R;
    // The plan was written by the route-list kernels, which precede the
    // previous kernel on the stream (at least the gate/up kernel runs in
    // between) and so have completed when this kernel starts; W_down is read
    // only.  So the CTA's range and its first round of weight rows are
    // fetched before waiting for the previous kernel; h and y after.  A batch
    // that routes itself has its plan written by the gate/up kernel, the
    // previous launch: it is read after the wait.
    const ThinUnit* U = units;
    int n_units, weight;
    if (sr.logits) {
        grid_dep_wait();
        load_small_plan(sr, hdr, sp);
        U = sp.units;
        n_units = sp.n_units;
        weight = sp.weight;
    } else {
        n_units = hdr->n_thin;
        weight = hdr->thin_weight;
    }
    const Range rg = cta_range(U, n_units, weight, ipe);
    const uint32_t bytes = (uint32_t)R * I * 2;
    const uint32_t hrow = (uint32_t)I * 2;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            auto copy_item = [&](int it, uint32_t dst, uint32_t bar) {
                const ThinUnit un = U[it / ipe];
                mbar_expect_tx(bar, bytes);
                bulk_g2s_evict_first(
                    dst, Wd + ((size_t)weight_block(wslot, un.expert) * H + (size_t)(it % ipe) * R) * I,
                    bytes, bar, policy);
            };
            const int pre = rg.cnt < m.slots ? (rg.cnt > 0 ? rg.cnt : 0) : m.slots;
            for (int i = 0; i < pre; ++i) copy_item(rg.beg + i, m.buf(i), m.full(i));
            grid_dep_wait();
            grid_dep_launch();
            const bool ok = produce(
                m, 0, rg, true, copy_item,
                [&](int u, uint32_t dst, uint32_t bar) {
                    const ThinUnit un = U[u];
                    // the unit's h rows are consecutive sorted positions
                    mbar_expect_tx(bar, (uint32_t)un.n * hrow);
                    bulk_g2s(dst, h + (size_t)un.row0 * I, (uint32_t)un.n * hrow, bar);
                },
                wait_cycles, pre);
            if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
        }
    } else {
        grid_dep_wait();      // consumers write y
        grid_dep_launch();
        constexpr int kExact =
            (VPL > 0 && DownRegSlots<VPL>::value > 0) ? DownRegSlots<VPL>::value : 16;
        const bool ok = consume<kExact>(m, rg, ipe, U, warp - kProducers, nc, wait_cycles,
                                        [&]<int N>(int it, int slot, const Smem& mu) {
            const ThinUnit un = U[it / ipe];
            __nv_bfloat16* ycol = y + (int64_t)un.row0 * H + (it % ipe) * R;
            down_slot<N, VPL>(mu, slot, R, vec, un.n, ycol, H);
        });
        if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
    }
    if (sr.out) {   // fused combine; every thread has waited for the gate/up kernel
        grid_dep_wait();
        combine_if_last(sr, sp, hdr, y, H);
    }
}

template <int V>
cudaError_t launch_d(const __nv_bfloat16* h, int H, int I, const __nv_bfloat16* Wd,
                     const Plan& plan, const Geometry& g, __nv_bfloat16* y, int num_sms,
                     cudaStream_t s, const SelfRoute& sr) {
    static std::atomic<int> done[kMaxDevices];
    cudaError_t e = smem_limit_once(thin_down_kernel<V>, kSmemBudget + 1024, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(thin_down_kernel<V>, dim3(num_sms), dim3(threads_for(g, 1)), g.smem, s, h,
                      H, I, g.R, Wd, plan.units, plan.wslot, plan.hdr, y, g.stage, g.slots, g.act,
                      sr, main_wait_cycles());
}

}  // namespace

cudaError_t launch_thin_down(const __nv_bfloat16* h, int H, int I, const __nv_bfloat16* Wd,
                             const Plan& plan, int64_t max_slots, __nv_bfloat16* y_sorted,
                             int num_sms, cudaStream_t s, const SelfRoute* sr) {
    const SelfRoute self = sr ? *sr : SelfRoute{};
    const int act_tokens =
        (int)std::min<int64_t>(plan.unit_tokens, std::max<int64_t>(max_slots, 1));
    const Geometry g = geometry(I * 2, I * 2, act_tokens, true);
    if (g.smem > kSmemBudget + 1024) {
        set_last_error("thin down: I = %d needs %d bytes of shared memory", I, g.smem);
        return cudaErrorInvalidConfiguration;
    }
    switch (g.stage == kStageTarget ? I : 0) {
        case 256: return launch_d<1>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        case 512: return launch_d<2>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        case 1024: return launch_d<4>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        case 2048: return launch_d<8>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        case 4096: return launch_d<16>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        case 8192: return launch_d<32>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
        default: return launch_d<0>(h, H, I, Wd, plan, g, y_sorted, num_sms, s, self);
    }
}

}  // namespace moe
