// thin.cu -- the gate/up kernel of the CUDA-core weight-streaming path and
// its launcher (the path and its ring: thin_dev.cuh; the down kernel:
// thin_down.cu).
#include "thin_dev.cuh"

namespace moe {
namespace {

// ---- kernels -------------------------------------------------------------------

// VPL = H / 256 when a 16 KB slot holds 16 / VPL whole rows each of gate and
// up (H = 256 ... 4096): register-cached path for units of <= 4 slots; 0: any
// H, rows read from shared memory.
template <int VPL>
__global__ void __launch_bounds__(kThreads, 1)
thin_gate_up_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm,
                    int k, int H, int I, int R, const __nv_bfloat16* __restrict__ Wg,
                    const __nv_bfloat16* __restrict__ Wu, const ThinUnit* __restrict__ units,
                    const int32_t* __restrict__ wslot,
                    WsHeader* hdr, __nv_bfloat16* __restrict__ h, int stage_bytes, int slots,
                    int act_bytes, SelfRoute sr, long long wait_cycles) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SmallPlan sp;
    constexpr int kProducers = 2;   // warp 0 issues the gate rows, warp 1 the up rows
    const int nc = (blockDim.x >> 5) - kProducers;
    const Smem m = smem_setup(smem, stage_bytes, slots, act_bytes, kProducers, nc);
    grid_dep_wait();      // the plan (or the logits) may come from the previous kernel
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int vec = H / 8;
    const int ipe = I / R;
    // The units and the slot order: the plan's, or the batch's own routing.
    const ThinUnit* U = units;
    const int32_t* order = perm;
    int n_units, weight;
    if (sr.logits) {
        build_small_plan(sr, sp);
        if (blockIdx.x == 0) write_small_plan(sr, sp, hdr);
        U = sp.units;
        order = sp.perm;
        n_units = sp.n_units;
        weight = sp.weight;
    } else {
        n_units = hdr->n_thin;
        weight = hdr->thin_weight;
    }
    const Range rg = cta_range(U, n_units, weight, ipe);
    const uint32_t half = (uint32_t)R * H * 2;
    const uint32_t xrow = (uint32_t)H * 2;

    if (warp < kProducers) {
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            const __nv_bfloat16* W = warp == 0 ? Wg : Wu;
            const uint32_t part = warp == 0 ? 0u : half;
            const bool ok = produce(
                m, warp, rg, warp == 0,
                [&](int it, uint32_t dst, uint32_t bar) {
                    const ThinUnit un = U[it / ipe];
                    const size_t off =
                        ((size_t)weight_block(wslot, un.expert) * I + (size_t)(it % ipe) * R) * H;
                    mbar_expect_tx(bar, half);
                    bulk_g2s_evict_first(dst + part, W + off, half, bar, policy);
                },
                [&](int u, uint32_t dst, uint32_t bar) {
                    const ThinUnit un = U[u];
                    mbar_expect_tx(bar, (uint32_t)un.n * xrow);
                    for (int t = 0; t < un.n; ++t)
                        bulk_g2s(dst + t * xrow, x + (size_t)(order[un.row0 + t] / k) * H, xrow, bar);
                },
                wait_cycles);
            if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
        }
        return;
    }

    const bool ok = consume<16>(m, rg, ipe, U, warp - kProducers, nc, wait_cycles,
                                [&]<int N>(int it, int slot, const Smem& mu) {
        const ThinUnit un = U[it / ipe];
        __nv_bfloat16* hcol = h + (int64_t)un.row0 * I + (it % ipe) * R;
        gate_up_slot<N, VPL>(mu, slot, R, vec, un.n, hcol, I);
    });
    if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
}

template <int V>
cudaError_t launch_gu(const __nv_bfloat16* x, const int32_t* perm, int k, int H, int I,
                      const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, const Plan& plan,
                      const Geometry& g, __nv_bfloat16* h, int num_sms, cudaStream_t s,
                      const SelfRoute& sr) {
    static std::atomic<int> done[kMaxDevices];
    cudaError_t e = smem_limit_once(thin_gate_up_kernel<V>, kSmemBudget + 1024, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(thin_gate_up_kernel<V>, dim3(num_sms), dim3(threads_for(g, 2)), g.smem, s,
                      x, perm, k, H, I, g.R, Wg, Wu, plan.units, plan.wslot, plan.hdr, h, g.stage,
                      g.slots, g.act, sr, main_wait_cycles());
}

}  // namespace

int thin_unit_tokens(int H, int I) {
    const int row = 2 * (H > I ? H : I);
    int nu = kActBudget / row;
    if (nu > kMaxUnitTokens) nu = kMaxUnitTokens;
    return nu < 1 ? 1 : nu;
}

cudaError_t launch_thin_gate_up(const __nv_bfloat16* x, const int32_t* perm, int k, int H,
                                int I, const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                                const Plan& plan, int64_t max_slots, __nv_bfloat16* h,
                                int num_sms, cudaStream_t s, const SelfRoute* sr) {
    const SelfRoute self = sr ? *sr : SelfRoute{};
    const int act_tokens =
        (int)std::min<int64_t>(plan.unit_tokens, std::max<int64_t>(max_slots, 1));
    const Geometry g = geometry(2 * H * 2, H * 2, act_tokens, false);
    if (g.smem > kSmemBudget + 1024) {
        set_last_error("thin gate/up: H = %d needs %d bytes of shared memory", H, g.smem);
        return cudaErrorInvalidConfiguration;
    }
    switch (g.stage == kStageTarget ? H : 0) {
        case 256: return launch_gu<1>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
        case 512: return launch_gu<2>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
        case 1024: return launch_gu<4>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
        case 2048: return launch_gu<8>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
        case 4096: return launch_gu<16>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
        default: return launch_gu<0>(x, perm, k, H, I, Wg, Wu, plan, g, h, num_sms, s, self);
    }
}

}  // namespace moe
