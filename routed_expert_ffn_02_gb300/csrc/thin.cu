// thin.cu -- weight-streaming expert path for experts holding fewer slots
// than the fat threshold (all experts in decode).
//
// In decode only a handful of experts per layer are touched per token
// (dsv41-flash-offload wiki, PCIe paragraph); each touched expert's weights
// are read from HBM once and applied to all of its slots.  The work is
// memory-bound for few slots and CUDA-core-bound for many; the kernel keeps
// HBM busy and the FMA pipes fed:
//
//   * Work units (from the planner) hold up to `unit_tokens` consecutive
//     sorted slots of one expert; their activations (x rows for gate/up, h
//     rows for down) are staged together in shared memory.  A unit's weight
//     rows are split into items of R consecutive rows: one 16 KB slot, one
//     contiguous range in HBM.
//   * One CTA per SM owns a contiguous range of items whose total cost is an
//     equal share of the layer's (the planner prices a row by its unit's slot
//     count: flat while HBM-bound, growing with the FMAs).
//   * Warp-specialised: producer lanes stream the items' weight rows into a
//     ring of shared-memory slots with bulk copies on the TMA engine
//     (cp.async.bulk + mbarrier) -- two producers for gate/up (gate rows and up
//     rows), since one issuing thread sustains only so many copies per second
//     -- and the first producer also stages each unit's activations once the
//     consumers have released the previous unit's.  Producers sleep in
//     try_wait while the ring is full.  The other warps consume slots
//     round-robin.
//   * Slot protocol: a consumer waits until the slot's previous round has been
//     released, then for the current round to land; with more slots than
//     consumers this makes every parity wait unambiguous.
//   * A consumer lane covers the 16-byte vectors lane, lane+32, ... of a row.
//     It copies its share of the whole slot into registers and releases the
//     slot at once, so the ring refills while it computes (row lengths of
//     256 ... 4096 elements; other lengths compute from shared memory).  Products are mixed-precision FMAs (fma.rn.f32.bf16: bf16
//     operands straight from the staged data, fp32 accumulators, no
//     conversions) spread over enough independent accumulators to cover the
//     FMA latency; the warp finishes each row with shuffle reductions and
//     lane t writes slot t's result.
//
//   gate/up: h[p, i] = bf16( silu(Wg[e,i,:] . x_t) * (Wu[e,i,:] . x_t) )
//   down:    y[p, r] = bf16( Wd[e,r,:] . h[p, :] )
// for every sorted position p of expert e (token t = perm[p] / k).
//
// Small batches (at most 32 slots, one unit per expert) route themselves: the
// gate/up kernel builds the plan in every CTA and CTA 0 stores it, the down
// kernel reads it back after its wait and its last CTA combines the batch
// (small_plan.cuh).
//
// Waits are bounded; on expiry the kernel records MOE_ERR_TIMEOUT, the
// producer waits (bounded) for its outstanding copies, and the CTA returns.
#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "combine_dev.cuh"
#include "small_plan.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kWarps = 8;                      // producers + consumers
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxSlots = 16;
constexpr int kSmemBudget = 224 * 1024;
constexpr int kActBudget = 96 * 1024;          // activation buffer
constexpr int kStageTarget = 16384;            // bytes per weight slot
constexpr int kMaxUnitTokens = 16;
// Register-cached path: a lane holds 32 vectors of a slot (128 registers) and
// the row loop is unrolled over them, so it is taken for units of at most 4
// slots (more would not fit the instruction cache).
template <int VPL>
struct RegSlots {
    static constexpr int value = 4;
};
// Down slots hold 32 / VPL rows, computed together (accumulators per row and
// slot): while that is at most 4 rows, else the shared-memory path.
template <int VPL>
struct DownRegSlots {
    static constexpr int value = VPL >= 8 ? 4 : 0;
};

// ---- shared loads, mixed-precision FMA ---------------------------------------

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// The two bf16 halves of a 32-bit word as 16-bit registers.
__device__ __forceinline__ void split_bf16x2(uint32_t w, unsigned short& lo, unsigned short& hi) {
    asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
}
// acc += w * x with bf16 operands, exact products, fp32 accumulation.
__device__ __forceinline__ void fma_bf16(float& acc, unsigned short w, unsigned short x) {
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(w), "h"(x));
}

struct Bf16x8 {   // eight bf16 values as 16-bit registers
    unsigned short h[8];
    __device__ __forceinline__ explicit Bf16x8(const uint4& v) {
        split_bf16x2(v.x, h[0], h[1]);
        split_bf16x2(v.y, h[2], h[3]);
        split_bf16x2(v.z, h[4], h[5]);
        split_bf16x2(v.w, h[6], h[7]);
    }
};

// Independent accumulators per slot and matrix: at least eight chains per
// warp to cover the FMA latency.  Divides 8 (element q goes to chain q % P).
template <int N>
struct Chains {
    static constexpr int P = N >= 8 ? 1 : (N >= 4 ? 2 : (N >= 2 ? 4 : 8));
};

template <int P>
__device__ __forceinline__ float sum_chains(const float (&a)[P]) {
    float s = a[0];
#pragma unroll
    for (int i = 1; i < P; ++i) s += a[i];
    return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

// ---- shared-memory layout and pipeline ------------------------------------

// [slots x stage_bytes weight ring][activation buffer][barriers]
// Each producer's copies into a slot complete on its own full barrier
// (full(s) for producer 0, full2(s) for producer 1), so a producer that
// stops early can still wait for exactly the copies it issued.
constexpr int kBarriers = 3 * kMaxSlots + 2;
struct Smem {
    uint32_t base;       // shared addresses
    uint32_t act;
    uint32_t bars;
    int stage_bytes;
    int slots;
    int producers;
    __device__ uint32_t buf(int s) const { return base + (uint32_t)(s * stage_bytes); }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (kMaxSlots + s); }
    __device__ uint32_t act_full() const { return bars + 8u * (2 * kMaxSlots); }
    __device__ uint32_t act_free() const { return bars + 8u * (2 * kMaxSlots + 1); }
    __device__ uint32_t full2(int s) const { return bars + 8u * (2 * kMaxSlots + 2 + s); }
    // full barrier of producer p
    __device__ uint32_t full_of(int p, int s) const { return p == 0 ? full(s) : full2(s); }
};

__device__ __forceinline__ Smem smem_setup(uint8_t* smem, int stage_bytes, int slots,
                                           int act_bytes, int producers, int consumers) {
    Smem m;
    m.base = smem_u32(smem);
    m.stage_bytes = stage_bytes;
    m.slots = slots;
    m.producers = producers;
    m.act = m.base + (uint32_t)(slots * stage_bytes);
    m.bars = m.act + (uint32_t)act_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            for (int p = 0; p < producers; ++p) mbar_init(m.full_of(p, s), 1);
            mbar_init(m.empty(s), 1);
        }
        mbar_init(m.act_full(), 1);
        mbar_init(m.act_free(), consumers);
        fence_mbar_init();
    }
    __syncthreads();
    return m;
}

struct Range {
    int beg, cnt;          // items [beg, beg + cnt)
    int u_first, u_last;   // units they span (u_last < u_first when cnt == 0)
};

// First item whose cumulative cost reaches c: units have ipe items each, all
// of cost thin_unit_cost(n); units[u].cost_before is the per-item cost of the
// units before u.
__device__ __forceinline__ int item_at(const ThinUnit* units, int n_units, int ipe, int64_t c) {
    int lo = 0, hi = n_units - 1;   // largest u with ipe * cost_before <= c
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)units[mid].cost_before * ipe <= c) lo = mid;
        else hi = mid - 1;
    }
    const int w = thin_unit_cost(units[lo].n);
    const int64_t off = c - (int64_t)units[lo].cost_before * ipe;
    const int64_t k = (off + w - 1) / w;
    return lo * ipe + (int)(k < ipe ? k : ipe);
}

// This CTA's contiguous share of the items of n_units units of total cost
// `weight` (per item), of (about) equal total cost.
__device__ __forceinline__ Range cta_range(const ThinUnit* units, int n_units, int weight, int ipe) {
    Range r;
    if (n_units <= 0) {
        r.beg = r.cnt = 0;
        r.u_first = 0;
        r.u_last = -1;
        return r;
    }
    const int64_t total = (int64_t)weight * ipe;
    const int64_t c0 = total * blockIdx.x / gridDim.x;
    const int64_t c1 = total * (blockIdx.x + 1) / gridDim.x;
    r.beg = item_at(units, n_units, ipe, c0);
    const int end = blockIdx.x + 1 == gridDim.x ? n_units * ipe : item_at(units, n_units, ipe, c1);
    r.cnt = end - r.beg;
    r.u_first = r.beg / ipe;
    r.u_last = r.cnt > 0 ? (r.beg + r.cnt - 1) / ipe : r.u_first - 1;
    return r;
}

// All lanes of a warp wait (bounded by `limit` cycles, convergent) for the
// phase with the given parity.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, long long limit) {
    const bool ok = mbar_wait_for(bar, parity, limit, nullptr);
    return __all_sync(0xffffffffu, ok);
}

// Producer (one lane): streams the range's items through the weight ring
// (copy_item) and, if it is the `stager`, stages each unit's activations
// (copy_act) once the consumers have released the previous unit's.  Items
// [0, pre) (pre <= slots) were already issued into slots [0, pre).  While a
// slot is still in use the lane sleeps in try_wait.  Each wait gives up after
// `limit` cycles; then the copies already issued are waited for (full bound)
// and it returns false.
template <typename ItemFn, typename ActFn>
__device__ bool produce(const Smem& m, int producer, const Range& rg, bool stager,
                        ItemFn copy_item, ActFn copy_act, long long limit, int pre = 0) {
    if (rg.cnt <= 0) return true;
    int last_round[kMaxSlots];
    for (int s = 0; s < kMaxSlots; ++s) last_round[s] = s < pre ? 0 : -1;
    const int n_units = stager ? rg.u_last - rg.u_first + 1 : 0;
    int act_issued = 0;                       // units whose activations are staged
    if (stager) {
        copy_act(rg.u_first, m.act, m.act_full());
        act_issued = 1;
    }
    auto try_stage = [&]() {   // never blocks
        if (act_issued < n_units &&
            mbar_test_wait(m.act_free(), (uint32_t)((act_issued - 1) & 1))) {
            copy_act(rg.u_first + act_issued, m.act, m.act_full());
            ++act_issued;
        }
    };
    bool ok = true;
    int slot = pre % m.slots, round = pre / m.slots;
    for (int seq = pre; ok && seq < rg.cnt; ++seq) {
        if (round > 0) {
            const uint32_t par = (uint32_t)((round - 1) & 1);
            const long long start = clock64();
            while (!mbar_try_wait_sleep(m.empty(slot), par, 2000)) {
                try_stage();
                if (clock64() - start > limit) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
        }
        copy_item(rg.beg + seq, m.buf(slot), m.full_of(producer, slot));
        last_round[slot] = round;
        try_stage();
        if (++slot == m.slots) {
            slot = 0;
            ++round;
        }
    }
    while (ok && act_issued < n_units) {
        if (!mbar_wait_for(m.act_free(), (uint32_t)((act_issued - 1) & 1), limit, nullptr)) {
            ok = false;
            break;
        }
        copy_act(rg.u_first + act_issued, m.act, m.act_full());
        ++act_issued;
    }
    if (!ok) {
        // Let the copies already issued land before the CTA exits.
        for (int s = 0; s < m.slots; ++s)
            if (last_round[s] >= 0)
                (void)mbar_wait(m.full_of(producer, s), (uint32_t)(last_round[s] & 1));
        if (act_issued > 0) (void)mbar_wait(m.act_full(), (uint32_t)((act_issued - 1) & 1));
    }
    return ok;
}

// Called by all lanes of a consumer warp once they are done reading a slot.
__device__ __forceinline__ void release_slot(const Smem& m, int slot) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(m.empty(slot));
}

// Calls f.template operator()<N>() for the runtime slot count n in [1, 16];
// with kExact < 16, counts above kExact all go to N = kExact + 1.
template <int kExact = 16, typename F>
__device__ __forceinline__ void with_slots(int n, F&& f) {
    if constexpr (kExact < 16) {
        if (n > kExact) {
            f.template operator()<kExact + 1>();
            return;
        }
    }
    switch (n) {
        case 1: f.template operator()<1>(); break;
        case 2: f.template operator()<2>(); break;
        case 3: f.template operator()<3>(); break;
        case 4: f.template operator()<4>(); break;
        case 5: f.template operator()<5>(); break;
        case 6: f.template operator()<6>(); break;
        case 7: f.template operator()<7>(); break;
        case 8: f.template operator()<8>(); break;
        case 9: f.template operator()<9>(); break;
        case 10: f.template operator()<10>(); break;
        case 11: f.template operator()<11>(); break;
        case 12: f.template operator()<12>(); break;
        case 13: f.template operator()<13>(); break;
        case 14: f.template operator()<14>(); break;
        case 15: f.template operator()<15>(); break;
        default: f.template operator()<16>(); break;
    }
}

// Consumer warp c of nc.  For each unit of the range: wait for its
// activations, then for the warp's items of that unit (seq = c mod nc) wait
// for the slot and run item.template operator()<N>(item, slot) with N the
// unit's slot count (the item releases the slot), then release the
// activations.  Returns false when a wait ran past `limit` cycles.
template <int kExact, typename ItemFn>
__device__ bool consume(const Smem& m, const Range& rg, int ipe, const ThinUnit* units, int c,
                        int nc, long long limit, ItemFn item) {
    const int lane = threadIdx.x & 31;
    for (int u = rg.u_first; u <= rg.u_last; ++u) {
        if (!warp_wait(m.act_full(), (uint32_t)((u - rg.u_first) & 1), limit)) return false;
        const int s0 = max(u * ipe, rg.beg) - rg.beg;
        const int s1 = min((u + 1) * ipe, rg.beg + rg.cnt) - rg.beg;
        const int first = s0 + ((c - s0 % nc) + nc) % nc;
        bool ok = true;
        with_slots<kExact>(units[u].n, [&]<int N>() {
            int slot = first % m.slots, round = first / m.slots;
            for (int seq = first; seq < s1; seq += nc) {
                if (round > 0 && !warp_wait(m.empty(slot), (uint32_t)((round - 1) & 1), limit)) {
                    ok = false;
                    return;
                }
                if (!warp_wait(m.full(slot), (uint32_t)(round & 1), limit) ||
                    (m.producers > 1 && !warp_wait(m.full2(slot), (uint32_t)(round & 1), limit))) {
                    ok = false;
                    return;
                }
                item.template operator()<N>(rg.beg + seq, slot);
                slot += nc;            // nc < slots: at most one wrap
                if (slot >= m.slots) {
                    slot -= m.slots;
                    ++round;
                }
            }
        });
        if (!ok) return false;
        __syncwarp();
        if (lane == 0) mbar_arrive(m.act_free());
    }
    return true;
}

// ---- compute ------------------------------------------------------------------
//
// Rows are read lane-interleaved: vector v of a row = lane + 32 * j.  `vec`
// is the row length in 16-byte vectors (a multiple of 32); activation row t
// starts at act + t * vec * 16.

// Gate and up dot products; weight vectors come from wg_at(j) / wu_at(j)
// (registers or shared memory).
template <int N, int VPL, typename WG, typename WU>
__device__ __forceinline__ void gate_up_dots(WG wg_at, WU wu_at, uint32_t act, int vec, int iters,
                                             float (&g)[N], float (&u)[N]) {
    constexpr int P = Chains<N>::P;
    const int lane = threadIdx.x & 31;
    float ga[N][P], ua[N][P];
#pragma unroll
    for (int t = 0; t < N; ++t)
#pragma unroll
        for (int p = 0; p < P; ++p) ga[t][p] = ua[t][p] = 0.f;
#pragma unroll(VPL > 0 ? VPL : 2)
    for (int j = 0; j < (VPL > 0 ? VPL : iters); ++j) {
        const Bf16x8 wg(wg_at(j)), wu(wu_at(j));
#pragma unroll
        for (int t = 0; t < N; ++t) {
            const Bf16x8 xa(lds128(act + (uint32_t)((t * vec + lane + 32 * j) * 16)));
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                fma_bf16(ga[t][q % P], wg.h[q], xa.h[q]);
                fma_bf16(ua[t][q % P], wu.h[q], xa.h[q]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < N; ++t) {
        g[t] = warp_sum(sum_chains<P>(ga[t]));
        u[t] = warp_sum(sum_chains<P>(ua[t]));
    }
}

template <int N, int VPL, typename W>
__device__ __forceinline__ void down_dots(W w_at, uint32_t act, int vec, int iters,
                                          float (&a)[N]) {
    constexpr int P = Chains<N>::P;
    const int lane = threadIdx.x & 31;
    float acc[N][P];
#pragma unroll
    for (int t = 0; t < N; ++t)
#pragma unroll
        for (int p = 0; p < P; ++p) acc[t][p] = 0.f;
#pragma unroll(VPL > 0 ? VPL : 2)
    for (int j = 0; j < (VPL > 0 ? VPL : iters); ++j) {
        const Bf16x8 fw(w_at(j));
#pragma unroll
        for (int t = 0; t < N; ++t) {
            const Bf16x8 xa(lds128(act + (uint32_t)((t * vec + lane + 32 * j) * 16)));
#pragma unroll
            for (int q = 0; q < 8; ++q) fma_bf16(acc[t][q % P], fw.h[q], xa.h[q]);
        }
    }
#pragma unroll
    for (int t = 0; t < N; ++t) a[t] = warp_sum(sum_chains<P>(acc[t]));
}

template <int N>
__device__ __forceinline__ void store_h(const float (&g)[N], const float (&u)[N],
                                        __nv_bfloat16* hcol, int64_t ldh) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < N; ++t)
        if (lane == t) hcol[t * ldh] = __float2bfloat16_rn(silu_mul(g[t], u[t]));
}

template <int N>
__device__ __forceinline__ void store_y(const float (&a)[N], __nv_bfloat16* ycol, int64_t ldy) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < N; ++t)
        if (lane == t) ycol[t * ldy] = __float2bfloat16_rn(a[t]);
}

// Register-cached down slots of units with more than 4 slots: runtime loop
// over groups of 4 slots, so one compiled body (4 slots x RR rows x VPL
// vectors) serves every count and the weights stay in registers across groups
// (measured faster than computing from shared memory for down; for gate/up,
// whose slot is one long row pair, it was slower).  The last group may read
// activation rows past n (the buffer is padded to a multiple of 4 rows); their
// results are not stored.
template <int VPL, int RR>
__device__ __forceinline__ void down_groups_regs(const uint4 (&w)[RR * VPL], uint32_t act,
                                                 int vec, int n, __nv_bfloat16* ycol,
                                                 int64_t ldy) {
    constexpr int G = 4;
    constexpr int P = Chains<G * RR>::P;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int t0 = 0; t0 < n; t0 += G) {
        float acc[RR][G][P];
#pragma unroll
        for (int r = 0; r < RR; ++r)
#pragma unroll
            for (int t = 0; t < G; ++t)
#pragma unroll
                for (int p = 0; p < P; ++p) acc[r][t][p] = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
#pragma unroll
            for (int t = 0; t < G; ++t) {
                const Bf16x8 xa(lds128(act + (uint32_t)(((t0 + t) * vec + lane + 32 * j) * 16)));
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                    const Bf16x8 fw(w[r * VPL + j]);
#pragma unroll
                    for (int q = 0; q < 8; ++q) fma_bf16(acc[r][t][q % P], fw.h[q], xa.h[q]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RR; ++r)
#pragma unroll
            for (int t = 0; t < G; ++t) {
                const float a = warp_sum(sum_chains<P>(acc[r][t]));
                if (lane == t && t0 + t < n)
                    ycol[(int64_t)(t0 + t) * ldy + r] = __float2bfloat16_rn(a);
            }
    }
}

// One gate/up slot: R rows of gate then R rows of up, rows of vec vectors.
// VPL > 0 (= vec / 32, R = 16 / VPL): the lane's share is copied to
// registers and the slot released before computing (N <= RegSlots).
template <int N, int VPL>
__device__ __forceinline__ void gate_up_slot(const Smem& m, int slot, int R, int vec, int n_slots,
                                             __nv_bfloat16* hcol, int64_t ldh) {
    const int lane = threadIdx.x & 31;
    const uint32_t sg = m.buf(slot);
    const uint32_t su = sg + (uint32_t)(R * vec * 16);
    if constexpr (VPL > 0 && N <= RegSlots<VPL>::value) {
        constexpr int RR = 16 / VPL;
        uint4 wg[RR * VPL], wu[RR * VPL];
#pragma unroll
        for (int i = 0; i < RR * VPL; ++i) {
            wg[i] = lds128(sg + (uint32_t)((i * 32 + lane) * 16));
            wu[i] = lds128(su + (uint32_t)((i * 32 + lane) * 16));
        }
        release_slot(m, slot);
#pragma unroll
        for (int r = 0; r < RR; ++r) {
            float g[N], u[N];
            gate_up_dots<N, VPL>([&](int j) { return wg[r * VPL + j]; },
                                 [&](int j) { return wu[r * VPL + j]; }, m.act, vec, VPL, g, u);
            store_h<N>(g, u, hcol + r, ldh);
        }
    } else {
        const int iters = vec >> 5;
        for (int r = 0; r < R; ++r) {
            const uint32_t rg = sg + (uint32_t)(r * vec * 16), ru = su + (uint32_t)(r * vec * 16);
            float g[N], u[N];
            gate_up_dots<N, 0>([&](int j) { return lds128(rg + (uint32_t)((lane + 32 * j) * 16)); },
                               [&](int j) { return lds128(ru + (uint32_t)((lane + 32 * j) * 16)); },
                               m.act, vec, iters, g, u);
            store_h<N>(g, u, hcol + r, ldh);
        }
        release_slot(m, slot);
    }
}

// All RR rows of a register-cached down slot at once: each activation vector
// is loaded once and applied to every row (w[r * VPL + j] = row r, vector j).
template <int N, int VPL, int RR>
__device__ __forceinline__ void down_rows_regs(const uint4 (&w)[RR * VPL], uint32_t act, int vec,
                                               float (&a)[RR][N]) {
    constexpr int P = Chains<N * RR>::P;
    const int lane = threadIdx.x & 31;
    float acc[RR][N][P];
#pragma unroll
    for (int r = 0; r < RR; ++r)
#pragma unroll
        for (int t = 0; t < N; ++t)
#pragma unroll
            for (int p = 0; p < P; ++p) acc[r][t][p] = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
#pragma unroll
        for (int t = 0; t < N; ++t) {
            const Bf16x8 xa(lds128(act + (uint32_t)((t * vec + lane + 32 * j) * 16)));
#pragma unroll
            for (int r = 0; r < RR; ++r) {
                const Bf16x8 fw(w[r * VPL + j]);
#pragma unroll
                for (int q = 0; q < 8; ++q) fma_bf16(acc[r][t][q % P], fw.h[q], xa.h[q]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RR; ++r)
#pragma unroll
        for (int t = 0; t < N; ++t) a[r][t] = warp_sum(sum_chains<P>(acc[r][t]));
}

// One down slot: R rows of W_down of vec vectors.  VPL > 0 (= vec / 32,
// R = 32 / VPL): the lane's share is copied to registers, the slot released,
// and all rows computed together.
template <int N, int VPL>
__device__ __forceinline__ void down_slot(const Smem& m, int slot, int R, int vec, int n_slots,
                                          __nv_bfloat16* ycol, int64_t ldy) {
    const int lane = threadIdx.x & 31;
    const uint32_t sw = m.buf(slot);
    if constexpr (VPL > 0 && DownRegSlots<VPL>::value > 0) {
        constexpr int RR = 32 / VPL;
        uint4 w[RR * VPL];
#pragma unroll
        for (int i = 0; i < RR * VPL; ++i) w[i] = lds128(sw + (uint32_t)((i * 32 + lane) * 16));
        release_slot(m, slot);
        if constexpr (N <= DownRegSlots<VPL>::value) {
            float a[RR][N];
            down_rows_regs<N, VPL, RR>(w, m.act, vec, a);
#pragma unroll
            for (int r = 0; r < RR; ++r) {
#pragma unroll
                for (int t = 0; t < N; ++t)
                    if (lane == t) ycol[t * ldy + r] = __float2bfloat16_rn(a[r][t]);
            }
        } else {
            down_groups_regs<VPL, RR>(w, m.act, vec, n_slots, ycol, ldy);
        }
    } else {
        const int iters = vec >> 5;
        for (int r = 0; r < R; ++r) {
            const uint32_t rw = sw + (uint32_t)(r * vec * 16);
            float a[N];
            down_dots<N, 0>([&](int j) { return lds128(rw + (uint32_t)((lane + 32 * j) * 16)); },
                            m.act, vec, iters, a);
            store_y<N>(a, ycol + r, ldy);
        }
        release_slot(m, slot);
    }
}

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
                                [&]<int N>(int it, int slot) {
        const ThinUnit un = U[it / ipe];
        __nv_bfloat16* hcol = h + (int64_t)un.row0 * I + (it % ipe) * R;
        gate_up_slot<N, VPL>(m, slot, R, vec, un.n, hcol, I);
    });
    if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
}

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
                                        [&]<int N>(int it, int slot) {
            const ThinUnit un = U[it / ipe];
            __nv_bfloat16* ycol = y + (int64_t)un.row0 * H + (it % ipe) * R;
            down_slot<N, VPL>(m, slot, R, vec, un.n, ycol, H);
        });
        if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
    }
    if (sr.out) {   // fused combine; every thread has waited for the gate/up kernel
        grid_dep_wait();
        combine_if_last(sr, sp, hdr, y, H);
    }
}

// Invalidates a ring's barriers (thread 0) so that its shared memory can be
// set up again for another geometry.  Every thread is past its last wait.
__device__ __forceinline__ void smem_teardown(const Smem& m) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < m.slots; ++s) {
            for (int p = 0; p < m.producers; ++p) mbar_inval(m.full_of(p, s));
            mbar_inval(m.empty(s));
        }
        mbar_inval(m.act_full());
        mbar_inval(m.act_free());
    }
}

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
template <int VG, int VD>
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
        const Smem m = smem_setup(smem, stage_g, slots_g, act_g, kProducers, nc);
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
                ok = produce(
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
            ok = consume<16>(m, rg, ipe, sp.units, warp - kProducers, nc, wait_cycles,
                             [&]<int N>(int it, int slot) {
                const ThinUnit un = sp.units[it / ipe];
                __nv_bfloat16* hcol = h + (int64_t)un.row0 * I + (it % ipe) * Rg;
                gate_up_slot<N, VG>(m, slot, Rg, vec, un.n, hcol, I);
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
        const Smem m = smem_setup(smem, stage_d, slots_d, act_d, kProducers, nc);
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
                const int pre = rg.cnt < m.slots ? (rg.cnt > 0 ? rg.cnt : 0) : m.slots;
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
                ok = produce(
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
            ok = consume<kExact>(m, rg, ipe, sp.units, warp - kProducers, nc, wait_cycles,
                                 [&]<int N>(int it, int slot) {
                const ThinUnit un = sp.units[it / ipe];
                __nv_bfloat16* ycol = y + (int64_t)un.row0 * H + (it % ipe) * Rd;
                down_slot<N, VD>(m, slot, Rd, vec, un.n, ycol, H);
            });
        }
        if (!ok) set_status(hdr, MOE_ERR_TIMEOUT);
    }
    combine_spread(sr, sp.inv_perm, sp.gates, hdr, y, H, wait_cycles);
}

// Rows per item so that a weight slot holds at most kStageTarget bytes (at
// least one row); a power of two, so it divides I and H (multiples of 256).
int rows_per_item(int row_bytes) {
    int r = 1;
    while (2 * r * row_bytes <= kStageTarget && r < 256) r *= 2;
    return r;
}

struct Geometry {
    int R, stage, slots, act, smem;
};

// act_tokens: most slots any unit can hold here (the activation buffer size);
// pad4: round the buffer up to a multiple of 4 rows (the down kernel's
// grouped register path reads whole groups of 4; gate/up reads exactly the
// unit's rows).  Every H, I the library accepts fits kSmemBudget.
Geometry geometry(int row_bytes, int act_row_bytes, int act_tokens, bool pad4) {
    Geometry g;
    g.R = rows_per_item(row_bytes);
    g.stage = g.R * row_bytes;
    g.act = (pad4 ? (act_tokens + 3) / 4 * 4 : act_tokens) * act_row_bytes;
    g.slots = (kSmemBudget - g.act) / g.stage;
    if (g.slots > kMaxSlots) g.slots = kMaxSlots;
    if (g.slots < 2) g.slots = 2;
    g.smem = g.slots * g.stage + g.act + 8 * kBarriers;
    return g;
}

// Producers + consumers, with fewer consumers than slots (slot protocol).
int threads_for(const Geometry& g, int producers) {
    int consumers = kWarps - producers;
    if (consumers > g.slots - 1) consumers = g.slots - 1;
    if (consumers < 1) consumers = 1;
    return 32 * (producers + consumers);
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

template <int VG, int VD>
cudaError_t launch_layer(const __nv_bfloat16* x, int k, int H, int I, const __nv_bfloat16* Wg,
                         const __nv_bfloat16* Wu, const __nv_bfloat16* Wd, const Plan& plan,
                         const Geometry& g1, const Geometry& g2, __nv_bfloat16* h,
                         __nv_bfloat16* y, int num_sms, cudaStream_t s, const SelfRoute& sr) {
    static std::atomic<int> done[kMaxDevices];
    cudaError_t e = smem_limit_once(thin_layer_kernel<VG, VD>, kSmemBudget + 1024, done);
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
    return cudaLaunchKernelEx(&cfg, thin_layer_kernel<VG, VD>, x, k, H, I, g1.R, g2.R, Wg, Wu,
                              Wd, plan.wslot, plan.hdr, h, y, g1.stage, g1.slots, g1.act,
                              g2.stage, g2.slots, g2.act, sr, main_wait_cycles());
}

}  // namespace

bool thin_layer_fused(int H, int I) {
    return (H == 4096 && I == 2048) || (H == 512 && I == 256);
}

cudaError_t launch_thin_layer(const __nv_bfloat16* x, int k, int H, int I,
                              const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                              const __nv_bfloat16* Wd, const Plan& plan, int64_t max_slots,
                              __nv_bfloat16* h, __nv_bfloat16* y_sorted, int num_sms,
                              cudaStream_t s, const SelfRoute& sr) {
    const int act_tokens =
        (int)std::min<int64_t>(plan.unit_tokens, std::max<int64_t>(max_slots, 1));
    const Geometry g1 = geometry(2 * H * 2, H * 2, act_tokens, false);
    const Geometry g2 = geometry(I * 2, I * 2, act_tokens, true);
    if (g1.stage != kStageTarget || g2.stage != kStageTarget)
        return cudaErrorInvalidConfiguration;
    if (H == 4096 && I == 2048)
        return launch_layer<16, 8>(x, k, H, I, Wg, Wu, Wd, plan, g1, g2, h, y_sorted, num_sms, s, sr);
    if (H == 512 && I == 256)
        return launch_layer<2, 1>(x, k, H, I, Wg, Wu, Wd, plan, g1, g2, h, y_sorted, num_sms, s, sr);
    return cudaErrorInvalidConfiguration;
}

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
