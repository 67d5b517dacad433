// thin_dev.cuh -- shared device code of the CUDA-core weight-streaming
// kernels (thin.cu: the gate/up and down kernels; thin_layer.cu: the
// one-launch decode layer): the slot ring, its producer and consumers, the
// mixed-precision dot products, and the host-side ring geometry.
//
// The path: weight-streaming expert path for experts holding fewer slots
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
#pragma once

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

// [slots x stage_bytes weight ring][activation buffers][barriers]
// Each producer's copies into a slot complete on its own full barrier
// (full(s) for producer 0, full2(s) for producer 1), so a producer that
// stops early can still wait for exactly the copies it issued.  With two
// activation buffers, unit i of a range is staged in buffer i % 2, so the
// next unit's rows arrive while the current one is consumed.
constexpr int kBarriers = 3 * kMaxSlots + 4;
struct Smem {
    uint32_t base;       // shared addresses
    uint32_t act;        // the activation buffer the consumers read
    uint32_t bars;
    uint32_t act_bytes;  // per buffer
    int act_bufs;
    int stage_bytes;
    int slots;
    int producers;
    __device__ uint32_t buf(int s) const { return base + (uint32_t)(s * stage_bytes); }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (kMaxSlots + s); }
    __device__ uint32_t act_buf(int b) const { return act + (uint32_t)b * act_bytes; }
    __device__ uint32_t act_full(int b = 0) const {
        return bars + 8u * (b == 0 ? 2 * kMaxSlots : 3 * kMaxSlots + 2);
    }
    __device__ uint32_t act_free(int b = 0) const {
        return bars + 8u * (b == 0 ? 2 * kMaxSlots + 1 : 3 * kMaxSlots + 3);
    }
    __device__ uint32_t full2(int s) const { return bars + 8u * (2 * kMaxSlots + 2 + s); }
    // full barrier of producer p
    __device__ uint32_t full_of(int p, int s) const { return p == 0 ? full(s) : full2(s); }
};

// act_bytes: one activation buffer; act_bufs: 1 or 2 buffers.
__device__ __forceinline__ Smem smem_setup(uint8_t* smem, int stage_bytes, int slots,
                                           int act_bytes, int producers, int consumers,
                                           int act_bufs = 1) {
    Smem m;
    m.base = smem_u32(smem);
    m.stage_bytes = stage_bytes;
    m.slots = slots;
    m.producers = producers;
    m.act = m.base + (uint32_t)(slots * stage_bytes);
    m.act_bytes = (uint32_t)act_bytes;
    m.act_bufs = act_bufs;
    m.bars = m.act + (uint32_t)(act_bytes * act_bufs);
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            for (int p = 0; p < producers; ++p) mbar_init(m.full_of(p, s), 1);
            mbar_init(m.empty(s), 1);
        }
        for (int b = 0; b < act_bufs; ++b) {
            mbar_init(m.act_full(b), 1);
            mbar_init(m.act_free(b), consumers);
        }
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
template <typename C>   // uint32_t when every cost fits, else int64_t
__device__ __forceinline__ int item_at(const ThinUnit* units, int n_units, int ipe, C c) {
    int lo = 0, hi = n_units - 1;   // largest u with ipe * cost_before <= c
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((C)units[mid].cost_before * (C)ipe <= c) lo = mid;
        else hi = mid - 1;
    }
    const C w = (C)thin_unit_cost(units[lo].n);
    const C off = c - (C)units[lo].cost_before * (C)ipe;
    const C k = (off + w - 1) / w;
    return lo * ipe + (int)(k < (C)ipe ? k : (C)ipe);
}

// This CTA's contiguous share of the items of n_units units of total cost
// `weight` (per item), of (about) equal total cost.  The arithmetic is 32-bit
// where the products fit (every self-routed batch: it runs before the first
// weight copy, so its length matters there), 64-bit otherwise.
__device__ __forceinline__ Range cta_range(const ThinUnit* units, int n_units, int weight, int ipe) {
    Range r;
    if (n_units <= 0) {
        r.beg = r.cnt = 0;
        r.u_first = 0;
        r.u_last = -1;
        return r;
    }
    const int64_t total = (int64_t)weight * ipe;
    const bool last = blockIdx.x + 1 == gridDim.x;
    if (total * gridDim.x < (int64_t)1 << 32) {
        const uint32_t t = (uint32_t)total;
        r.beg = item_at<uint32_t>(units, n_units, ipe, t * blockIdx.x / gridDim.x);
        const int end = last ? n_units * ipe
                             : item_at<uint32_t>(units, n_units, ipe,
                                                 t * (blockIdx.x + 1) / gridDim.x);
        r.cnt = end - r.beg;
    } else {
        r.beg = item_at<int64_t>(units, n_units, ipe, total * blockIdx.x / gridDim.x);
        const int end = last ? n_units * ipe
                             : item_at<int64_t>(units, n_units, ipe,
                                                total * (blockIdx.x + 1) / gridDim.x);
        r.cnt = end - r.beg;
    }
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
// (copy_act) into buffer i % kBufs (i: the unit's place in the range) once
// the consumers have released the unit that used that buffer before.  Items
// [0, pre) (pre <= slots) were already issued into slots [0, pre).  While a
// slot is still in use the lane sleeps in try_wait.  Each wait gives up after
// `limit` cycles; then the copies already issued are waited for (full bound)
// and it returns false.
template <int kBufs = 1, typename ItemFn, typename ActFn>
__device__ bool produce(const Smem& m, int producer, const Range& rg, bool stager,
                        ItemFn copy_item, ActFn copy_act, long long limit, int pre = 0) {
    if (rg.cnt <= 0) return true;
    int last_round[kMaxSlots];
    for (int s = 0; s < kMaxSlots; ++s) last_round[s] = s < pre ? 0 : -1;
    const int n_units = stager ? rg.u_last - rg.u_first + 1 : 0;
    int act_issued = 0;                       // units whose activations are staged
    for (; act_issued < kBufs && act_issued < n_units; ++act_issued)
        copy_act(rg.u_first + act_issued, m.act_buf(act_issued), m.act_full(act_issued));
    // Unit i goes to buffer i % kBufs once the release of unit i - kBufs
    // (that buffer's use number i / kBufs - 1) has completed.
    auto stage_next = [&]() {
        const int b = act_issued % kBufs;
        copy_act(rg.u_first + act_issued, m.act_buf(b), m.act_full(b));
        ++act_issued;
    };
    auto freed_parity = [&]() { return (uint32_t)((act_issued / kBufs - 1) & 1); };
    auto try_stage = [&]() {   // never blocks
        if (act_issued < n_units && mbar_test_wait(m.act_free(act_issued % kBufs), freed_parity()))
            stage_next();
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
        if (!mbar_wait_for(m.act_free(act_issued % kBufs), freed_parity(), limit, nullptr)) {
            ok = false;
            break;
        }
        stage_next();
    }
    if (!ok) {
        // Let the copies already issued land before the CTA exits.
        for (int s = 0; s < m.slots; ++s)
            if (last_round[s] >= 0)
                (void)mbar_wait(m.full_of(producer, s), (uint32_t)(last_round[s] & 1));
        for (int b = 0; b < kBufs; ++b) {
            const int uses = (act_issued - b + kBufs - 1) / kBufs;   // units staged in b
            if (uses > 0) (void)mbar_wait(m.act_full(b), (uint32_t)((uses - 1) & 1));
        }
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

// Consumer warp c of nc.  For each unit of the range (the i-th, in buffer
// i % kBufs): wait for its activations, then for the warp's items of that
// unit (seq = c mod nc) wait for the slot and run
// item.template operator()<N>(item, slot, mu) with N the unit's slot count
// and mu the ring with its act pointing at the unit's buffer (the item
// releases the slot), then release the activations.  Returns false when a
// wait ran past `limit` cycles.
template <int kExact, int kBufs = 1, typename ItemFn>
__device__ bool consume(const Smem& m, const Range& rg, int ipe, const ThinUnit* units, int c,
                        int nc, long long limit, ItemFn item) {
    const int lane = threadIdx.x & 31;
    for (int u = rg.u_first; u <= rg.u_last; ++u) {
        const int i = u - rg.u_first, b = i % kBufs;
        if (!warp_wait(m.act_full(b), (uint32_t)((i / kBufs) & 1), limit)) return false;
        Smem mu = m;
        mu.act = m.act_buf(b);
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
                item.template operator()<N>(rg.beg + seq, slot, mu);
                slot += nc;            // nc < slots: at most one wrap
                if (slot >= m.slots) {
                    slot -= m.slots;
                    ++round;
                }
            }
        });
        if (!ok) return false;
        __syncwarp();
        if (lane == 0) mbar_arrive(m.act_free(b));
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

// Invalidates a ring's barriers (thread 0) so that its shared memory can be
// set up again for another geometry.  Every thread is past its last wait.
__device__ __forceinline__ void smem_teardown(const Smem& m) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < m.slots; ++s) {
            for (int p = 0; p < m.producers; ++p) mbar_inval(m.full_of(p, s));
            mbar_inval(m.empty(s));
        }
        for (int b = 0; b < m.act_bufs; ++b) {
            mbar_inval(m.act_full(b));
            mbar_inval(m.act_free(b));
        }
    }
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
// unit's rows); bufs: activation buffers (act is one buffer's bytes).  Every
// H, I the library accepts fits kSmemBudget.
Geometry geometry(int row_bytes, int act_row_bytes, int act_tokens, bool pad4, int bufs = 1) {
    Geometry g;
    g.R = rows_per_item(row_bytes);
    g.stage = g.R * row_bytes;
    g.act = (pad4 ? (act_tokens + 3) / 4 * 4 : act_tokens) * act_row_bytes;
    g.slots = (kSmemBudget - bufs * g.act) / g.stage;
    if (g.slots > kMaxSlots) g.slots = kMaxSlots;
    if (g.slots < 2) g.slots = 2;
    g.smem = g.slots * g.stage + bufs * g.act + 8 * kBarriers;
    return g;
}

// Producers + consumers, with fewer consumers than slots (slot protocol).
int threads_for(const Geometry& g, int producers) {
    int consumers = kWarps - producers;
    if (consumers > g.slots - 1) consumers = g.slots - 1;
    if (consumers < 1) consumers = 1;
    return 32 * (producers + consumers);
}

}  // namespace
}  // namespace moe
