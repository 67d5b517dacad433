// moe_internal.cuh -- shared definitions of libmoe's CUDA translation units:
// limits, the workspace header, and the launchers each stage exports to the
// C ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

#include "moe.h"

namespace moe {

constexpr int kMaxK = 8;             // experts per token
constexpr int kMaxE = 1024;          // experts per layer
constexpr int kThinMaxTokens = 32;   // slots one weight-streaming expert may hold
constexpr int kPermChunk = 2048;     // slots per block in the route-list kernels
// The row gather of a batch with fat experts runs in two parts: the gather
// kernel copies the rows of the first 1/kGatherFirstDen of the pair tiles;
// the gate/up GEMM launch over those tiles copies the other rows with its
// idle warps, for the second launch over the other pair tiles.
constexpr int kGatherFirstDen = 3;
constexpr int kTileM = 128;          // rows (slots) per grouped-GEMM tile
constexpr int kMaxHidden = 16384;    // H and I (a weight-streaming stage holds a row)

// First 256 bytes of every workspace.
struct WsHeader {
    int32_t status;        // moe_status recorded by kernels (sticky)
    int32_t n_fat_tiles;   // grouped-GEMM row tiles built by the planner
    int32_t n_thin;        // work units on the weight-streaming path
    int32_t thin_weight;   // sum of thin_unit_cost over those units
    int32_t n_thin_mma;    // thin experts on the tensor-core streaming kernel
    int32_t n_solo;        // fat experts' leftover 128-row tiles (one-CTA GEMM)
    int32_t ticket;        // CTAs of a streaming down kernel done (fused combine)
    uint32_t layer_sync;   // grid-wide waits of the one-kernel decode layer (after gate/up,
                           // before the combine): CTA arrivals, monotonic; each wait
                           // ends at the next multiple of the grid size
    int32_t reserved[56];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// One grouped-GEMM row tile: rows [row0, row0 + rows) of expert `expert`
// in sorted-slot order (rows may be 0 for the second tile of a pair).
struct FatTile {
    int32_t expert;
    int32_t row0;
    int32_t rows;
    int32_t pad;
};

// One weight-streaming work unit: up to `unit_tokens` consecutive sorted slots
// [row0, row0 + n) of expert `expert`.  An expert with more slots than a
// unit holds is split into several units, each streaming the expert's weights.
struct ThinUnit {
    int32_t expert;
    int32_t row0;
    int32_t n;
    int32_t cost_before;   // sum of thin_unit_cost over the preceding units
};

// Pair tiles of the first gather part (of n_pairs).
__host__ __device__ inline int gather_first_pairs(int n_pairs) {
    return (n_pairs + kGatherFirstDen - 1) / kGatherFirstDen;
}

// Relative cost of one weight row of a unit with n slots on the CUDA-core
// streaming path (used to split units' rows evenly over CTAs).  Measured per
// row with every SM streaming (full-size decode layers, batches 1-4): 1,
// 1.05-1.07, 1.12-1.17 and 1.27-1.30 times a one-slot row for 1..4 slots
// (register-cached rows, the FMAs partly hidden under the HBM read); beyond
// 4 slots rows are read from shared memory and the cost grows with n.
__host__ __device__ inline int thin_unit_cost(int n) {
    return n <= 1 ? 20 : n == 2 ? 21 : n == 3 ? 23 : 13 * (n + 2) / 3;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kMaxDevices = 64;

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (`done`: one flag per device, per kernel).
template <typename K>
cudaError_t smem_limit_once(K kernel, int bytes, std::atomic<int> (&done)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

// Programmatic dependent launch is on for the calling thread's launches while
// a PdlScope(true) is alive.  The layer entry points turn it on for small
// batches (decode), where kernel boundaries are a large share of the step;
// at the prefill chunk, successor CTAs waiting on the SMs cost the GEMMs
// ~1.5% (measured), so it stays off there.
extern thread_local bool t_pdl;
struct PdlScope {
    bool prev;
    explicit PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
    ~PdlScope() { t_pdl = prev; }
};

// Limit (SM cycles) of each main-loop mbarrier wait in the calling thread's
// launches of the expert kernels: the default bound (~2 s), unless
// moe_debug_set_wait_limit shortened it for a test.
extern thread_local long long t_wait_cycles;   // 0: default
long long main_wait_cycles();

// Launches `kernel` on s, with programmatic stream serialisation when enabled
// (it may then start while the previous kernel on s finishes; the kernel calls
// grid_dep_wait() before touching data of earlier kernels).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = t_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl, and with coop also a cooperative launch (every block resident
// at once, or the launch fails): for kernels whose blocks wait on one another.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_coop(bool coop, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                            size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (t_pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (coop) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Planner outputs (the split of experts between the expert kernels).  A thin
// expert (0 < count < fat_threshold) with at least thin_mma_min slots streams
// its weights through the tensor cores (one FatTile of <= kThinMaxTokens rows
// in mma_tiles); the others take the CUDA-core streaming kernel (units).
struct Plan {
    FatTile* tiles;      // [max_fat_tiles(P, E)], in pairs of one expert
    FatTile* solo_tiles; // [E]: experts with a single tile (at most kTileM slots)
    ThinUnit* units;     // [max_thin_units(E, unit_tokens)], expert-major
    FatTile* mma_tiles;  // [E]
    WsHeader* hdr;
    int32_t fat_threshold;
    int32_t unit_tokens; // slots per weight-streaming unit (thin_unit_tokens)
    int32_t thin_mma_min;
    // Weight blocks: expert e's matrices are block wslot[e] of W_gate / W_up /
    // W_down, which hold n_wblocks blocks (wslot == nullptr: block e, E blocks).
    const int32_t* wslot;
    int32_t n_wblocks;
};

// Weight block of expert e (see Plan::wslot).
__device__ __forceinline__ int weight_block(const int32_t* wslot, int e) {
    return wslot ? __ldg(wslot + e) : e;
}

// Small batches route inside the streaming kernels: with at most
// kSelfRouteSlots token slots, every touched expert thin and on one streaming
// kernel (CUDA cores, each expert in one unit; or tensor cores, each expert
// one tile), each CTA of the gate/up kernel computes the top-k,
// the route lists and the units of the whole batch in shared memory
// (small_plan.cuh) instead of reading a plan written by the router and
// route-list kernels, CTA 0 stores them, the down kernel reads them, and the
// last CTA of the down kernel combines the batch: a decode step is two
// launches, and the weight stream starts right after the first one's wait.
// logits == nullptr: the kernels read the Plan instead.  Larger batches run
// faster through the router and route-list kernels (measured with up to 256
// slots routed this way, 4-layer decode sweep: batch 8 / 16 / 24 in 871 /
// 1121 / 1290 us planned vs 993 / 1503 / 2068 us): every gate/up CTA routes
// the batch's tokens a warp each, in turn, before its first weight copy, and
// a hot expert's activation rows arrive one row per copy.
constexpr int kSelfRouteSlots = 32;
struct SelfRoute {
    const float* logits;   // [T, E] fp32
    int32_t T, E, k;
    // Written by CTA 0 of the gate/up kernel as the router, route-list and
    // planner kernels would write them; read back by the down kernel.
    int32_t* idx;          // [T * k]
    float* gates;          // [T * k]
    int32_t* counts;       // [E]
    int32_t* offsets;      // [E + 1]
    int32_t* perm;         // [T * k]
    int32_t* inv_perm;     // [T * k]
    ThinUnit* units;       // the plan's unit list
    // Layer output [T, H]: the last CTA of the down kernel to finish combines
    // the batch (the combine kernel's arithmetic) and no combine is launched.
    __nv_bfloat16* out;
};


// By default every thin expert streams on the tensor cores once at least this
// many 128-row gate/up work items can exist (touched experts x I/128), and
// on CUDA cores below it.  Measured on GB300 (H=4096, I=2048): decode batch 2
// (<= 256 items) is faster on CUDA cores, batch 4 (<= 512) on tensor cores.
constexpr int kThinMmaAutoItems = 384;

// Fat tiles come in pairs per expert: sum_e 2*ceil(c_e/256) <= P/128 + 2E.
inline int64_t max_fat_tiles(int64_t P, int E) { return P / kTileM + 2 * (int64_t)E + 2; }
inline int64_t max_thin_units(int E, int unit_tokens) {
    return (int64_t)E * ((kThinMaxTokens + unit_tokens - 1) / unit_tokens);
}
// Slots per weight-streaming unit for these sizes (their activations are
// staged in shared memory together).
int thin_unit_tokens(int H, int I);

// Launchers (all asynchronous on `s`; they return the launch's cudaError_t).
cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int32_t* idx, float* gates, cudaStream_t s);

// flags[e] = 1 for every expert e in idx[0, P) (flags: device-visible memory,
// e.g. mapped pinned host memory; never cleared here).
cudaError_t launch_mark_touched(const int32_t* idx, int64_t P, int E, uint8_t* flags,
                                cudaStream_t s);

// Route lists; when plan != nullptr the planner runs in the same kernels.
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, int32_t* chunk_hist,
                           int32_t* chunk_base, WsHeader* hdr,
                           const Plan* plan, cudaStream_t s);
size_t permute_scratch_ints(int64_t P, int E);   // chunk_hist + chunk_base

cudaError_t launch_plan(const int32_t* counts, const int32_t* offsets, int E,
                        const Plan& plan, cudaStream_t s);

// part: 0 every row; 1 the rows of the first gather_first_pairs() pair
// tiles; 2 the other rows (the later pair tiles, solo and tensor-core tiles).
cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* perm, int k,
                          int H, const Plan& plan, __nv_bfloat16* x_sorted,
                          int num_sms, cudaStream_t s, int part = 0);

// max_slots: an upper bound of any expert's slot count (sizes the staged
// activation buffer; units never hold more than plan.unit_tokens).
// sr != nullptr: the kernels route the batch themselves (see SelfRoute).
cudaError_t launch_thin_gate_up(const __nv_bfloat16* x, const int32_t* perm, int k, int H,
                                int I, const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                                const Plan& plan, int64_t max_slots, __nv_bfloat16* h,
                                int num_sms, cudaStream_t s, const SelfRoute* sr = nullptr);

cudaError_t launch_thin_down(const __nv_bfloat16* h, int H, int I, const __nv_bfloat16* Wd,
                             const Plan& plan, int64_t max_slots, __nv_bfloat16* y_sorted,
                             int num_sms, cudaStream_t s, const SelfRoute* sr = nullptr);

// A self-routed batch on the CUDA-core streaming path as one cooperative
// kernel: gate/up, a grid-wide wait (bounded) until every CTA's h rows are
// stored, down (its first weight rows copied before that wait), and the
// last CTA's combine.  thin_layer_fused(H, I) says whether it is built for
// those sizes; otherwise the two kernels above run.
bool thin_layer_fused(int H, int I);
cudaError_t launch_thin_layer(const __nv_bfloat16* x, int k, int H, int I,
                              const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                              const __nv_bfloat16* Wd, const Plan& plan, int64_t max_slots,
                              __nv_bfloat16* h, __nv_bfloat16* y_sorted, int num_sms,
                              cudaStream_t s, const SelfRoute& sr);

// Weight streaming on tcgen05 for the thin experts in plan.mma_tiles:
// gate_up: h[rows] = silu(x_sorted[rows] Wg_e^T) * (x_sorted[rows] Wu_e^T);
// down: y[rows] = h[rows] Wd_e^T.  x_sorted / h hold rows_alloc rows.
// sr != nullptr: the batch routes itself (see SelfRoute); the gate/up kernel
// then reads the tokens' rows of x [sr->T, H] directly (x_sorted unused).
cudaError_t launch_thin_mma_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                    const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H,
                                    int I, const Plan& plan, __nv_bfloat16* h, int num_sms,
                                    cudaStream_t s, const SelfRoute* sr = nullptr,
                                    const __nv_bfloat16* x = nullptr);
// down with sr->out set: the combine is fused (a cooperative launch; every
// CTA combines its share of out after a bounded grid-wide wait), by the
// batch's own plan (sr->logits set) or, for a planned batch whose only expert
// kernel this is, by sr's route lists (inv_perm, gates; sr->logits null).
cudaError_t launch_thin_mma_down(const __nv_bfloat16* h, int64_t rows_alloc,
                                 const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                                 __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s,
                                 const SelfRoute* sr = nullptr);

// One-CTA grouped GEMMs (tcgen05 cta_group::1, 128 x 256 tiles) over
// plan.solo_tiles, the same products as the pair GEMMs below.
cudaError_t launch_gemm_solo_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                     const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H,
                                     int I, const Plan& plan, __nv_bfloat16* h, int num_sms,
                                     cudaStream_t s);
cudaError_t launch_gemm_solo_down(const __nv_bfloat16* h, int64_t rows_alloc,
                                  const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                                  __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s);

// Grouped GEMMs on tcgen05.  gate_up: h = silu(A Wg^T) * (A Wu^T) for the
// fat tiles, A = x_sorted [rows_alloc, H].  down: y = h Wd^T, A = h.
// gate_up part: 0 every pair tile; 1 the first gather_first_pairs() pair
// tiles, the launch also gathering the gather's part-2 rows from x (by perm
// and k) into x_sorted; 2 the other pair tiles.
cudaError_t launch_gemm_gate_up(const __nv_bfloat16* x_sorted, int64_t rows_alloc,
                                const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int H, int I,
                                const Plan& plan, __nv_bfloat16* h, int num_sms,
                                cudaStream_t s, int part = 0, const __nv_bfloat16* x = nullptr,
                                const int32_t* perm = nullptr, int k = 0);
cudaError_t launch_gemm_down(const __nv_bfloat16* h, int64_t rows_alloc,
                             const __nv_bfloat16* Wd, int H, int I, const Plan& plan,
                             __nv_bfloat16* y_sorted, int num_sms, cudaStream_t s);

cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* inv_perm,
                           const float* gates, int T, int k, int H,
                           __nv_bfloat16* out, int num_sms, cudaStream_t s);

// Experts to copy: entry j copies expert src_e[j] of the source matrices
// into block dst_e[j] of the destination matrices.
struct ExpertCopyList {
    int32_t n;
    int32_t src_e[kMaxE];
    int32_t dst_e[kMaxE];
};

// The device's pointer to pinned host memory `host` (cudaHostAlloc or
// cudaHostRegister); cudaErrorInvalidValue for any other memory.
cudaError_t device_view_of_host(const void* host, const void** dev);

// For each list entry and matrix m < 3: copies expert_bytes from
// src[m] + src_e * expert_bytes (device-visible host memory, see
// device_view_of_host) to dst[m] + dst_e * expert_bytes (device), in one
// kernel whose CTAs drive the host link with SM loads.  Every pointer and
// expert_bytes must be 16-byte aligned (else cudaErrorInvalidValue, nothing
// launched).
cudaError_t launch_expert_copy(const ExpertCopyList& list, const void* const src[3],
                               void* const dst[3], size_t expert_bytes, cudaStream_t s);

// Routes `logits` into the routing buffers of a moe_forward workspace and
// sets flags[e] = 1 for each expert the layer touches (asynchronous on s).
moe_status mark_touched_experts(const moe_shape* shape, const float* logits, void* ws,
                                size_t ws_bytes, uint8_t* flags, cudaStream_t s);

// moe_forward with expert e's weights in block wslot[e] (device table of E
// entries) of W_gate / W_up / W_down, which hold n_wblocks blocks.
moe_status forward_blocks(const moe_shape* shape, const float* logits, const moe_bf16* x,
                          const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                          const int32_t* wslot, int32_t n_wblocks, moe_bf16* out, void* ws,
                          size_t ws_bytes, moe_stream_t stream);

// Validates a moe_shape as every entry point does (sets moe_last_error()).
moe_status check_shape_status(const moe_shape* shape);

// Sets the calling thread's moe_last_error() message (printf format).
void set_last_error(const char* fmt, ...);

// Records a device-side condition in the workspace status word (first one wins).
__device__ __forceinline__ void set_status(WsHeader* hdr, int code) {
    atomicCAS(&hdr->status, 0, code);
}

}  // namespace moe
