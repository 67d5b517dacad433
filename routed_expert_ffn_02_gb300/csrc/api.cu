// api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace layout and the launch sequence of each entry point.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

using namespace moe;

thread_local bool moe::t_pdl = false;
thread_local long long moe::t_wait_cycles = 0;

long long moe::main_wait_cycles() {
    return t_wait_cycles > 0 ? t_wait_cycles : ptx::kWaitCycles;
}

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

}  // namespace

void moe::set_last_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

namespace {

moe_status ok() {
    g_err[0] = '\0';
    return MOE_OK;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct DeviceInfo {
    int checked = 0;
    int supported = 0;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Current device must be sm_103 (the library carries sm_103a code only).
moe_status device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.checked) {
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.supported = (d.cc_major == 10 && d.cc_minor == 3);
        d.checked = 1;
    }
    if (!d.supported)
        return fail(MOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; libmoe is built for sm_103a",
                    dev, d.cc_major, d.cc_minor);
    *out = d;
    return MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status check_route_args(int32_t T, int32_t E, int32_t k) {
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (E < 1 || E > kMaxE) return fail(MOE_ERR_INVALID_ARG, "E = %d outside [1, %d]", E, kMaxE);
    if (k < 1 || k > kMaxK || k > E)
        return fail(MOE_ERR_INVALID_ARG, "k = %d outside [1, min(E, %d)]", k, kMaxK);
    if ((int64_t)T * k > (int64_t)INT32_MAX - kTileM)
        return fail(MOE_ERR_INVALID_ARG, "T*k = %lld too large", (long long)T * k);
    return MOE_OK;
}

moe_status check_shape(const moe_shape* sh) {
    if (!sh) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
    moe_status st = check_route_args(sh->T, sh->E, sh->k);
    if (st != MOE_OK) return st;
    if (sh->H < 256 || sh->H % 256) return fail(MOE_ERR_INVALID_ARG, "H = %d is not a positive multiple of 256", sh->H);
    if (sh->I < 256 || sh->I % 256) return fail(MOE_ERR_INVALID_ARG, "I = %d is not a positive multiple of 256", sh->I);
    if (sh->H > kMaxHidden || sh->I > kMaxHidden)
        return fail(MOE_ERR_UNSUPPORTED, "H and I are limited to %d", kMaxHidden);
    if (sh->fat_threshold < 0 || sh->fat_threshold > kThinMaxTokens + 1)
        return fail(MOE_ERR_INVALID_ARG, "fat_threshold = %d outside [0, %d]", sh->fat_threshold,
                    kThinMaxTokens + 1);
    if (sh->thin_mma_min < 0 || sh->thin_mma_min > kThinMaxTokens + 1)
        return fail(MOE_ERR_INVALID_ARG, "thin_mma_min = %d outside [0, %d]", sh->thin_mma_min,
                    kThinMaxTokens + 1);
    return MOE_OK;
}

// thin_mma_min == 0 picks the streaming kernel from the shape: the tensor-core
// kernel's work items are 128-row weight blocks of whole experts, so it needs
// enough thin experts to fill the GPU; below that the CUDA-core kernel, which
// splits weight rows finely over all SMs, is faster.  At most min(E, T*k)
// experts are touched.
}  // namespace

moe_status moe::check_shape_status(const moe_shape* shape) { return check_shape(shape); }


namespace {

int thin_mma_min(const moe_shape* sh) {
    if (sh->thin_mma_min > 0) return sh->thin_mma_min;
    const int64_t touched = std::min<int64_t>(sh->E, (int64_t)sh->T * sh->k);
    return touched * (sh->I / 128) >= kThinMmaAutoItems ? 1 : kThinMaxTokens + 1;
}

// Small batches whose touched experts are all thin and on one streaming
// kernel (CUDA cores with one unit per expert, or tensor cores) are routed
// inside the streaming kernels and combined by the down kernel (see
// SelfRoute): no router, route-list, planner, gather or combine launch.  A
// token's k experts are distinct, so no expert holds more than T slots.
enum SelfMode { kPlanned = 0, kSelfUnits, kSelfMma };
SelfMode self_mode(const moe_shape* sh) {
    if ((int64_t)sh->T * sh->k > kSelfRouteSlots || sh->T >= sh->fat_threshold) return kPlanned;
    const int mm = thin_mma_min(sh);
    if (mm <= 1) return kSelfMma;
    if (sh->T < mm && sh->T <= thin_unit_tokens(sh->H, sh->I)) return kSelfUnits;
    return kPlanned;
}

// Which expert kernels can have work, given an upper bound of any expert's
// slot count (the planner decides on the device; a kernel with an empty
// list returns at once, but one that cannot have work is not launched).
struct ExpertKernels {
    bool fat, units, mma;
    bool gather() const { return fat || mma; }
};
ExpertKernels expert_kernels(const moe_shape* sh, int64_t fat_bound) {
    const int thr = sh->fat_threshold, mm = thin_mma_min(sh);
    ExpertKernels k;
    k.fat = fat_bound >= std::max(thr, 1);
    k.units = std::min(thr, mm) > 1;                     // counts in [1, min(thr, mm))
    k.mma = thr > mm && fat_bound >= mm;                 // counts in [mm, thr)
    return k;
}

Plan make_plan(const moe_shape* sh, FatTile* tiles, FatTile* solo_tiles, ThinUnit* units,
               FatTile* mma_tiles, WsHeader* hdr) {
    return Plan{tiles, solo_tiles, units, mma_tiles, hdr, sh->fat_threshold,
                thin_unit_tokens(sh->H, sh->I), thin_mma_min(sh), nullptr, sh->E};
}

// Bump allocator over the caller's workspace (256-byte aligned regions).
struct Carver {
    uint8_t* base;
    size_t off = 0;
    explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
    template <typename T>
    T* take(size_t count) {
        off = align_up(off, 256);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

int64_t rows_alloc(int64_t P) { return std::max<int64_t>(P, kTileM); }

struct FfnBufs {
    WsHeader* hdr;
    FatTile* tiles;
    FatTile* solo_tiles;
    ThinUnit* units;
    FatTile* mma_tiles;
    __nv_bfloat16* x_sorted;
    __nv_bfloat16* h;
};

struct FwdBufs {
    WsHeader* hdr;
    int32_t *idx, *counts, *offsets, *perm, *inv_perm, *chunk;
    float* gates;
    FatTile* tiles;
    FatTile* solo_tiles;
    ThinUnit* units;
    FatTile* mma_tiles;
    __nv_bfloat16* xy;   // x_sorted, later reused for y_sorted
    __nv_bfloat16* h;
};

size_t carve_ffn(const moe_shape* sh, void* ws, FfnBufs* b) {
    const int64_t P = (int64_t)sh->T * sh->k;
    Carver c(ws);
    b->hdr = c.take<WsHeader>(1);
    b->tiles = c.take<FatTile>((size_t)max_fat_tiles(P, sh->E));
    b->solo_tiles = c.take<FatTile>((size_t)sh->E);
    b->units = c.take<ThinUnit>((size_t)max_thin_units(sh->E, thin_unit_tokens(sh->H, sh->I)));
    b->mma_tiles = c.take<FatTile>((size_t)sh->E);
    b->x_sorted = c.take<__nv_bfloat16>((size_t)(rows_alloc(P) * sh->H));
    b->h = c.take<__nv_bfloat16>((size_t)(rows_alloc(P) * sh->I));
    return align_up(c.off, 256);
}

size_t carve_fwd(const moe_shape* sh, void* ws, FwdBufs* b) {
    const int64_t P = (int64_t)sh->T * sh->k;
    Carver c(ws);
    b->hdr = c.take<WsHeader>(1);
    b->idx = c.take<int32_t>((size_t)P);
    b->gates = c.take<float>((size_t)P);
    b->counts = c.take<int32_t>((size_t)sh->E);
    b->offsets = c.take<int32_t>((size_t)sh->E + 1);
    b->perm = c.take<int32_t>((size_t)P);
    b->inv_perm = c.take<int32_t>((size_t)P);
    b->chunk = c.take<int32_t>(permute_scratch_ints(P, sh->E));
    b->tiles = c.take<FatTile>((size_t)max_fat_tiles(P, sh->E));
    b->solo_tiles = c.take<FatTile>((size_t)sh->E);
    b->units = c.take<ThinUnit>((size_t)max_thin_units(sh->E, thin_unit_tokens(sh->H, sh->I)));
    b->mma_tiles = c.take<FatTile>((size_t)sh->E);
    b->xy = c.take<__nv_bfloat16>((size_t)(rows_alloc(P) * sh->H));
    b->h = c.take<__nv_bfloat16>((size_t)(rows_alloc(P) * sh->I));
    return align_up(c.off, 256);
}

size_t permute_ws_bytes(int32_t T, int32_t E, int32_t k) {
    const int64_t P = (int64_t)T * k;
    return align_up(sizeof(WsHeader), 256) + align_up(permute_scratch_ints(P, E) * 4, 256);
}

moe_status check_ws(void* ws, size_t have, size_t need) {
    if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    if (have < need)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
    return MOE_OK;
}

#define CHECK_PTR(p)                                                              \
    do {                                                                          \
        if (!(p)) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);             \
        if (!aligned((p), 16)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
    } while (0)

#define CUDA_TRY(expr, where)                         \
    do {                                              \
        cudaError_t e_ = (expr);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, where); \
    } while (0)

// Stage boundaries recorded by moe_forward_profiled (event i is recorded on
// the stream after stage i; index 0 before the first launch).
enum {
    kEvStart = 0, kEvRoute, kEvPermute, kEvGather, kEvGemmGateUp, kEvThinGateUp,
    kEvGemmDown, kEvThinDown, kEvCombine, kEvCount
};

cudaError_t mark(cudaEvent_t* ev, int i, cudaStream_t s) {
    return (ev && ev[i]) ? cudaEventRecord(ev[i], s) : cudaSuccess;
}

// NVTX range around the host-side launch of one stage (profilers attribute
// the stage's kernels to it; without a profiler attached it costs a check).
struct Nvtx {
    explicit Nvtx(const char* name) { nvtxRangePushA(name); }
    ~Nvtx() { nvtxRangePop(); }
    Nvtx(const Nvtx&) = delete;
    Nvtx& operator=(const Nvtx&) = delete;
};

// Expert stage shared by moe_expert_ffn and moe_forward.  `fat_bound` is an
// upper bound of any expert's count (no GEMM launch when it is below the
// threshold; it also sizes the streaming kernels' activation buffers).
moe_status run_experts(const moe_shape* sh, const DeviceInfo& dev, const __nv_bfloat16* x,
                       const int32_t* perm, const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                       const __nv_bfloat16* Wd, __nv_bfloat16* x_sorted,
                       __nv_bfloat16* h, __nv_bfloat16* y, const Plan& plan,
                       int64_t fat_bound, cudaStream_t s, cudaEvent_t* ev,
                       const SelfRoute* sr = nullptr, const SelfRoute* comb = nullptr,
                       bool* combined = nullptr) {
    const int64_t P = (int64_t)sh->T * sh->k;
    const ExpertKernels kn = expert_kernels(sh, fat_bound);
    const int64_t ra = rows_alloc(P);
    const int H = sh->H, I = sh->I, sms = dev.num_sms;
    // With fat experts the gather kernel copies only the rows of the first
    // pair tiles; the gate/up GEMM launch over those tiles copies the rest
    // with its idle warps, and a second launch runs the other pair tiles.
    if (kn.gather() && !sr) {   // a self-routed batch loads its x rows itself
        const Nvtx r("moe.gather");
        CUDA_TRY(launch_gather(x, perm, sh->k, H, plan, x_sorted, sms, s, kn.fat ? 1 : 0),
                 "gather");
    }
    CUDA_TRY(mark(ev, kEvGather, s), "cudaEventRecord");
    if (kn.fat) {
        const Nvtx r("moe.gemm_gate_up");
        CUDA_TRY(launch_gemm_gate_up(x_sorted, ra, Wg, Wu, H, I, plan, h, sms, s, 1, x, perm,
                                     sh->k),
                 "grouped GEMM gate/up");
        CUDA_TRY(launch_gemm_gate_up(x_sorted, ra, Wg, Wu, H, I, plan, h, sms, s, 2),
                 "grouped GEMM gate/up (second part)");
        CUDA_TRY(launch_gemm_solo_gate_up(x_sorted, ra, Wg, Wu, H, I, plan, h, sms, s),
                 "grouped GEMM gate/up (solo tiles)");
    }
    CUDA_TRY(mark(ev, kEvGemmGateUp, s), "cudaEventRecord");
    // A self-routed batch on the CUDA-core streaming kernel alone runs the
    // whole layer in one cooperative launch where that kernel has a build for
    // the layer's width (its stage events then bracket it as gate/up).
    const bool one_launch = sr && kn.units && !kn.mma && !kn.fat && thin_layer_fused(H, I);
    if (one_launch) {
        const Nvtx r("moe.thin_layer");
        CUDA_TRY(launch_thin_layer(x, sh->k, H, I, Wg, Wu, Wd, plan, fat_bound, h, y, sms, s,
                                   *sr),
                 "thin layer");
    } else {
        const Nvtx r("moe.thin_gate_up");
        if (kn.units)
            CUDA_TRY(launch_thin_gate_up(x, perm, sh->k, H, I, Wg, Wu, plan, fat_bound, h, sms, s,
                                         sr),
                     "thin gate/up");
        if (kn.mma)
            CUDA_TRY(launch_thin_mma_gate_up(x_sorted, ra, Wg, Wu, H, I, plan, h, sms, s, sr, x),
                     "thin gate/up (tensor cores)");
    }
    CUDA_TRY(mark(ev, kEvThinGateUp, s), "cudaEventRecord");
    if (kn.fat) {
        const Nvtx r("moe.gemm_down");
        CUDA_TRY(launch_gemm_down(h, ra, Wd, H, I, plan, y, sms, s), "grouped GEMM down");
        CUDA_TRY(launch_gemm_solo_down(h, ra, Wd, H, I, plan, y, sms, s),
                 "grouped GEMM down (solo tiles)");
    }
    CUDA_TRY(mark(ev, kEvGemmDown, s), "cudaEventRecord");
    {
        const Nvtx r("moe.thin_down");
        if (kn.units && !one_launch)
            CUDA_TRY(launch_thin_down(h, H, I, Wd, plan, fat_bound, y, sms, s, sr), "thin down");
        // A planned batch whose only expert kernel is the tensor-core one
        // combines in that kernel's down launch (comb: its route lists).
        const bool fuse = comb && !sr && kn.mma && !kn.fat && !kn.units;
        if (kn.mma)
            CUDA_TRY(launch_thin_mma_down(h, ra, Wd, H, I, plan, y, sms, s, fuse ? comb : sr),
                     "thin down (tensor cores)");
        if (combined) *combined = fuse;
    }
    CUDA_TRY(mark(ev, kEvThinDown, s), "cudaEventRecord");
    return MOE_OK;
}

}  // namespace

moe_status moe::mark_touched_experts(const moe_shape* shape, const float* logits, void* ws,
                                     size_t ws_bytes, uint8_t* flags, cudaStream_t s) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return MOE_OK;
    if (!logits || !flags) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    FwdBufs b;
    if ((st = check_ws(ws, ws_bytes, carve_fwd(shape, nullptr, &b))) != MOE_OK) return st;
    carve_fwd(shape, ws, &b);
    CUDA_TRY(launch_route(logits, shape->T, shape->E, shape->k, b.idx, b.gates, s), "route");
    CUDA_TRY(launch_mark_touched(b.idx, (int64_t)shape->T * shape->k, shape->E, flags, s),
             "mark touched experts");
    return MOE_OK;
}

extern "C" {

const char* moe_last_error(void) { return g_err; }

const char* moe_version(void) { return "libmoe 0.1 (sm_103a)"; }

moe_status moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                     int32_t* topk_idx, float* gates, moe_stream_t stream) {
    moe_status st = check_route_args(T, E, k);
    if (st != MOE_OK) return st;
    if (T == 0) return ok();
    if (!logits || !topk_idx || !gates) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    CUDA_TRY(launch_route(logits, T, E, k, topk_idx, gates, (cudaStream_t)stream), "route");
    return ok();
}

size_t moe_permute_workspace_size(int32_t T, int32_t E, int32_t k) {
    if (check_route_args(T, E, k) != MOE_OK) return 0;
    return permute_ws_bytes(T, E, k);
}

moe_status moe_permute(const int32_t* topk_idx, int32_t T, int32_t E, int32_t k,
                       int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    moe_status st = check_route_args(T, E, k);
    if (st != MOE_OK) return st;
    if (!counts || !offsets) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if (T > 0 && (!topk_idx || !perm || !inv_perm)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if ((st = check_ws(ws, ws_bytes, permute_ws_bytes(T, E, k))) != MOE_OK) return st;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    Carver c(ws);
    WsHeader* hdr = c.take<WsHeader>(1);
    int32_t* chunk = c.take<int32_t>(permute_scratch_ints((int64_t)T * k, E));
    const int64_t nch = ((int64_t)T * k + kPermChunk - 1) / kPermChunk;
    CUDA_TRY(launch_permute(topk_idx, T, E, k, counts, offsets, perm, inv_perm, chunk,
                            chunk + nch * E, hdr, nullptr, (cudaStream_t)stream), "permute");
    return ok();
}

size_t moe_expert_ffn_workspace_size(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    FfnBufs b;
    return carve_ffn(shape, nullptr, &b);
}

moe_status moe_expert_ffn(const moe_shape* shape, const moe_bf16* x, const int32_t* perm,
                          const int32_t* offsets, const int32_t* counts,
                          const moe_bf16* W_gate, const moe_bf16* W_up,
                          const moe_bf16* W_down, moe_bf16* y_sorted, void* ws,
                          size_t ws_bytes, moe_stream_t stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return ok();
    CHECK_PTR(x); CHECK_PTR(perm); CHECK_PTR(offsets); CHECK_PTR(counts);
    CHECK_PTR(W_gate); CHECK_PTR(W_up); CHECK_PTR(W_down); CHECK_PTR(y_sorted);
    FfnBufs b;
    if ((st = check_ws(ws, ws_bytes, carve_ffn(shape, nullptr, &b))) != MOE_OK) return st;
    carve_ffn(shape, ws, &b);
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const Plan plan = make_plan(shape, b.tiles, b.solo_tiles, b.units, b.mma_tiles, b.hdr);
    const PdlScope pdl((int64_t)shape->T * shape->k <= kPermChunk);
    CUDA_TRY(launch_plan(counts, offsets, shape->E, plan, s), "plan");
    st = run_experts(shape, dev, (const __nv_bfloat16*)x, perm, (const __nv_bfloat16*)W_gate,
                     (const __nv_bfloat16*)W_up, (const __nv_bfloat16*)W_down, b.x_sorted, b.h,
                     (__nv_bfloat16*)y_sorted, plan, (int64_t)shape->T * shape->k, s, nullptr);
    return st == MOE_OK ? ok() : st;
}

moe_status moe_combine(const moe_bf16* y_sorted, const int32_t* inv_perm, const float* gates,
                       int32_t T, int32_t k, int32_t H, moe_bf16* out, moe_stream_t stream) {
    if (T < 0 || k < 1 || k > kMaxK) return fail(MOE_ERR_INVALID_ARG, "bad T or k");
    if (H < 8 || H % 8) return fail(MOE_ERR_INVALID_ARG, "H = %d is not a positive multiple of 8", H);
    if (T == 0) return ok();
    CHECK_PTR(y_sorted); CHECK_PTR(out);
    if (!inv_perm || !gates) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    moe_status st;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    CUDA_TRY(launch_combine((const __nv_bfloat16*)y_sorted, inv_perm, gates, T, k, H,
                            (__nv_bfloat16*)out, dev.num_sms, (cudaStream_t)stream), "combine");
    return ok();
}

size_t moe_workspace_size(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    FwdBufs b;
    return carve_fwd(shape, nullptr, &b);
}

}  // extern "C"

static moe_status forward_impl(const moe_shape* shape, const float* logits, const moe_bf16* x,
                               const moe_bf16* W_gate, const moe_bf16* W_up,
                               const moe_bf16* W_down, moe_bf16* out, int32_t* topk_idx,
                               float* gates, void* ws, size_t ws_bytes, moe_stream_t stream,
                               cudaEvent_t* ev, const int32_t* wslot = nullptr,
                               int32_t n_wblocks = 0) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return ok();
    if (!logits) return fail(MOE_ERR_INVALID_ARG, "logits is NULL");
    CHECK_PTR(x); CHECK_PTR(W_gate); CHECK_PTR(W_up); CHECK_PTR(W_down); CHECK_PTR(out);
    FwdBufs b;
    if ((st = check_ws(ws, ws_bytes, carve_fwd(shape, nullptr, &b))) != MOE_OK) return st;
    carve_fwd(shape, ws, &b);
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const int T = shape->T, E = shape->E, k = shape->k;
    const PdlScope pdl((int64_t)T * k <= kPermChunk);
    int32_t* idx = topk_idx ? topk_idx : b.idx;
    float* g = gates ? gates : b.gates;
    const Nvtx range("moe_forward");
    CUDA_TRY(mark(ev, kEvStart, s), "cudaEventRecord");
    Plan plan = make_plan(shape, b.tiles, b.solo_tiles, b.units, b.mma_tiles, b.hdr);
    if (wslot) {
        plan.wslot = wslot;
        plan.n_wblocks = n_wblocks;
    }
    // Small batches route inside the streaming kernels and combine in the down
    // kernel (the route, permute and combine stages are then empty); the
    // others run the router, the route lists and the combine kernel.
    const bool self = self_mode(shape) != kPlanned;
    const SelfRoute sr{logits, T, E, k, idx, g, b.counts, b.offsets, b.perm, b.inv_perm,
                       b.units, (__nv_bfloat16*)out};
    if (!self) {
        const Nvtx r("moe.route");
        CUDA_TRY(launch_route(logits, T, E, k, idx, g, s), "route");
    }
    CUDA_TRY(mark(ev, kEvRoute, s), "cudaEventRecord");
    const int64_t P = (int64_t)T * k;
    const int64_t nch = (P + kPermChunk - 1) / kPermChunk;
    if (!self) {
        const Nvtx r("moe.permute");
        CUDA_TRY(launch_permute(idx, T, E, k, b.counts, b.offsets, b.perm, b.inv_perm, b.chunk,
                                b.chunk + nch * E, b.hdr, &plan, s), "permute");
    }
    CUDA_TRY(mark(ev, kEvPermute, s), "cudaEventRecord");
    // The router sends a token to k distinct experts, so no expert holds more
    // than T slots.  x_sorted is dead once the gate/up GEMM is done, so
    // y_sorted reuses its storage.
    const SelfRoute comb{nullptr, T, E, k, idx, g, b.counts, b.offsets, b.perm, b.inv_perm,
                         b.units, (__nv_bfloat16*)out};
    bool combined = false;
    st = run_experts(shape, dev, (const __nv_bfloat16*)x, b.perm, (const __nv_bfloat16*)W_gate,
                     (const __nv_bfloat16*)W_up, (const __nv_bfloat16*)W_down, b.xy, b.h, b.xy,
                     plan, T, s, ev, self ? &sr : nullptr, &comb, &combined);
    if (st != MOE_OK) return st;
    if (!self && !combined) {
        const Nvtx r("moe.combine");
        CUDA_TRY(launch_combine(b.xy, b.inv_perm, g, T, k, shape->H, (__nv_bfloat16*)out,
                                dev.num_sms, s), "combine");
    }
    CUDA_TRY(mark(ev, kEvCombine, s), "cudaEventRecord");
    return ok();
}

moe_status moe::forward_blocks(const moe_shape* shape, const float* logits, const moe_bf16* x,
                              const moe_bf16* W_gate, const moe_bf16* W_up,
                              const moe_bf16* W_down, const int32_t* wslot, int32_t n_wblocks,
                              moe_bf16* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!wslot || n_wblocks < 1) return fail(MOE_ERR_INVALID_ARG, "bad weight-block table");
    return forward_impl(shape, logits, x, W_gate, W_up, W_down, out, nullptr, nullptr, ws,
                        ws_bytes, stream, nullptr, wslot, n_wblocks);
}

extern "C" {

moe_status moe_forward(const moe_shape* shape, const float* logits, const moe_bf16* x,
                       const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                       moe_bf16* out, int32_t* topk_idx, float* gates, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(shape, logits, x, W_gate, W_up, W_down, out, topk_idx, gates, ws,
                        ws_bytes, stream, nullptr);
}

moe_status moe_forward_profiled(const moe_shape* shape, const float* logits,
                                const moe_bf16* x, const moe_bf16* W_gate,
                                const moe_bf16* W_up, const moe_bf16* W_down, moe_bf16* out,
                                int32_t* topk_idx, float* gates, void* ws, size_t ws_bytes,
                                moe_stream_t stream, void* const* stage_events,
                                int32_t n_events) {
    if (!stage_events || n_events < MOE_PROFILE_EVENTS)
        return fail(MOE_ERR_INVALID_ARG, "stage_events needs %d entries", MOE_PROFILE_EVENTS);
    cudaEvent_t ev[kEvCount];
    for (int i = 0; i < kEvCount; ++i) ev[i] = (cudaEvent_t)stage_events[i];
    return forward_impl(shape, logits, x, W_gate, W_up, W_down, out, topk_idx, gates, ws,
                        ws_bytes, stream, ev);
}

int32_t moe_forward_launches(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return -1;
    if (shape->T == 0) return 0;
    const SelfMode sm = self_mode(shape);
    if (sm == kSelfUnits && thin_layer_fused(shape->H, shape->I)) return 1;   // the whole layer
    if (sm != kPlanned) return 2;                    // gate/up, down (routing, combine inside)
    const int64_t P = (int64_t)shape->T * shape->k;
    int32_t n = 1;                                   // route
    n += (P <= kPermChunk) ? 1 : 3;                  // route lists (+ planner)
    const ExpertKernels kn = expert_kernels(shape, shape->T);
    if (kn.gather()) n += 1;
    if (kn.fat) n += 5;                              // grouped GEMMs (gate/up pairs in two
                                                     // parts, down pairs, solo tiles)
    if (kn.units) n += 2;                            // CUDA-core streaming
    if (kn.mma) n += 2;                              // tensor-core streaming
    if (kn.fat || kn.units || !kn.mma) n += 1;       // combine (else fused into the last)
    return n;
}

moe_status moe_debug_set_wait_limit(int64_t cycles) {
    if (cycles < 0) return fail(MOE_ERR_INVALID_ARG, "cycles = %lld < 0", (long long)cycles);
    t_wait_cycles = (long long)cycles;
    return ok();
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ws || ws_bytes < sizeof(WsHeader)) return fail(MOE_ERR_WORKSPACE, "workspace too small");
    CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(WsHeader), (cudaStream_t)stream), "cudaMemsetAsync");
    return ok();
}

moe_status moe_workspace_status(void* ws, moe_stream_t stream, int32_t clear) {
    if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    int32_t code = 0;
    cudaStream_t s = (cudaStream_t)stream;
    CUDA_TRY(cudaMemcpyAsync(&code, ws, sizeof code, cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync");
    CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (clear && code != 0) {
        CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(int32_t), s), "cudaMemsetAsync");
        CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    }
    if (code == MOE_ERR_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a bounded device wait ran out");
    if (code == MOE_ERR_BAD_INDEX) return fail(MOE_ERR_BAD_INDEX, "a routed index was outside [0, E)");
    if (code != 0) return fail((moe_status)code, "device status %d", code);
    return ok();
}

}  // extern "C"
