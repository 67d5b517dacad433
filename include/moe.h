/*
 * moe.h -- C ABI of libmoe, the routed mixture-of-experts FFN layer on
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (dsv41-flash-offload wiki, overview: "384 routed experts" per MoE
 * layer, busy experts run as dense GEMMs; file map: route lists with positive
 * counts, split/combine on the GPU) computes, for T tokens, E experts,
 * top-k routing, hidden size H and expert intermediate size I:
 *
 *   route    : per token, the k largest router logits (ties to the lower
 *              expert index; outputs in that order) and gates
 *              g_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k
 *              selected logits;
 *   permute  : per-expert counts, their exclusive prefix sum (offsets) and a
 *              stable counting sort of the T*k token slots (slot s = t*k + j)
 *              by expert; within an expert, slots ascend;
 *   expert   : per slot routed to expert e, SwiGLU
 *              y = W_down[e] . (silu(W_gate[e] . x) * (W_up[e] . x));
 *              experts holding >= fat_threshold slots (default 32, the
 *              "fat threshold" of the model page's launch flags) run on the
 *              tensor-core grouped GEMM, the rest on the weight-streaming path;
 *   combine  : out_t = sum_j g_j * y_{t,j}, fp32 in fixed j order, rounded to
 *              bf16.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer.  Nothing here allocates device memory; scratch lives in
 *     the caller's workspace ("ws").  Buffers must be 16-byte aligned, the
 *     workspace 256-byte aligned.
 *   - bf16 tensors are passed as moe_bf16 (the raw 16-bit pattern).
 *   - Layouts are row-major:  logits fp32 [T, E]; x bf16 [T, H];
 *     W_gate, W_up bf16 [E, I, H]; W_down bf16 [E, H, I] (the [out, in]
 *     convention, contiguous along the reduction dimension); topk_idx int32
 *     [T, k]; gates fp32 [T, k]; counts int32 [E]; offsets int32 [E + 1];
 *     perm, inv_perm int32 [T*k]; y_sorted bf16 [T*k, H]; out bf16 [T, H].
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value covers argument validation and the
 *     kernel launches; it is MOE_OK or an error code, and moe_last_error()
 *     gives a message for the calling thread.  Faults inside kernels surface
 *     from later CUDA calls.  Kernels never trap: a condition found on the
 *     device (a routed index outside [0, E), a bounded wait that ran out)
 *     is recorded in the workspace's status word, read with
 *     moe_workspace_status().
 *   - Limits: 1 <= k <= min(E, 8); 1 <= E <= 1024; T >= 0 with T*k < 2^31;
 *     H and I positive multiples of 256, at most 16384 (MOE_ERR_UNSUPPORTED
 *     above); 0 <= fat_threshold <= 33 (experts
 *     with fewer slots than the threshold take the weight-streaming path,
 *     which holds at most 32 slots per expert).
 *   - Preconditions not checked: logits hold no NaN and no +inf, and each
 *     token's largest logit is finite; buffers do not overlap unless stated.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;            /* bf16 bit pattern */
typedef struct CUstream_st* moe_stream_t;  /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* no sm_103a device, or outside the limits */
    MOE_ERR_WORKSPACE = 3,     /* ws too small or misaligned */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    MOE_ERR_TIMEOUT = 5,       /* device status: a bounded wait ran out */
    MOE_ERR_BAD_INDEX = 6      /* device status: routed index outside [0, E) */
} moe_status;

typedef struct {
    int32_t T;              /* tokens */
    int32_t E;              /* routed experts */
    int32_t k;              /* experts per token */
    int32_t H;              /* hidden size */
    int32_t I;              /* expert intermediate size */
    int32_t fat_threshold;  /* slots at which an expert takes the GEMM; 32 */
    int32_t thin_mma_min;   /* slots at which a thin expert streams its weights
                               through the tensor cores instead of CUDA-core
                               FMAs, 0..33.  0 = by shape: 1 when
                               min(E, T*k) * I/128 >= 384 (enough 128-row work
                               items to fill the GPU), else 33.  Values above
                               fat_threshold - 1 keep every thin expert on
                               CUDA cores. */
} moe_shape;

/* ---- routing -------------------------------------------------------- */

/* Top-k router (dsv41-flash-offload wiki, overview: each token is routed to
 * k of the layer's experts).  Selection compares the raw fp32 logits with
 * (value descending, index ascending); gates are the softmax over the k
 * selected logits, computed in fp32.
 *   logits   [T, E] fp32, read only.
 *   topk_idx [T, k] int32, written; gates [T, k] fp32, written.
 * Errors: MOE_ERR_INVALID_ARG for bad sizes or null pointers (T == 0 is a
 * no-op). */
moe_status moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                     int32_t* topk_idx, float* gates, moe_stream_t stream);

/* ---- route lists ----------------------------------------------------- */

/* Bytes of workspace moe_permute needs for these sizes. */
size_t moe_permute_workspace_size(int32_t T, int32_t E, int32_t k);

/* Per-expert route lists (dsv41-flash-offload wiki, file map: route lists
 * with positive counts): counts[e] = #slots routed to e; offsets = exclusive
 * prefix sum with offsets[E] = T*k; perm[p] = slot at sorted position p
 * (expert-major, slots ascending within an expert); inv_perm[s] = position of
 * slot s.  Bit-exact: the result is unique.
 *   topk_idx [T, k] int32, read only; counts, offsets, perm, inv_perm
 *   written.  ws: scratch of moe_permute_workspace_size() bytes, whose status
 *   word must have been cleared once with moe_workspace_init().
 * A routed index outside [0, E) is skipped and sets MOE_ERR_BAD_INDEX in the
 * workspace status; the outputs are then unspecified. */
moe_status moe_permute(const int32_t* topk_idx, int32_t T, int32_t E, int32_t k,
                       int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory: a serving process that has already handed all of HBM to weights
 * and caches and has no pool left to carve a workspace from, or host code
 * that must keep cudaMalloc (which may synchronise the device) off its hot
 * path.  The pages describe nothing like it; it exists for such embedders.
 * Same arguments, results and bit-exactness as moe_permute, minus ws.
 * Scratch lives in a fixed array inside the library (about 1 MiB, held by
 * every GPU that loads libmoe until the process exits), so:
 *   - T*k may not exceed 262144 (MOE_ERR_UNSUPPORTED otherwise);
 *   - nothing is allocated: no cudaMalloc/cudaFree, no allocating library
 *     call; the first call on each device looks the array's device address
 *     up (cudaGetSymbolAddress, that device current) -- make that first call
 *     before any stream capture.  After a device reset (cudaDeviceReset) the
 *     next call on that device finds a new context and looks it up again, so
 *     make that call before any capture too;
 *   - device ordinals 0..63 only (MOE_ERR_UNSUPPORTED beyond);
 *   - all calls share the array and it keeps the last call's contents; each
 *     call clears the status it needs.  Calls that overlap on the GPU (e.g.
 *     on unordered streams) race and give wrong results.
 * device_status (device int32, may be NULL) receives this call's device
 * status: MOE_OK or MOE_ERR_BAD_INDEX. */
moe_status moe_permute_noalloc(const int32_t* topk_idx, int32_t T, int32_t E, int32_t k,
                               int32_t* counts, int32_t* offsets, int32_t* perm,
                               int32_t* inv_perm, int32_t* device_status,
                               moe_stream_t stream);

/* ---- experts ----------------------------------------------------------- */

/* Bytes of workspace moe_expert_ffn needs for this shape. */
size_t moe_expert_ffn_workspace_size(const moe_shape* shape);

/* Expert SwiGLU FFN over the sorted slots (dsv41-flash-offload wiki,
 * overview: busy experts run as dense GEMMs; model page launch flags: fat
 * threshold 32).  For sorted position p with slot s = perm[p], token
 * t = s / k and expert e (offsets[e] <= p < offsets[e+1]):
 *   y_sorted[p] = bf16( W_down[e] . bf16( silu(W_gate[e] . x[t]) * (W_up[e] . x[t]) ) )
 * with fp32 accumulation; the intermediate is rounded to bf16 once.
 * Experts with counts[e] >= fat_threshold run on the tcgen05 grouped GEMM,
 * experts with 0 < counts[e] < fat_threshold on the weight-streaming path.
 *   x [T, H], W_gate/W_up [E, I, H], W_down [E, H, I] bf16, read only;
 *   perm, offsets, counts as moe_permute wrote them; y_sorted [T*k, H] bf16
 *   written.  ws: moe_expert_ffn_workspace_size() bytes, initialised once
 *   with moe_workspace_init(). */
moe_status moe_expert_ffn(const moe_shape* shape, const moe_bf16* x,
                          const int32_t* perm, const int32_t* offsets,
                          const int32_t* counts, const moe_bf16* W_gate,
                          const moe_bf16* W_up, const moe_bf16* W_down,
                          moe_bf16* y_sorted, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* ---- combine --------------------------------------------------------- */

/* Gate-weighted un-permute (dsv41-flash-offload wiki, file map:
 * split/combine on the GPU):
 *   out[t] = bf16( sum_{j=0}^{k-1} gates[t, j] * y_sorted[inv_perm[t*k + j]] )
 * accumulated in fp32 in ascending j, no atomics: run-to-run identical.
 *   y_sorted [T*k, H] bf16, inv_perm [T*k], gates [T, k] read only;
 *   out [T, H] bf16 written (must not overlap y_sorted). */
moe_status moe_combine(const moe_bf16* y_sorted, const int32_t* inv_perm,
                       const float* gates, int32_t T, int32_t k, int32_t H,
                       moe_bf16* out, moe_stream_t stream);

/* ---- whole layer ----------------------------------------------------- */

/* Bytes of workspace moe_forward needs for this shape. */
size_t moe_workspace_size(const moe_shape* shape);

/* route -> permute -> expert -> combine on one stream, no host
 * synchronisation.  logits [T, E] fp32, x [T, H] bf16, weights as above;
 * out [T, H] bf16 written.  topk_idx [T, k] / gates [T, k] may be NULL; when
 * given they receive the routing.  ws: moe_workspace_size() bytes,
 * initialised once with moe_workspace_init().  Batches of at most 32 token
 * slots whose experts all stream on one weight-streaming kernel (decode) run
 * as two kernels that route and combine inside themselves, or, on the
 * CUDA-core kernel at (H, I) = (4096, 2048), (2048, 1024) and (512, 256), as
 * one cooperative kernel (one CTA per SM) whose CTAs also wait, bounded, for
 * one another after the gate/up phase and before the combine (the
 * tensor-core kernel's down launch is cooperative too and waits likewise
 * before its combine); the results, topk_idx and gates
 * included, are bit-identical to the separate stages.  Calls that share a
 * workspace must be ordered on one stream (or otherwise serialised). */
moe_status moe_forward(const moe_shape* shape, const float* logits,
                       const moe_bf16* x, const moe_bf16* W_gate,
                       const moe_bf16* W_up, const moe_bf16* W_down,
                       moe_bf16* out, int32_t* topk_idx, float* gates,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Number of stage events moe_forward_profiled records. */
#define MOE_PROFILE_EVENTS 9

/* moe_forward, recording caller-created CUDA events (cudaEvent_t, passed as
 * void*) on `stream` at the stage boundaries, so a caller can time each
 * kernel on the stream it runs on:
 *   [0] before routing       [1] after routing        [2] after route lists
 *   [3] after the GEMM row gather                     [4] after the gate/up GEMM
 *   [5] after the thin gate/up                        [6] after the down GEMM
 *   [7] after the thin down  [8] after the combine
 * A stage with nothing to do still records its event (for the two-kernel
 * small batches, routing and route lists are inside the thin gate/up stage
 * and the combine inside the thin down stage; the one-kernel layer is all
 * inside the thin gate/up stage).  stage_events must
 * hold n_events >= MOE_PROFILE_EVENTS entries; a NULL entry is skipped.
 * Results are identical to moe_forward. */
moe_status moe_forward_profiled(const moe_shape* shape, const float* logits,
                                const moe_bf16* x, const moe_bf16* W_gate,
                                const moe_bf16* W_up, const moe_bf16* W_down,
                                moe_bf16* out, int32_t* topk_idx, float* gates,
                                void* ws, size_t ws_bytes, moe_stream_t stream,
                                void* const* stage_events, int32_t n_events);

/* Number of kernels one moe_forward call with this shape launches (the
 * launch sequence depends only on the shape; 1 or 2 for the small batches
 * above),
 * or -1 for an invalid shape. */
int32_t moe_forward_launches(const moe_shape* shape);

/* ---- expert offload: pinned host memory -> HBM staging slots ---------- */

/* Expert weights kept in pinned host memory and streamed into a ring of
 * device staging slots on a side copy stream, overlapped with compute, the
 * copies running ahead into the next layers (dsv41-flash-offload wiki,
 * overview: experts pinned in host RAM, copied into VRAM slots in batches on
 * the copy engine, 8 staging slots, cross-layer DMA prefetch).  The copies
 * here are one kernel per layer that reads host memory with SM loads: on a
 * GB300 with a Grace host it holds the host link at its full rate, where the
 * copy engine's one copy per run of experts does not.  One slot holds one
 * layer's whole expert set. */
typedef struct moe_stager moe_stager;

/* Bytes of one layer's expert set: W_gate | W_up | W_down, bf16, in that
 * order and in the layouts moe_forward takes (0 for an invalid shape). */
size_t moe_layer_weight_bytes(const moe_shape* shape);

/* Creates a stager over caller-owned device memory `slots` (n_slots slots of
 * slot_bytes each, 256-byte aligned, slot_bytes a multiple of 256).  The
 * stager allocates no device memory; it owns two CUDA events per slot and a
 * pinned host flag array (n_layers x E bytes, allocated by the first forward
 * that needs it).  The slots must outlive the stager and every forward
 * enqueued with it. */
moe_status moe_stager_create(void* slots, int32_t n_slots, size_t slot_bytes,
                             moe_stager** out);
moe_status moe_stager_destroy(moe_stager* stager);

/* Runs n_layers independent layers on the same activations x [T, H] (device)
 * with logits[l] [T, E] and out[l] [T, H] (device), expert weights in
 * host_weights[l] (pinned host memory from cudaHostAlloc or
 * cudaHostRegister, 16-byte aligned, moe_layer_weight_bytes bytes,
 * W_gate | W_up | W_down).  First every layer is routed on `compute` and the
 * experts it touches are marked in a pinned flag array owned by the stager;
 * the call synchronises `compute` once to read them (wiki file map: only
 * experts with positive counts are copied).  Then, for layer l, one copy
 * kernel on `copy` moves the touched experts' three matrices into the same
 * offsets of slot l mod n_slots, reading the host memory with SM loads over
 * the host link, once the compute that last used that slot has finished, and
 * moe_forward runs on `compute` once the copy has landed; untouched experts'
 * regions of the slot are neither copied nor read.  All copies are enqueued
 * up front, so they run up to n_slots layers ahead.  `copy` must differ from
 * `compute`; ws as for moe_forward.  Errors as moe_forward, plus
 * MOE_ERR_INVALID_ARG (nothing enqueued) if a host_weights[l] is not 16-byte
 * aligned pinned host memory and MOE_ERR_CUDA if the flag array cannot be
 * allocated. */
moe_status moe_forward_offload(moe_stager* stager, const moe_shape* shape, int32_t n_layers,
                               const float* const* logits, const moe_bf16* x,
                               const void* const* host_weights, moe_bf16* const* out,
                               void* ws, size_t ws_bytes, moe_stream_t compute,
                               moe_stream_t copy);

/* ---- expert cache (models larger than HBM) ---------------------------- */

/* An HBM-resident expert cache in front of experts kept in host memory
 * (dsv41-flash-offload wiki, overview and file map: a VRAM expert cache over
 * experts in host RAM).  n_slots expert slots live in one caller-owned device
 * block; an expert of any layer stays resident across calls until it is the
 * least recently used one and its slot is needed. */
typedef struct moe_cache moe_cache;

/* Bytes of the device block for n_slots slots (each one expert's W_gate, W_up
 * and W_down) and per-layer expert -> slot tables for up to max_layers layers
 * per call (0 for invalid arguments). */
size_t moe_cache_bytes(const moe_shape* shape, int32_t n_slots, int32_t max_layers);

/* Creates a cache for experts of shape->E, H, I over `mem` (device,
 * moe_cache_bytes bytes, 256-byte aligned, caller-owned, outliving the cache
 * and every forward enqueued with it).  The cache owns 2 x max_layers CUDA
 * events and pinned host staging (max_layers x E x 5 bytes). */
moe_status moe_cache_create(const moe_shape* shape, int32_t n_slots, int32_t max_layers,
                            void* mem, size_t mem_bytes, moe_cache** out);
moe_status moe_cache_destroy(moe_cache* cache);

/* Expert lookups since creation that found the expert resident / copied it. */
moe_status moe_cache_stats(const moe_cache* cache, int64_t* hits, int64_t* misses);

/* Runs n_layers independent layers on x [T, H] (device) with logits[l]
 * [T, E] and out[l] [T, H] (device); layer l's experts are host_weights[l]
 * (16-byte aligned pinned host memory, W_gate | W_up | W_down as for
 * moe_forward_offload), cached under the key (layer_ids[l], expert),
 * layer_ids[l] >= 0.  First every layer is routed on `compute` and its
 * touched experts marked in pinned host flags; the call synchronises
 * `compute` once to read them.  Then, per layer: each touched expert not
 * resident is assigned the least recently used slot that layer l does not
 * need, and one copy kernel on `copy` moves the layer's misses in (SM loads
 * over the host link, as in moe_forward_offload) once the compute of the
 * last layers that read those slots has finished; the layer runs on
 * `compute` once its copies have landed.  n_layers <= max_layers; every
 * layer must touch at most n_slots experts (else MOE_ERR_INVALID_ARG, with
 * the earlier layers already enqueued).  `copy` must differ from `compute`;
 * ws as for moe_forward.  Errors as moe_forward, plus MOE_ERR_INVALID_ARG
 * (nothing enqueued) for host weights that are not 16-byte aligned pinned
 * host memory. */
moe_status moe_forward_cached(moe_cache* cache, const moe_shape* shape, int32_t n_layers,
                              const int32_t* layer_ids, const float* const* logits,
                              const moe_bf16* x, const void* const* host_weights,
                              moe_bf16* const* out, void* ws, size_t ws_bytes,
                              moe_stream_t compute, moe_stream_t copy);

/* ---- activations in host memory --------------------------------------- */

/* The layer on host-resident activations, as a serving process feeds it:
 * every call copies its logits and x in from host memory, runs moe_forward
 * and copies out back, and successive calls on one pipe overlap (call i's
 * inputs arrive and call i-2's output leaves while call i-1 computes).  Not
 * on the pages: their layer's activations already live on the GPU. */
typedef struct moe_pipe moe_pipe;

/* Bytes of device workspace moe_forward_host needs: moe_workspace_size()
 * plus two staging slots of x [T, H] bf16, logits [T, E] fp32 and
 * out [T, H] bf16 (0 for an invalid shape). */
size_t moe_pipe_workspace_size(const moe_shape* shape);

/* A pipe owns six CUDA events and a call counter, no device memory. */
moe_status moe_pipe_create(moe_pipe** out);
moe_status moe_pipe_destroy(moe_pipe* pipe);

/* moe_forward with logits_h [T, E] fp32, x_h [T, H] bf16 and out_h [T, H]
 * bf16 in host memory (pinned, or the copies serialise with the host).
 * Call i stages through slot i mod 2 at the end of ws:
 *   h2d:     once call i-2's compute has read the slot's inputs, copy
 *            logits_h and x_h in;
 *   compute: once they have landed and call i-2's output has left the slot,
 *            moe_forward into the slot;
 *   d2h:     once that is done, copy the slot's out to out_h.
 * Asynchronous: out_h is complete when `d2h` passes that copy (synchronise
 * d2h).  The three streams must differ; every call on a pipe uses the same
 * shape, ws (moe_pipe_workspace_size bytes, moe_workspace_init'ed) and
 * streams; host buffers must stay valid until their copies are done.
 * Errors: as moe_forward, plus MOE_ERR_INVALID_ARG for a NULL pipe or host
 * buffer or equal streams. */
moe_status moe_forward_host(moe_pipe* pipe, const moe_shape* shape, const float* logits_h,
                            const moe_bf16* x_h, const moe_bf16* W_gate, const moe_bf16* W_up,
                            const moe_bf16* W_down, moe_bf16* out_h, void* ws,
                            size_t ws_bytes, moe_stream_t compute, moe_stream_t h2d,
                            moe_stream_t d2h);

/* ---- workspace status ---------------------------------------------- */

/* Clears the status word of a fresh workspace (asynchronous on stream). */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream`, then returns the workspace's device status:
 * MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_BAD_INDEX (MOE_ERR_CUDA if the copy
 * fails).  The status is sticky; clear != 0 resets it to MOE_OK. */
moe_status moe_workspace_status(void* ws, moe_stream_t stream, int32_t clear);

/* Test hook for the timeout path (the pages' fail-loud guards, engram
 * prestage page: a failure is reported, never hidden).  Every mbarrier wait
 * in the main loops of the expert kernels (grouped GEMMs, both weight-
 * streaming kernels) gives up after a bounded number of SM cycles -- by
 * default about 2 s -- and the kernel then records MOE_ERR_TIMEOUT in the
 * workspace status, stops issuing work, waits with that default bound for
 * every copy and MMA it has issued, frees its tensor memory and returns.
 * This call sets the main-loop bound of the calling thread's later launches
 * to `cycles` (> 0), or restores the default (0); the drain waits keep the
 * default.  With a short bound the kernels give up on waits that would have
 * completed: the outputs of those launches are unspecified and the status
 * reads MOE_ERR_TIMEOUT.  MOE_ERR_INVALID_ARG for cycles < 0.  Nothing else
 * changes; it is meant for tests of the timeout path only. */
moe_status moe_debug_set_wait_limit(int64_t cycles);

/* Message for the last error returned to the calling thread ("" if none). */
const char* moe_last_error(void);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
