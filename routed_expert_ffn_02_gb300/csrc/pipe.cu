// pipe.cu -- the layer on activations held in host memory, with the
// host<->device copies of one call overlapping the compute of its
// neighbours.
//
// Each call i uses staging slot s = i mod 2 at the end of the workspace
// (x [T, H] bf16, logits [T, E] fp32, out [T, H] bf16):
//
//   h2d stream:     wait until the compute of call i-2 has consumed slot s's
//                   inputs; copy logits and x in; record in_ready[s]
//   compute stream: wait in_ready[s] and out_free[s] (call i-2's output has
//                   left slot s); moe_forward into slot s; record computed[s]
//   d2h stream:     wait computed[s]; copy slot s's output to the host;
//                   record out_free[s]
//
// so while call i computes, call i+1's inputs arrive and call i-1's output
// leaves.  The pipe owns only its events; the caller owns every buffer.
#include <new>

#include "moe_internal.cuh"

struct moe_pipe {
    int64_t calls;
    cudaEvent_t in_ready[2];
    cudaEvent_t computed[2];
    cudaEvent_t out_free[2];
};

namespace {

moe_status pipe_fail(moe_status st, const char* msg) {
    moe::set_last_error("%s", msg);
    return st;
}

struct Slot {
    moe_bf16* x;
    float* logits;
    moe_bf16* out;
};

size_t slot_bytes(const moe_shape* sh) {
    const size_t T = (size_t)sh->T;
    return moe::align_up(T * sh->H * 2, 256) + moe::align_up(T * sh->E * 4, 256) +
           moe::align_up(T * sh->H * 2, 256);
}

Slot slot_at(const moe_shape* sh, void* ws, size_t fwd_bytes, int s) {
    uint8_t* p = static_cast<uint8_t*>(ws) + fwd_bytes + (size_t)s * slot_bytes(sh);
    const size_t T = (size_t)sh->T;
    Slot sl;
    sl.x = reinterpret_cast<moe_bf16*>(p);
    p += moe::align_up(T * sh->H * 2, 256);
    sl.logits = reinterpret_cast<float*>(p);
    p += moe::align_up(T * sh->E * 4, 256);
    sl.out = reinterpret_cast<moe_bf16*>(p);
    return sl;
}

}  // namespace

extern "C" size_t moe_pipe_workspace_size(const moe_shape* shape) {
    const size_t fwd = moe_workspace_size(shape);
    if (fwd == 0) return 0;
    return moe::align_up(fwd, 256) + 2 * slot_bytes(shape);
}

extern "C" moe_status moe_pipe_create(moe_pipe** out) {
    if (!out) return pipe_fail(MOE_ERR_INVALID_ARG, "moe_pipe_create: out is NULL");
    *out = nullptr;
    moe_pipe* p = new (std::nothrow) moe_pipe();
    if (!p) return pipe_fail(MOE_ERR_CUDA, "moe_pipe_create: out of host memory");
    cudaEvent_t* all[6] = {&p->in_ready[0], &p->in_ready[1], &p->computed[0],
                           &p->computed[1], &p->out_free[0], &p->out_free[1]};
    for (int i = 0; i < 6; ++i) {
        if (cudaEventCreateWithFlags(all[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(*all[j]);
            delete p;
            return pipe_fail(MOE_ERR_CUDA, "moe_pipe_create: cudaEventCreate failed");
        }
    }
    *out = p;
    moe::set_last_error("");
    return MOE_OK;
}

extern "C" moe_status moe_pipe_destroy(moe_pipe* p) {
    if (!p) return MOE_OK;
    for (int s = 0; s < 2; ++s) {
        cudaEventDestroy(p->in_ready[s]);
        cudaEventDestroy(p->computed[s]);
        cudaEventDestroy(p->out_free[s]);
    }
    delete p;
    return MOE_OK;
}

extern "C" moe_status moe_forward_host(moe_pipe* p, const moe_shape* shape,
                                       const float* logits_h, const moe_bf16* x_h,
                                       const moe_bf16* W_gate, const moe_bf16* W_up,
                                       const moe_bf16* W_down, moe_bf16* out_h, void* ws,
                                       size_t ws_bytes, moe_stream_t compute, moe_stream_t h2d,
                                       moe_stream_t d2h) {
    if (!p) return pipe_fail(MOE_ERR_INVALID_ARG, "moe_forward_host: pipe is NULL");
    if (!shape) return pipe_fail(MOE_ERR_INVALID_ARG, "moe_forward_host: shape is NULL");
    if (compute == h2d || compute == d2h || h2d == d2h)
        return pipe_fail(MOE_ERR_INVALID_ARG,
                         "moe_forward_host: compute, h2d and d2h must be three different streams");
    const moe_status st = moe::check_shape_status(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return MOE_OK;
    const size_t need = moe_pipe_workspace_size(shape);
    if (!logits_h || !x_h || !out_h)
        return pipe_fail(MOE_ERR_INVALID_ARG, "moe_forward_host: NULL host buffer");
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256))
        return pipe_fail(MOE_ERR_WORKSPACE,
                         "moe_forward_host: workspace NULL, misaligned or below moe_pipe_workspace_size");
    const size_t fwd = moe::align_up(moe_workspace_size(shape), 256);
    const int s = (int)(p->calls & 1);
    const Slot sl = slot_at(shape, ws, fwd, s);
    const size_t T = (size_t)shape->T;
    cudaStream_t cs = (cudaStream_t)compute, hs = (cudaStream_t)h2d, ds = (cudaStream_t)d2h;
    cudaError_t e = cudaSuccess;
    const bool reuse = p->calls >= 2;   // slot s was used by call i-2
    if (reuse) e = cudaStreamWaitEvent(hs, p->computed[s], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(sl.logits, logits_h, T * shape->E * 4, cudaMemcpyHostToDevice, hs);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(sl.x, x_h, T * shape->H * 2, cudaMemcpyHostToDevice, hs);
    if (e == cudaSuccess) e = cudaEventRecord(p->in_ready[s], hs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p->in_ready[s], 0);
    if (e == cudaSuccess && reuse) e = cudaStreamWaitEvent(cs, p->out_free[s], 0);
    if (e != cudaSuccess) {
        moe::set_last_error("moe_forward_host: %s", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    const moe_status fs = moe_forward(shape, sl.logits, sl.x, W_gate, W_up, W_down, sl.out,
                                      nullptr, nullptr, ws, fwd, compute);
    if (fs != MOE_OK) return fs;
    e = cudaEventRecord(p->computed[s], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds, p->computed[s], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_h, sl.out, T * shape->H * 2, cudaMemcpyDeviceToHost, ds);
    if (e == cudaSuccess) e = cudaEventRecord(p->out_free[s], ds);
    if (e != cudaSuccess) {
        moe::set_last_error("moe_forward_host: %s", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    ++p->calls;
    moe::set_last_error("");
    return MOE_OK;
}
