"""Thin ctypes binding of libmoe (include/moe.h).

Argument marshalling only: every step of the layer runs in libmoe's CUDA
kernels.  Tensors are torch CUDA tensors; their data pointers and the current
torch stream are handed to the C entry points.  Missing outputs and
workspaces are allocated with torch (device memory is torch's job here).  If
libmoe.so is missing this module raises on import: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python routed_expert_ffn_02_gb300/_build.py`")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_BAD_INDEX"}

# Every function declared in include/moe.h.
EXPORTED = ("moe_route", "moe_permute_workspace_size", "moe_permute", "moe_permute_noalloc",
            "moe_expert_ffn_workspace_size", "moe_expert_ffn", "moe_combine",
            "moe_workspace_size", "moe_forward", "moe_forward_profiled",
            "moe_forward_launches", "moe_layer_weight_bytes", "moe_stager_create",
            "moe_stager_destroy", "moe_forward_offload", "moe_workspace_init",
            "moe_workspace_status", "moe_last_error", "moe_version",
            "moe_pipe_workspace_size", "moe_pipe_create", "moe_pipe_destroy",
            "moe_forward_host", "moe_cache_bytes", "moe_cache_create", "moe_cache_destroy",
            "moe_cache_stats", "moe_forward_cached", "moe_debug_set_wait_limit")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("fat_threshold", ctypes.c_int32),
                ("thin_mma_min", ctypes.c_int32)]


@dataclass(frozen=True)
class Shape:
    T: int
    E: int
    k: int
    H: int
    I: int
    fat_threshold: int = 32
    thin_mma_min: int = 0     # 0: library default; > fat_threshold - 1: CUDA cores only

    def c(self) -> MoeShape:
        return MoeShape(self.T, self.E, self.k, self.H, self.I, self.fat_threshold,
                        self.thin_mma_min)

    @property
    def P(self) -> int:
        return self.T * self.k


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.moe_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_P = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_SP = ctypes.POINTER(MoeShape)

_sig = {
    "moe_route": ([_P, _i32, _i32, _i32, _P, _P, _P], _i32),
    "moe_permute_workspace_size": ([_i32, _i32, _i32], _sz),
    "moe_permute": ([_P, _i32, _i32, _i32, _P, _P, _P, _P, _P, _sz, _P], _i32),
    "moe_permute_noalloc": ([_P, _i32, _i32, _i32, _P, _P, _P, _P, _P, _P], _i32),
    "moe_expert_ffn_workspace_size": ([_SP], _sz),
    "moe_expert_ffn": ([_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _sz, _P], _i32),
    "moe_combine": ([_P, _P, _P, _i32, _i32, _i32, _P, _P], _i32),
    "moe_workspace_size": ([_SP], _sz),
    "moe_forward": ([_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _sz, _P], _i32),
    "moe_forward_profiled": ([_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _sz, _P,
                              ctypes.POINTER(ctypes.c_void_p), _i32], _i32),
    "moe_forward_launches": ([_SP], _i32),
    "moe_layer_weight_bytes": ([_SP], _sz),
    "moe_stager_create": ([_P, _i32, _sz, ctypes.POINTER(_P)], _i32),
    "moe_stager_destroy": ([_P], _i32),
    "moe_forward_offload": ([_P, _SP, _i32, ctypes.POINTER(_P), _P, ctypes.POINTER(_P),
                             ctypes.POINTER(_P), _P, _sz, _P, _P], _i32),
    "moe_workspace_init": ([_P, _sz, _P], _i32),
    "moe_pipe_workspace_size": ([_SP], _sz),
    "moe_cache_bytes": ([_SP, _i32, _i32], _sz),
    "moe_cache_create": ([_SP, _i32, _i32, _P, _sz, ctypes.POINTER(_P)], _i32),
    "moe_cache_destroy": ([_P], _i32),
    "moe_cache_stats": ([_P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)], _i32),
    "moe_forward_cached": ([_P, _SP, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_P), _P,
                            ctypes.POINTER(_P), ctypes.POINTER(_P), _P, _sz, _P, _P], _i32),
    "moe_pipe_create": ([ctypes.POINTER(_P)], _i32),
    "moe_pipe_destroy": ([_P], _i32),
    "moe_forward_host": ([_P, _SP, _P, _P, _P, _P, _P, _P, _P, _sz, _P, _P, _P], _i32),
    "moe_workspace_status": ([_P, _P, _i32], _i32),
    "moe_debug_set_wait_limit": ([ctypes.c_int64], _i32),
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_version": ([], ctypes.c_char_p),
}
for _name, (_args, _ret) in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _ret


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(t: torch.Tensor):
    assert not t.is_cuda and t.is_contiguous(), "expected a contiguous host tensor"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def version() -> str:
    return _lib.moe_version().decode()


def debug_set_wait_limit(cycles: int) -> None:
    """Test hook (moe_debug_set_wait_limit): main-loop waits of this thread's
    later expert-kernel launches give up after `cycles` SM cycles (0: the
    default bound).  Only for tests of the timeout path."""
    _check(_lib.moe_debug_set_wait_limit(int(cycles)), "moe_debug_set_wait_limit")


class Workspace:
    """Device scratch for libmoe calls: a 256-byte-aligned torch buffer whose
    status word is cleared once at creation."""

    def __init__(self, nbytes: int, device=None, stream=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        self._buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self._buf.data_ptr()) % 256
        self.tensor = self._buf[off:off + nbytes]
        self.nbytes = nbytes
        _check(_lib.moe_workspace_init(self.ptr, nbytes, _stream(stream)), "moe_workspace_init")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())

    def status(self, clear: bool = True, stream=None) -> int:
        """Synchronises the stream and returns the device status code."""
        return _lib.moe_workspace_status(self.ptr, _stream(stream), int(clear))


def workspace_size(shape: Shape) -> int:
    n = _lib.moe_workspace_size(ctypes.byref(shape.c()))
    if n == 0:
        raise MoeError(1, "moe_workspace_size")
    return n


def permute_workspace_size(T: int, E: int, k: int) -> int:
    n = _lib.moe_permute_workspace_size(T, E, k)
    if n == 0:
        raise MoeError(1, "moe_permute_workspace_size")
    return n


def expert_ffn_workspace_size(shape: Shape) -> int:
    n = _lib.moe_expert_ffn_workspace_size(ctypes.byref(shape.c()))
    if n == 0:
        raise MoeError(1, "moe_expert_ffn_workspace_size")
    return n


def moe_route(logits: torch.Tensor, k: int, topk_idx=None, gates=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    topk_idx = topk_idx if topk_idx is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = gates if gates is not None else torch.empty((T, k), dtype=torch.float32, device=dev)
    _check(_lib.moe_route(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(gates), _stream(stream)),
           "moe_route")
    return topk_idx, gates


def moe_permute(topk_idx: torch.Tensor, E: int, ws: Workspace | None = None, out=None,
                stream=None):
    """Returns (counts [E], offsets [E+1], perm [T*k], inv_perm [T*k])."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    P = T * k
    if out is None:
        out = (torch.empty(E, dtype=torch.int32, device=dev),
               torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(max(P, 1), dtype=torch.int32, device=dev)[:P],
               torch.empty(max(P, 1), dtype=torch.int32, device=dev)[:P])
    counts, offsets, perm, inv_perm = out
    ws = ws or Workspace(permute_workspace_size(T, E, k), dev, stream)
    _check(_lib.moe_permute(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm),
                            _ptr(inv_perm), ws.ptr, ws.nbytes, _stream(stream)), "moe_permute")
    return counts, offsets, perm, inv_perm


def moe_permute_noalloc(topk_idx: torch.Tensor, E: int, out, device_status=None, stream=None):
    """moe_permute with the library's fixed scratch (no workspace, no device
    allocation inside the call).  `out` = (counts, offsets, perm, inv_perm)
    must be supplied by the caller; device_status (int32 [1]) is optional."""
    T, k = topk_idx.shape
    counts, offsets, perm, inv_perm = out
    _check(_lib.moe_permute_noalloc(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets),
                                    _ptr(perm), _ptr(inv_perm), _ptr(device_status),
                                    _stream(stream)), "moe_permute_noalloc")
    return out


def moe_expert_ffn(shape: Shape, x, perm, offsets, counts, W_gate, W_up, W_down,
                   y_sorted=None, ws: Workspace | None = None, stream=None):
    dev = x.device
    y_sorted = y_sorted if y_sorted is not None else torch.empty(
        (shape.P, shape.H), dtype=torch.bfloat16, device=dev)
    ws = ws or Workspace(expert_ffn_workspace_size(shape), dev, stream)
    _check(_lib.moe_expert_ffn(ctypes.byref(shape.c()), _ptr(x), _ptr(perm), _ptr(offsets),
                               _ptr(counts), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
                               _ptr(y_sorted), ws.ptr, ws.nbytes, _stream(stream)),
           "moe_expert_ffn")
    return y_sorted


def moe_combine(y_sorted, inv_perm, gates, T: int, k: int, H: int, out=None, stream=None):
    out = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16,
                                                  device=y_sorted.device)
    _check(_lib.moe_combine(_ptr(y_sorted), _ptr(inv_perm), _ptr(gates), T, k, H, _ptr(out),
                            _stream(stream)), "moe_combine")
    return out


def moe_forward(shape: Shape, logits, x, W_gate, W_up, W_down, out=None, topk_idx=None,
                gates=None, ws: Workspace | None = None, stream=None):
    dev = x.device
    out = out if out is not None else torch.empty((shape.T, shape.H), dtype=torch.bfloat16,
                                                  device=dev)
    ws = ws or Workspace(workspace_size(shape), dev, stream)
    _check(_lib.moe_forward(ctypes.byref(shape.c()), _ptr(logits), _ptr(x), _ptr(W_gate),
                            _ptr(W_up), _ptr(W_down), _ptr(out), _ptr(topk_idx), _ptr(gates),
                            ws.ptr, ws.nbytes, _stream(stream)), "moe_forward")
    return out


PROFILE_EVENTS = 9
PROFILE_STAGES = ("route", "permute", "gather", "gemm_gate_up", "thin_gate_up",
                  "gemm_down", "thin_down", "combine")


def moe_forward_profiled(shape: Shape, logits, x, W_gate, W_up, W_down, events, out=None,
                         topk_idx=None, gates=None, ws: Workspace | None = None,
                         stream=None):
    """moe_forward recording `events` (PROFILE_EVENTS torch.cuda.Event objects,
    created with enable_timing=True) at the stage boundaries."""
    assert len(events) == PROFILE_EVENTS
    dev = x.device
    out = out if out is not None else torch.empty((shape.T, shape.H), dtype=torch.bfloat16,
                                                  device=dev)
    ws = ws or Workspace(workspace_size(shape), dev, stream)
    for e in events:
        if e.cuda_event == 0:   # torch creates the CUDA event on first record
            e.record(stream if stream is not None else torch.cuda.current_stream())
    arr = (ctypes.c_void_p * PROFILE_EVENTS)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_lib.moe_forward_profiled(ctypes.byref(shape.c()), _ptr(logits), _ptr(x),
                                     _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(out),
                                     _ptr(topk_idx), _ptr(gates), ws.ptr, ws.nbytes,
                                     _stream(stream), arr, PROFILE_EVENTS),
           "moe_forward_profiled")
    return out


def forward_launches(shape: Shape) -> int:
    """Kernels one moe_forward call launches for this shape."""
    return _lib.moe_forward_launches(ctypes.byref(shape.c()))


def layer_weight_bytes(shape: Shape) -> int:
    """Bytes of one layer's expert set (W_gate | W_up | W_down, bf16)."""
    return _lib.moe_layer_weight_bytes(ctypes.byref(shape.c()))


def pack_layer_weights(W_gate, W_up, W_down, pin: bool = True) -> torch.Tensor:
    """One layer's experts as the contiguous W_gate | W_up | W_down block the
    stager copies (pinned host memory by default)."""
    parts = [W_gate.reshape(-1), W_up.reshape(-1), W_down.reshape(-1)]
    out = torch.empty(sum(p.numel() for p in parts), dtype=torch.bfloat16, pin_memory=pin)
    off = 0
    for p in parts:   # straight into the (pinned) block, no intermediate copy
        out[off:off + p.numel()].copy_(p)
        off += p.numel()
    return out


class Stager:
    """Ring of `n_slots` device staging slots (allocated here with torch, owned
    by this object) plus the library's stager over them."""

    def __init__(self, shape: Shape, n_slots: int, device=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.slot_bytes = (layer_weight_bytes(shape) + 255) // 256 * 256
        self.n_slots = n_slots
        self._mem = torch.empty(n_slots * self.slot_bytes + 256, dtype=torch.uint8, device=device)
        off = (-self._mem.data_ptr()) % 256
        self.slots = self._mem[off:off + n_slots * self.slot_bytes]
        self._h = ctypes.c_void_p()
        _check(_lib.moe_stager_create(ctypes.c_void_p(self.slots.data_ptr()), n_slots,
                                      self.slot_bytes, ctypes.byref(self._h)), "moe_stager_create")

    def close(self):
        if self._h:
            _lib.moe_stager_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, shape: Shape, logits, x, host_weights, outs=None, ws: Workspace | None = None,
                compute=None, copy=None):
        """Runs len(host_weights) layers; logits[l] and outs[l] are device
        tensors, host_weights[l] pinned host blocks from pack_layer_weights.
        Returns the outputs."""
        L = len(host_weights)
        dev = x.device
        outs = outs if outs is not None else [
            torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        ws = ws or Workspace(workspace_size(shape), dev, compute)
        compute = compute if compute is not None else torch.cuda.current_stream()
        copy = copy if copy is not None else torch.cuda.Stream(device=dev)
        PA = ctypes.c_void_p * max(L, 1)
        lg = PA(*[ctypes.c_void_p(t.data_ptr()) for t in logits])
        hw = PA(*[ctypes.c_void_p(t.data_ptr()) for t in host_weights])
        op = PA(*[ctypes.c_void_p(t.data_ptr()) for t in outs])
        _check(_lib.moe_forward_offload(self._h, ctypes.byref(shape.c()), L, lg, _ptr(x), hw, op,
                                        ws.ptr, ws.nbytes, ctypes.c_void_p(compute.cuda_stream),
                                        ctypes.c_void_p(copy.cuda_stream)), "moe_forward_offload")
        return outs


def pipe_workspace_size(shape: Shape) -> int:
    n = _lib.moe_pipe_workspace_size(ctypes.byref(shape.c()))
    if n == 0:
        raise MoeError(1, "moe_pipe_workspace_size")
    return n


class Pipe:
    """The layer on activations in host memory: each forward() copies its
    inputs in on an h2d stream, computes on `compute` and copies the output
    back on a d2h stream, overlapping with the neighbouring calls.  Owns the
    library pipe, its workspace (with two staging slots) and the two copy
    streams; all calls use one shape and one compute stream."""

    def __init__(self, shape: Shape, device=None, compute=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.shape = shape
        self.compute = compute if compute is not None else torch.cuda.current_stream(device)
        self.h2d = torch.cuda.Stream(device=device)
        self.d2h = torch.cuda.Stream(device=device)
        self.ws = Workspace(pipe_workspace_size(shape), device, self.compute)
        self._h = ctypes.c_void_p()
        _check(_lib.moe_pipe_create(ctypes.byref(self._h)), "moe_pipe_create")

    def close(self):
        if self._h:
            _lib.moe_pipe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, logits_h, x_h, W_gate, W_up, W_down, out_h):
        """Enqueues one layer: logits_h [T, E] fp32, x_h [T, H] bf16 and
        out_h [T, H] bf16 are (pinned) host tensors; out_h is written when
        the d2h stream reaches it (see synchronize())."""
        _check(_lib.moe_forward_host(self._h, ctypes.byref(self.shape.c()), _host_ptr(logits_h),
                                     _host_ptr(x_h), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
                                     _host_ptr(out_h), self.ws.ptr, self.ws.nbytes,
                                     _stream(self.compute), _stream(self.h2d),
                                     _stream(self.d2h)), "moe_forward_host")
        return out_h

    def synchronize(self):
        self.d2h.synchronize()


class ExpertCache:
    """HBM expert cache (n_slots experts, least recently used evicted) over
    experts kept in pinned host memory; owns its device block (torch) and the
    library's cache."""

    def __init__(self, shape: Shape, n_slots: int, max_layers: int, device=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.shape = shape
        nbytes = _lib.moe_cache_bytes(ctypes.byref(shape.c()), n_slots, max_layers)
        if nbytes == 0:
            raise MoeError(1, "moe_cache_bytes")
        self._mem = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self._mem.data_ptr()) % 256
        self.mem = self._mem[off:off + nbytes]
        self._h = ctypes.c_void_p()
        _check(_lib.moe_cache_create(ctypes.byref(shape.c()), n_slots, max_layers,
                                     ctypes.c_void_p(self.mem.data_ptr()), nbytes,
                                     ctypes.byref(self._h)), "moe_cache_create")

    def close(self):
        if self._h:
            _lib.moe_cache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self):
        """(hits, misses) since creation."""
        h, m = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.moe_cache_stats(self._h, ctypes.byref(h), ctypes.byref(m)), "moe_cache_stats")
        return h.value, m.value

    def forward(self, layer_ids, logits, x, host_weights, outs=None, ws: Workspace | None = None,
                compute=None, copy=None):
        """Runs len(layer_ids) layers: logits[l], outs[l] device tensors,
        host_weights[l] pinned blocks from pack_layer_weights."""
        L = len(layer_ids)
        dev = x.device
        shape = self.shape
        outs = outs if outs is not None else [
            torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        ws = ws or Workspace(workspace_size(shape), dev, compute)
        compute = compute if compute is not None else torch.cuda.current_stream()
        copy = copy if copy is not None else torch.cuda.Stream(device=dev)
        PA = ctypes.c_void_p * max(L, 1)
        ids = (ctypes.c_int32 * max(L, 1))(*layer_ids)
        lg = PA(*[ctypes.c_void_p(t.data_ptr()) for t in logits])
        hw = PA(*[ctypes.c_void_p(t.data_ptr()) for t in host_weights])
        op = PA(*[ctypes.c_void_p(t.data_ptr()) for t in outs])
        _check(_lib.moe_forward_cached(self._h, ctypes.byref(shape.c()), L, ids, lg, _ptr(x), hw,
                                       op, ws.ptr, ws.nbytes,
                                       ctypes.c_void_p(compute.cuda_stream),
                                       ctypes.c_void_p(copy.cuda_stream)), "moe_forward_cached")
        return outs


class DecodeGraph:
    """moe_forward for one fixed shape (a decode batch) captured once in a
    CUDA graph, as a serving engine runs decode steps: write the step's
    inputs into the static buffers `logits` [T, E] fp32 and `x` [T, H] bf16
    (device), call replay(), read `out` [T, H].  The weights are captured by
    address and must stay allocated."""

    def __init__(self, shape: Shape, W_gate, W_up, W_down, device=None):
        device = device or W_gate.device
        self.shape = shape
        self.logits = torch.zeros((shape.T, shape.E), dtype=torch.float32, device=device)
        self.x = torch.zeros((shape.T, shape.H), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=device)
        self.topk_idx = torch.empty((shape.T, shape.k), dtype=torch.int32, device=device)
        self.gates = torch.empty((shape.T, shape.k), dtype=torch.float32, device=device)
        self._W = (W_gate, W_up, W_down)
        self.stream = torch.cuda.Stream(device=device)
        self.ws = Workspace(workspace_size(shape), device, self.stream)
        self.stream.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(self.stream):
            self._forward()                     # resolves lazy state before capture
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._forward()

    def _forward(self):
        moe_forward(self.shape, self.logits, self.x, *self._W, out=self.out,
                    topk_idx=self.topk_idx, gates=self.gates, ws=self.ws, stream=self.stream)

    def replay(self):
        """Runs the captured layer on the current stream's timeline."""
        self.graph.replay()
        return self.out


def raw_lib():
    """The loaded ctypes library (for callers that pass raw pointers)."""
    return _lib
