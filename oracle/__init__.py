"""Oracle for the routed mixture-of-experts FFN layer.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain CPU definition of
what the CUDA library computes; the test suite, the smoke check and the
benchmark's CPU-baseline leg are its only users.  The library never imports
it, and it imports nothing from the library.  The arithmetic lives in
``moe_oracle.c`` (single-threaded, fp64); this module compiles it with gcc and
marshals numpy arrays to it.  Pages followed: dsv41-flash-offload wiki
(overview: routed experts, busy experts as dense GEMMs; file map: route lists
with positive counts, split/combine on GPU).

bf16 tensors cross this boundary as numpy ``uint16`` arrays holding the raw
bit patterns; :func:`bf16_bits_to_f64` widens them exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C99, no FMA contraction, no
    fast-math, so fp64 results do not depend on the host CPU)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.oracle_route.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_route.restype = i32
            lib.oracle_permute.argtypes = [P, i64, i32, i32, P, P, P, P]
            lib.oracle_permute.restype = i32
            lib.oracle_expert_ffn.argtypes = [P, P, P, P, i32, i32, P, P]
            lib.oracle_expert_ffn.restype = None
            lib.oracle_moe_tokens.argtypes = [i64, P, P, i32, i32, i32, i32,
                                              P, P, P, P, P, P]
            lib.oracle_moe_tokens.restype = i32
            lib.oracle_combine.argtypes = [P, P, P, i64, i32, i32, P]
            lib.oracle_combine.restype = i32
            lib.oracle_array_to_bf16.argtypes = [P, i64, P]
            lib.oracle_array_to_bf16.restype = None
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(ValueError):
    pass


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even) in one step."""
    v = _c(values, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_array_to_bf16(_ptr(v), v.size, _ptr(out))
    return out


def route(logits: np.ndarray, k: int):
    """Top-k selection (larger logit first, ties to the lower index) and
    softmax-over-selection gates.  logits: float32 [T, E].
    Returns (idx int32 [T, k], gates float64 [T, k])."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    if _load().oracle_route(_ptr(lg), T, E, k, _ptr(idx), _ptr(gates)) != 0:
        raise OracleError("routing precondition violated")
    return idx, gates


def permute(idx: np.ndarray, E: int):
    """Stable counting sort of the T*k slots by expert.
    Returns (counts [E], offsets [E+1], perm [T*k], inv_perm [T*k]), int32."""
    ix = _c(idx, np.int32)
    T, k = ix.shape
    P = T * k
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(P, dtype=np.int32)
    inv_perm = np.empty(P, dtype=np.int32)
    if _load().oracle_permute(_ptr(ix), T, E, k, _ptr(counts), _ptr(offsets),
                              _ptr(perm), _ptr(inv_perm)) != 0:
        raise OracleError("routed index out of range")
    return counts, offsets, perm, inv_perm


def expert_ffn(x_bits: np.ndarray, Wg_bits: np.ndarray, Wu_bits: np.ndarray,
               Wd_bits: np.ndarray):
    """One SwiGLU expert on one token, fp64.  x: [H]; Wg, Wu: [I, H];
    Wd: [H, I] (bf16 bit patterns).  Returns (h [I], y [H]) as float64."""
    x = _c(x_bits, np.uint16)
    Wg = _c(Wg_bits, np.uint16)
    Wu = _c(Wu_bits, np.uint16)
    Wd = _c(Wd_bits, np.uint16)
    I, H = Wg.shape
    assert x.shape == (H,) and Wu.shape == (I, H) and Wd.shape == (H, I)
    h = np.empty(I, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    _load().oracle_expert_ffn(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), H, I,
                              _ptr(h), _ptr(y))
    return h, y


def moe_tokens(x_bits: np.ndarray, logits: np.ndarray, k: int, expert_weights):
    """Whole layer for n tokens: routing, the selected experts, combine.

    x_bits: uint16 [n, H]; logits: float32 [n, E]; expert_weights: callable
    e -> (Wg_e, Wu_e, Wd_e) uint16 arrays, or a sequence indexable by e.
    Only experts selected by these tokens are requested.
    Returns (out float64 [n, H], idx int32 [n, k], gates float64 [n, k]).
    """
    x = _c(x_bits, np.uint16)
    lg = _c(logits, np.float32)
    n, H = x.shape
    E = lg.shape[1]
    idx, _ = route(lg, k)
    needed = sorted(set(int(e) for e in idx.reshape(-1)))
    keep = []
    tabs = [(ctypes.c_void_p * E)() for _ in range(3)]
    I = None
    for e in needed:
        ws = expert_weights(e) if callable(expert_weights) else expert_weights[e]
        ws = [_c(w, np.uint16) for w in ws]
        I = ws[0].shape[0]
        keep.append(ws)
        for tab, w in zip(tabs, ws):
            tab[e] = w.ctypes.data
    out = np.empty((n, H), dtype=np.float64)
    oidx = np.empty((n, k), dtype=np.int32)
    ogates = np.empty((n, k), dtype=np.float64)
    tp = [ctypes.cast(tab, ctypes.c_void_p) for tab in tabs]
    rc = _load().oracle_moe_tokens(n, _ptr(x), _ptr(lg), E, k, H, I or 1,
                                   tp[0], tp[1], tp[2],
                                   _ptr(out), _ptr(oidx), _ptr(ogates))
    del keep
    if rc != 0:
        raise OracleError(f"oracle_moe_tokens failed ({rc})")
    return out, oidx, ogates


def combine(y_sorted: np.ndarray, inv_perm: np.ndarray, gates: np.ndarray):
    """out[t] = sum_j gates[t, j] * y_sorted[inv_perm[t*k + j]] in fp64.
    y_sorted: float [T*k, H]; inv_perm: int [T*k]; gates: float [T, k]."""
    y = _c(y_sorted, np.float64)
    ip = _c(inv_perm, np.int32).reshape(-1)
    g = _c(gates, np.float64)
    T, k = g.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    if _load().oracle_combine(_ptr(y), _ptr(ip), _ptr(g), T, k, H, _ptr(out)) != 0:
        raise OracleError("inv_perm out of range")
    return out
