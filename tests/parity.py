"""Helpers shared by the GPU parity tests: tolerances, comparison against the
oracle, and oracle views of device-resident weights."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Output tolerance for bf16 results against the fp64 oracle: relative RMS
# <= 5e-3 and max-abs <= 2e-2 (the pages report a relative RMS of 0.0037
# between two expert tiers computing the same experts).
REL_RMS_TOL = 5e-3
MAX_ABS_TOL = 2e-2
# fp32 gates against the fp64 oracle: a handful of fp32 roundings of values
# in [0, 1].
GATE_ATOL = 2e-6


def errors(got: torch.Tensor | np.ndarray, ref: np.ndarray):
    if isinstance(got, torch.Tensor):
        got = got.float().cpu().numpy()
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    denom = np.sqrt(np.mean(ref ** 2)) if ref.size else 1.0
    rel_rms = float(np.sqrt(np.mean(diff ** 2)) / denom) if ref.size else 0.0
    max_abs = float(np.abs(diff).max()) if ref.size else 0.0
    return rel_rms, max_abs


def assert_close(got, ref, what=""):
    rel_rms, max_abs = errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got.float().cpu() if isinstance(got, torch.Tensor) else got)))
    assert rel_rms <= REL_RMS_TOL and max_abs <= MAX_ABS_TOL, \
        f"{what}: rel_rms={rel_rms:.3e} max_abs={max_abs:.3e}"
    return rel_rms, max_abs


class DeviceExperts:
    """e -> (Wg_e, Wu_e, Wd_e) bf16 bit patterns copied from device tensors,
    cached (the oracle reads exactly the bytes the GPU used)."""

    def __init__(self, Wg, Wu, Wd):
        self.W = (Wg, Wu, Wd)
        self.cache = {}

    def __call__(self, e: int):
        if e not in self.cache:
            self.cache[e] = tuple(synth.bf16_bits(w[e]) for w in self.W)
        return self.cache[e]


def oracle_rows(x_bits, logits_np, k, experts, tokens):
    """Oracle outputs (fp64) for the listed token ids."""
    tokens = np.asarray(tokens, dtype=np.int64)
    out, idx, gates = oracle.moe_tokens(x_bits[tokens], logits_np[tokens], k, experts)
    return out, idx, gates
