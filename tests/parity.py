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


def sample_tokens(idx_np, counts_np, thr, rng, n_random=24, hot_tiles=32):
    """Token ids for an oracle check of a large layer: random tokens, tokens
    of thin experts, of the smallest and the hottest fat expert, and of
    experts holding exactly 31/32/33 slots (the fat-threshold boundary).
    The hottest expert also gets one token in each of up to `hot_tiles`
    evenly spaced 256-row pair tiles of its sorted rows, at a different row
    of each tile, so a tile- or row-indexing fault anywhere in the grouped
    GEMM shows."""
    T = idx_np.shape[0]
    picks = set(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    thin = np.where((counts_np > 0) & (counts_np < thr))[0]
    fat = np.where(counts_np >= thr)[0]
    thin_tokens = np.where(np.isin(idx_np, thin).any(1))[0]
    picks.update(rng.choice(thin_tokens, size=min(8, len(thin_tokens)), replace=False).tolist())
    if len(fat):
        smallest = fat[np.argmin(counts_np[fat])]
        hottest = fat[np.argmax(counts_np[fat])]
        for e in (smallest, hottest):
            toks = np.where((idx_np == e).any(1))[0]
            picks.update(toks[:3].tolist())
    for c in (31, 32, 33):
        for e in np.where(counts_np == c)[0][:1]:
            picks.update(np.where((idx_np == e).any(1))[0][:2].tolist())
    if len(fat) and hot_tiles:
        hottest = fat[np.argmax(counts_np[fat])]
        # the expert's slots in sorted order (ascending slot id), 256 per tile
        slots = np.flatnonzero(idx_np.reshape(-1) == hottest)
        n_tiles = (len(slots) + 255) // 256
        for q in np.unique(np.linspace(0, n_tiles - 1, min(hot_tiles, n_tiles)).astype(int)):
            r = min(256 * q + (53 * q) % 256, len(slots) - 1)
            picks.add(int(slots[r]) // idx_np.shape[1])
    return np.array(sorted(picks))
