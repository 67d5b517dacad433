"""GPU parity on seeded random layer shapes.

Each case draws a layer (tokens, experts, top-k, widths, fat threshold,
thin-kernel split) from a fixed seed, so the list is the same on every run,
and checks moe_forward against the oracle on every output (routing
bit-exact) and bit-identical to the separate entry points (router, route
lists, expert FFN, combine).  The draws cross the path boundaries the
library picks by shape: self-routed batches (at most 32 slots), the planned
batches with and without fat experts, the one-launch widths, the gather
split under the gate/up GEMM and the fused combines.
"""
import numpy as np
import pytest
import torch

import synth
from parity import DeviceExperts, GATE_ATOL, assert_close, oracle_rows

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        E = int(rng.choice([1, 3, 8, 16, 40, 64]))
        k = int(rng.integers(1, min(8, E) + 1))
        T = int(rng.choice([1, 2, 3, 4, 5, 8, 13, 24, 33, 64, 130, 200]))
        H = int(rng.choice([256, 512, 768, 1024]))
        I = int(rng.choice([256, 512, 768]))
        thr = int(rng.choice([0, 1, 8, 32, 33]))
        mma = int(rng.choice([0, 1, 3, 33]))
        out.append((T, E, k, H, I, thr, mma))
    return out


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


@pytest.mark.parametrize("T,E,k,H,I,thr,mma", _cases())
def test_forward_random_shape(moe, T, E, k, H, I, thr, mma):
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    inp = synth.make_layer(s, seed=7000 + T * 31 + E, zipf_s=synth.ZIPF_S)
    d = {key: v.cuda() for key, v in inp.items()}
    shape = moe.Shape(T, E, k, H, I, fat_threshold=thr, thin_mma_min=mma)
    ws = moe.Workspace(moe.workspace_size(shape))
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = moe.moe_forward(shape, d["logits"], d["x"], d["Wg"], d["Wu"], d["Wd"],
                          topk_idx=idx, gates=gates, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref, ridx, rgates = oracle_rows(synth.bf16_bits(inp["x"]), inp["logits"].numpy(), k,
                                    DeviceExperts(d["Wg"], d["Wu"], d["Wd"]), np.arange(T))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(gates.cpu().numpy(), rgates, rtol=0, atol=GATE_ATOL)
    assert_close(out, ref, f"random shape {(T, E, k, H, I, thr, mma)}")
    idx2, gates2 = moe.moe_route(d["logits"], k)
    counts, offsets, perm, inv = moe.moe_permute(idx2, E)
    y = moe.moe_expert_ffn(shape, d["x"], perm, offsets, counts, d["Wg"], d["Wu"], d["Wd"])
    out2 = moe.moe_combine(y, inv, gates2, T, k, H)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(gates, gates2)
    assert torch.equal(out, out2)
