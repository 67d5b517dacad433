"""GPU parity: router and route lists against the oracle, bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import GATE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


def _route_check(moe, logits_cpu, k):
    T, E = logits_cpu.shape
    idx, gates = moe.moe_route(logits_cpu.cuda(), k)
    torch.cuda.synchronize()
    ridx, rgates = oracle.route(logits_cpu.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(gates.cpu().numpy(), rgates, rtol=0, atol=GATE_ATOL)
    return idx


ROUTE_CASES = [  # (T, E, k, zipf)
    (64, 16, 2, None), (1, 384, 8, 1.1), (4, 384, 8, 1.1), (24, 384, 8, 1.1),
    (16384, 384, 8, 1.1), (100, 1, 1, None), (77, 3, 3, None), (50, 33, 5, None),
    (300, 1024, 8, 1.1), (40, 100, 7, None), (513, 32, 8, None), (9, 64, 1, None),
    # batches of prefill size at every k, E a multiple of 4 or not
    (4096, 384, 8, 1.1), (5000, 1024, 8, 1.1), (4099, 100, 3, None), (4161, 4, 4, None),
    (6000, 132, 1, None), (4500, 64, 2, 1.1), (4100, 256, 5, None), (4127, 20, 6, None),
    (4096, 512, 7, 1.1), (4096, 33, 5, None), (5000, 7, 7, None),
]


@pytest.mark.parametrize("T,E,k,zipf", ROUTE_CASES)
def test_route_bitexact(moe, T, E, k, zipf):
    _route_check(moe, synth.make_logits(T, E, seed=11, zipf_s=zipf), k)


def test_route_ties_and_special_values(moe):
    lg = synth.tied_logits(500, 64, seed=1, levels=3)
    _route_check(moe, lg, 8)
    lg = synth.tied_logits(300, 40, seed=2, levels=2)
    lg[:, 5::3] = -float("inf")
    _route_check(moe, lg, 8)
    # -0.0 and +0.0 are the same logit: the lower index wins
    lg = torch.tensor([[-0.0, 0.0, -1.0, 0.0], [0.0, -0.0, -0.0, -2.0]], dtype=torch.float32)
    _route_check(moe, lg, 2)
    # all experts selected
    _route_check(moe, synth.make_logits(33, 8, seed=3), 8)


def test_route_ties_and_special_values_large_batch(moe):
    """The same cases in batches of prefill size."""
    _route_check(moe, synth.tied_logits(5000, 64, seed=4, levels=3), 8)
    lg = synth.tied_logits(4200, 40, seed=5, levels=2)
    lg[:, 5::3] = -float("inf")
    _route_check(moe, lg, 8)
    lg = torch.tensor([[-0.0, 0.0, -1.0, 0.0], [0.0, -0.0, -0.0, -2.0]], dtype=torch.float32)
    _route_check(moe, lg.repeat(2100, 1), 2)
    _route_check(moe, synth.make_logits(4100, 8, seed=6), 8)


def test_route_independent_of_placement_and_batch(moe):
    """A token's routing does not depend on where the logits start in
    memory (4 bytes past a 16-byte boundary here) nor on the batch it is
    routed in: bit-identical indices and gates."""
    T, E, k = 4500, 384, 8
    lg = synth.make_logits(T, E, seed=12, zipf_s=1.1)
    buf = torch.empty(T * E + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(lg.reshape(-1).cuda())
    skew = buf[1:].view(T, E)                   # 4 bytes past a 16-byte boundary
    idx_a, g_a = moe.moe_route(lg.cuda(), k)
    idx_b, g_b = moe.moe_route(skew, k)
    idx_c, g_c = moe.moe_route(lg[:40].cuda(), k)
    torch.cuda.synchronize()
    assert torch.equal(idx_a, idx_b) and torch.equal(g_a, g_b)
    assert torch.equal(idx_a[:40], idx_c) and torch.equal(g_a[:40], g_c)


def _permute_check(moe, idx_cpu, E):
    T, k = idx_cpu.shape
    counts, offsets, perm, inv = moe.moe_permute(idx_cpu.cuda(), E)
    torch.cuda.synchronize()
    rc, ro, rp, ri = oracle.permute(idx_cpu.numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)


PERMUTE_CASES = [  # (T, E, k, zipf): small single-block and multi-chunk paths
    (64, 16, 2, None), (1, 384, 8, 1.1), (4, 384, 8, 1.1), (256, 384, 8, 1.1),
    (257, 384, 8, 1.1), (1000, 384, 3, 1.1), (16384, 384, 8, 1.1), (5000, 1024, 8, 1.1),
    (3000, 7, 2, None), (2048, 1, 1, None), (2049, 1, 1, None),
]


@pytest.mark.parametrize("T,E,k,zipf", PERMUTE_CASES)
def test_permute_bitexact(moe, T, E, k, zipf):
    ridx, _ = oracle.route(synth.make_logits(T, E, seed=5, zipf_s=zipf).numpy(), k)
    _permute_check(moe, torch.from_numpy(ridx), E)


def test_permute_all_tokens_one_expert(moe):
    for T in (100, 3000):
        idx = torch.zeros((T, 2), dtype=torch.int32)
        idx[:, 1] = 3
        _permute_check(moe, idx, 8)


def test_permute_empty(moe):
    counts, offsets, perm, inv = moe.moe_permute(torch.empty((0, 4), dtype=torch.int32,
                                                             device="cuda"), 16)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and offsets[-1].item() == 0


@pytest.mark.parametrize("T", [10, 5000])
def test_permute_bad_index_status(moe, T):
    E, k = 16, 2
    idx = torch.randint(0, E, (T, k), dtype=torch.int32)
    idx[T // 2, 1] = E  # out of range
    ws = moe.Workspace(moe.permute_workspace_size(T, E, k))
    moe.moe_permute(idx.cuda(), E, ws=ws)
    assert ws.status(clear=True) == 6  # MOE_ERR_BAD_INDEX
    assert ws.status() == 0
