"""GPU: the timeout path of the expert kernels (the engram-disk-prestage page's
fail-loud guards: a failure is reported, never hidden).

Every main-loop mbarrier wait of the grouped GEMMs and of both weight-
streaming kernels is bounded.  moe_debug_set_wait_limit shortens that bound
to one SM cycle, so the waits give up under normal load -- nothing is broken
or withheld.  Each kernel must then record MOE_ERR_TIMEOUT in the workspace
status, stop issuing work, wait (with the full bound) for the copies and MMAs
it has issued, free its tensor memory and return.  Checked: the status reads
MOE_ERR_TIMEOUT, and the next call on the same workspace with the default
bound gives exactly the outputs of a call before it (so no copy, MMA or
tensor-memory allocation was left behind)."""
import numpy as np
import pytest
import torch

import synth
from parity import DeviceExperts, assert_close, oracle_rows

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5
MMA_ALL, MMA_NONE = 1, 33


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


def _timed_out(moe, call):
    moe.debug_set_wait_limit(1)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        moe.debug_set_wait_limit(0)


# (T, E, k, H, I, fat_threshold, thin_mma_min): which expert kernels run
CASES = {
    "grouped GEMM (pairs and solo tiles)": (700, 6, 2, 512, 256, 1, 0),
    "tensor-core weight streaming": (64, 16, 2, 512, 256, 33, MMA_ALL),
    "CUDA-core weight streaming": (64, 16, 2, 512, 256, 33, MMA_NONE),
}


@pytest.mark.parametrize("case", list(CASES))
def test_expert_kernel_wait_expiry(moe, case):
    T, E, k, H, I, thr, mma = CASES[case]
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    d = {key: v.cuda() for key, v in synth.make_layer(s, seed=31, zipf_s=synth.ZIPF_S).items()}
    shape = moe.Shape(T, E, k, H, I, fat_threshold=thr, thin_mma_min=mma)
    idx, _ = moe.moe_route(d["logits"], k)
    counts, offsets, perm, _ = moe.moe_permute(idx, E)
    ws = moe.Workspace(moe.expert_ffn_workspace_size(shape))

    def ffn():
        return moe.moe_expert_ffn(shape, d["x"], perm, offsets, counts, d["Wg"], d["Wu"], d["Wd"],
                                  ws=ws)

    before = ffn()
    torch.cuda.synchronize()
    assert ws.status() == 0
    _timed_out(moe, ffn)
    assert ws.status(clear=True) == MOE_ERR_TIMEOUT, case
    for _ in range(2):
        after = ffn()
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert torch.equal(after, before), case


@pytest.mark.parametrize("H,I,mma_min,launches", [(1024, 2048, MMA_NONE, 2),
                                                  (1024, 2048, MMA_ALL, 2),
                                                  (2048, 1024, MMA_NONE, 1)])
def test_self_routed_decode_wait_expiry(moe, H, I, mma_min, launches):
    """A decode step routed inside the streaming kernels (two launches, the
    combine fused into the down kernel; or, at H=2048, I=1024 on CUDA cores,
    the whole layer in one cooperative launch whose down phase also waits,
    bounded, for every CTA's gate/up phase) that times out, then normal steps
    on the same workspace: status MOE_ERR_TIMEOUT once, then correct
    outputs.  The layers are large enough that every CTA's weight ring wraps
    several times, so its producer must wait for released slots."""
    B, E, k = 2, 64, 8
    Wg, Wu, Wd = synth.make_weights(E, H, I, seed=41, layer=0, device="cuda")
    shape = moe.Shape(B, E, k, H, I, fat_threshold=32, thin_mma_min=mma_min)
    assert moe.forward_launches(shape) == launches
    ws = moe.Workspace(moe.workspace_size(shape))
    x = synth.make_x(B, H, seed=41)
    lg = synth.make_logits(B, E, seed=41, zipf_s=synth.ZIPF_S)
    xd, lgd = x.cuda(), lg.cuda()
    before = moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _timed_out(moe, lambda: moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws))
    assert ws.status(clear=True) == MOE_ERR_TIMEOUT
    for _ in range(2):
        after = moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert torch.equal(after, before)
    ref, _, _ = oracle_rows(synth.bf16_bits(x), lg.numpy(), k, DeviceExperts(Wg, Wu, Wd),
                            np.arange(B))
    assert_close(after, ref, "decode after a timed-out step")


def test_planned_batch_fused_combine_wait_expiry(moe):
    """A planned batch of 8 tokens on the tensor-core streaming kernel alone
    (router, route lists, gather, gate/up, and a cooperative down launch that
    waits, bounded, for every CTA before combining) that times out, then
    normal steps on the same workspace: MOE_ERR_TIMEOUT once, then outputs
    identical to a step before it and close to the oracle."""
    B, E, k, H, I = 8, 64, 8, 512, 256
    Wg, Wu, Wd = synth.make_weights(E, H, I, seed=43, layer=0, device="cuda")
    shape = moe.Shape(B, E, k, H, I, fat_threshold=32, thin_mma_min=MMA_ALL)
    assert moe.forward_launches(shape) == 5
    ws = moe.Workspace(moe.workspace_size(shape))
    x = synth.make_x(B, H, seed=43)
    lg = synth.make_logits(B, E, seed=43, zipf_s=synth.ZIPF_S)
    xd, lgd = x.cuda(), lg.cuda()
    before = moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _timed_out(moe, lambda: moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws))
    assert ws.status(clear=True) == MOE_ERR_TIMEOUT
    for _ in range(2):
        after = moe.moe_forward(shape, lgd, xd, Wg, Wu, Wd, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert torch.equal(after, before)
    ref, _, _ = oracle_rows(synth.bf16_bits(x), lg.numpy(), k, DeviceExperts(Wg, Wu, Wd),
                            np.arange(B))
    assert_close(after, ref, "planned batch after a timed-out step")


def test_wait_limit_argument_checked(moe):
    with pytest.raises(moe.MoeError):
        moe.debug_set_wait_limit(-1)
    moe.debug_set_wait_limit(0)
