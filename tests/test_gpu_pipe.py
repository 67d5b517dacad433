"""GPU: the host-buffer pipeline (moe_forward_host) gives, call after call,
exactly the outputs of moe_forward on device copies of the same inputs, and
matches the oracle."""
import numpy as np
import pytest
import torch

import synth
from parity import DeviceExperts, assert_close, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


@pytest.mark.parametrize("T,E,k,H,I,calls", [(64, 16, 2, 512, 256, 5),
                                              (1024, 32, 8, 2048, 1024, 4),
                                              (3, 64, 8, 2048, 1024, 3)])
def test_pipe_matches_device_forward(moe, T, E, k, H, I, calls):
    shape = moe.Shape(T, E, k, H, I)
    dev = torch.device("cuda")
    Wg, Wu, Wd = synth.make_weights(E, H, I, seed=0, layer=0, device=dev)
    xs = [synth.make_x(T, H, seed=c).pin_memory() for c in range(calls)]
    lgs = [synth.make_logits(T, E, seed=c, zipf_s=synth.ZIPF_S).pin_memory() for c in range(calls)]
    outs = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    pipe = moe.Pipe(shape, dev)
    for c in range(calls):          # enqueued back to back: slots are reused
        pipe.forward(lgs[c], xs[c], Wg, Wu, Wd, outs[c])
    pipe.synchronize()
    assert pipe.ws.status() == 0
    for c in range(calls):
        ref = moe.moe_forward(shape, lgs[c].to(dev), xs[c].to(dev), Wg, Wu, Wd)
        torch.cuda.synchronize()
        assert torch.equal(outs[c], ref.cpu()), f"call {c}"
    toks = np.arange(min(T, 32))
    ref0, _, _ = oracle_rows(synth.bf16_bits(xs[0]), lgs[0].numpy(), k,
                             DeviceExperts(Wg, Wu, Wd), toks)
    assert_close(outs[0][:len(toks)], ref0, "pipe call 0")
    pipe.close()
