"""GPU: a captured decode step (DecodeGraph) replayed over changing inputs
gives exactly what moe_forward gives on the same inputs, and matches the
oracle."""
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


@pytest.mark.parametrize("B,E,H,I", [(1, 64, 2048, 1024), (4, 64, 2048, 1024),
                                     (24, 96, 1024, 512)])
def test_decode_graph_replays_match_forward(moe, B, E, H, I):
    k = 8
    shape = moe.Shape(B, E, k, H, I)
    dev = torch.device("cuda")
    W = synth.make_weights(E, H, I, seed=2, layer=0, device=dev)
    g = moe.DecodeGraph(shape, *W)
    for step in range(4):
        lg = synth.make_logits(B, E, seed=step, zipf_s=synth.ZIPF_S).to(dev)
        x = synth.make_x(B, H, seed=100 + step).to(dev)
        g.logits.copy_(lg)
        g.x.copy_(x)
        out = g.replay().clone()
        ref = moe.moe_forward(shape, lg, x, *W)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"step {step}"
        assert torch.equal(g.topk_idx, moe.moe_route(lg, k)[0])
    assert g.ws.status() == 0
    ref0, _, _ = oracle_rows(synth.bf16_bits(x.cpu()), lg.cpu().numpy(), k, DeviceExperts(*W),
                             np.arange(B))
    assert_close(out, ref0, "decode graph")
