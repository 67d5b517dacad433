"""GPU: expert weights streamed from pinned host memory through HBM staging
slots (moe_forward_offload) give exactly the outputs of moe_forward on
device-resident copies of the same weights, and match the oracle."""
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


@pytest.mark.parametrize("T,E,k,H,I,L,slots", [(64, 16, 2, 512, 256, 4, 1),
                                                (64, 16, 2, 512, 256, 5, 2),
                                                (1024, 32, 8, 2048, 1024, 4, 3),
                                                (4, 64, 8, 2048, 1024, 3, 8),
                                                (512, 1024, 8, 256, 256, 2, 2)])
def test_offload_matches_resident_forward(moe, T, E, k, H, I, L, slots):
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    shape = moe.Shape(T, E, k, H, I)
    dev = torch.device("cuda")
    x = synth.make_x(T, H, seed=0).to(dev)
    logits = [synth.make_logits(T, E, seed=0, layer=l, zipf_s=synth.ZIPF_S).to(dev) for l in range(L)]
    weights = [synth.make_weights(E, H, I, seed=0, layer=l, device=dev) for l in range(L)]
    host = [moe.pack_layer_weights(*w) for w in weights]
    st = moe.Stager(shape, slots)
    outs = st.forward(shape, logits, x, host)
    torch.cuda.synchronize()
    for l in range(L):
        ref = moe.moe_forward(shape, logits[l], x, *weights[l])
        torch.cuda.synchronize()
        assert torch.equal(outs[l], ref), f"layer {l}"
    # layer 0 against the oracle
    experts = DeviceExperts(*weights[0])
    toks = np.arange(min(T, 48))
    ref0, _, _ = oracle_rows(synth.bf16_bits(x.cpu()), logits[0].cpu().numpy(), k, experts, toks)
    assert_close(outs[0][:len(toks)], ref0, "offload layer 0")
    st.close()


@pytest.mark.parametrize("T,E,k,H,I,L,slots", [(4, 64, 8, 512, 256, 3, 2),
                                                (512, 48, 4, 1024, 512, 4, 3)])
def test_offload_copies_exactly_the_touched_experts(moe, T, E, k, H, I, L, slots):
    """Slots are filled with NaN before the forward: only the experts a
    layer's tokens are routed to are copied, and nothing else is read, so the
    outputs still equal the resident forward (and hold no NaN)."""
    shape = moe.Shape(T, E, k, H, I)
    dev = torch.device("cuda")
    x = synth.make_x(T, H, seed=1).to(dev)
    logits = [synth.make_logits(T, E, seed=1, layer=l, zipf_s=synth.ZIPF_S).to(dev) for l in range(L)]
    weights = [synth.make_weights(E, H, I, seed=1, layer=l, device=dev) for l in range(L)]
    host = [moe.pack_layer_weights(*w) for w in weights]
    st = moe.Stager(shape, slots)
    st.slots.view(torch.int16).fill_(0x7FC0)        # bf16 quiet NaN
    torch.cuda.synchronize()
    outs = st.forward(shape, logits, x, host)
    torch.cuda.synchronize()
    touched = [torch.unique(moe.moe_route(lg, k)[0]).numel() for lg in logits]
    assert min(touched) < E                         # some experts are never copied
    for l in range(L):
        ref = moe.moe_forward(shape, logits[l], x, *weights[l])
        torch.cuda.synchronize()
        assert torch.isfinite(outs[l].float()).all(), f"layer {l}"
        assert torch.equal(outs[l], ref), f"layer {l}"
    st.close()


def test_offload_argument_errors(moe):
    shape = moe.Shape(8, 16, 2, 512, 256)
    small = moe.Shape(8, 8, 2, 512, 256)
    st = moe.Stager(small, 2)      # slots sized for 8 experts
    x = torch.zeros((8, 512), dtype=torch.bfloat16, device="cuda")
    lg = [torch.zeros((8, 16), device="cuda")]
    host = [torch.zeros(moe.layer_weight_bytes(shape) // 2, dtype=torch.bfloat16).pin_memory()]
    with pytest.raises(moe.MoeError):
        st.forward(shape, lg, x, host)            # 16 experts do not fit a slot
    s2 = torch.cuda.current_stream()
    with pytest.raises(moe.MoeError):
        st.forward(small, [torch.zeros((8, 8), device="cuda")], x,
                   [torch.zeros(moe.layer_weight_bytes(small) // 2, dtype=torch.bfloat16).pin_memory()],
                   compute=s2, copy=s2)          # copy stream must differ
    nbytes = moe.layer_weight_bytes(small)
    pageable = torch.zeros(nbytes // 2, dtype=torch.bfloat16)
    with pytest.raises(moe.MoeError, match="pinned"):
        st.forward(small, [torch.zeros((8, 8), device="cuda")], x, [pageable])
    pinned = torch.zeros(nbytes // 2 + 8, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(moe.MoeError, match="16-byte aligned"):
        st.forward(small, [torch.zeros((8, 8), device="cuda")], x, [pinned[1:1 + nbytes // 2]])
    st.close()
