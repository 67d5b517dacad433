"""GPU: the HBM expert cache (moe_forward_cached) gives exactly the outputs
of moe_forward on device-resident weights, across calls and evictions, and
copies only what is not resident."""
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


def _layers(moe, E, H, I, L, seed, dev):
    weights = [synth.make_weights(E, H, I, seed=seed, layer=l, device=dev) for l in range(L)]
    host = [moe.pack_layer_weights(*w) for w in weights]
    return weights, host


def _touched(moe, logits, k):
    return [set(torch.unique(moe.moe_route(lg, k)[0]).tolist()) for lg in logits]


@pytest.mark.parametrize("T,E,k,H,I,n_slots", [(64, 32, 4, 512, 256, 40),
                                               (160, 16, 4, 1024, 512, 20),
                                               (3, 64, 8, 1024, 512, 24)])
def test_cache_matches_resident_forward(moe, T, E, k, H, I, n_slots):
    """Three calls over three layers with a cache smaller than their experts
    (evictions across layers and calls); slots start as NaN."""
    L = 3
    dev = torch.device("cuda")
    shape = moe.Shape(T, E, k, H, I)
    weights, host = _layers(moe, E, H, I, L, seed=3, dev=dev)
    cache = moe.ExpertCache(shape, n_slots, L)
    cache.mem.view(torch.int16).fill_(0x7FC0)   # bf16 NaN in every slot
    x = synth.make_x(T, H, seed=5).to(dev)
    ws = moe.Workspace(moe.workspace_size(shape), dev)
    looked_up = 0
    for call in range(3):
        logits = [synth.make_logits(T, E, seed=10 * call + l, zipf_s=synth.ZIPF_S).to(dev)
                  for l in range(L)]
        outs = cache.forward(list(range(L)), logits, x, host, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        for l in range(L):
            ref = moe.moe_forward(shape, logits[l], x, *weights[l])
            torch.cuda.synchronize()
            assert torch.isfinite(outs[l].float()).all(), f"call {call} layer {l}"
            assert torch.equal(outs[l], ref), f"call {call} layer {l}"
        hits, misses = cache.stats()
        looked_up += sum(len(t) for t in _touched(moe, logits, k))
        assert hits + misses == looked_up      # one lookup per touched expert per layer
    assert misses > n_slots                    # the cache was too small: evictions happened
    ref0, _, _ = oracle_rows(synth.bf16_bits(x.cpu()), logits[0].cpu().numpy(), k,
                             DeviceExperts(*weights[0]), np.arange(min(T, 24)))
    assert_close(outs[0][: min(T, 24)], ref0, "cached layer 0")
    cache.close()


def test_cache_hits_when_everything_fits(moe):
    """A cache with room for every touched expert copies each one once: the
    second call with the same routing is all hits."""
    T, E, k, H, I, L = 48, 32, 4, 512, 256, 2
    dev = torch.device("cuda")
    shape = moe.Shape(T, E, k, H, I)
    weights, host = _layers(moe, E, H, I, L, seed=4, dev=dev)
    cache = moe.ExpertCache(shape, L * E, L)
    x = synth.make_x(T, H, seed=6).to(dev)
    logits = [synth.make_logits(T, E, seed=20 + l, zipf_s=synth.ZIPF_S).to(dev) for l in range(L)]
    touched = sum(len(t) for t in _touched(moe, logits, k))
    cache.forward([7, 9], logits, x, host)
    torch.cuda.synchronize()
    assert cache.stats() == (0, touched)
    outs = cache.forward([7, 9], logits, x, host)
    torch.cuda.synchronize()
    assert cache.stats() == (touched, touched)
    for l in range(L):
        assert torch.equal(outs[l], moe.moe_forward(shape, logits[l], x, *weights[l]))
    cache.close()


def test_cache_too_small_for_a_layer(moe):
    T, E, k, H, I = 32, 32, 4, 512, 256
    dev = torch.device("cuda")
    shape = moe.Shape(T, E, k, H, I)
    weights, host = _layers(moe, E, H, I, 1, seed=5, dev=dev)
    cache = moe.ExpertCache(shape, 2, 1)
    x = synth.make_x(T, H, seed=7).to(dev)
    logits = [synth.make_logits(T, E, seed=30).to(dev)]
    with pytest.raises(moe.MoeError) as ei:
        cache.forward([0], logits, x, host)
    assert ei.value.status == 1
    torch.cuda.synchronize()
    cache.close()


def test_cache_rejects_host_weights_it_cannot_read(moe):
    """The misses are copied by a kernel that reads host memory through the
    device's mapping: pageable or misaligned host weights are refused before
    anything is enqueued."""
    T, E, k, H, I = 8, 16, 2, 512, 256
    dev = torch.device("cuda")
    shape = moe.Shape(T, E, k, H, I)
    cache = moe.ExpertCache(shape, E, 1)
    x = synth.make_x(T, H, seed=8).to(dev)
    logits = [synth.make_logits(T, E, seed=31).to(dev)]
    n = moe.layer_weight_bytes(shape) // 2
    with pytest.raises(moe.MoeError, match="pinned"):
        cache.forward([0], logits, x, [torch.zeros(n, dtype=torch.bfloat16)])
    pinned = torch.zeros(n + 8, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(moe.MoeError, match="16-byte aligned"):
        cache.forward([0], logits, x, [pinned[1:1 + n]])
    assert cache.stats() == (0, 0)
    cache.close()
