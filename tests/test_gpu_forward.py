"""GPU parity: expert FFN, combine and the whole layer against the oracle.

Routing indices, counts and the permutation must match bit-exactly; bf16
outputs within relative RMS 5e-3 and max-abs 2e-2.  Small layers are checked
on every output; full-size layers on every token whose oracle cost is
bounded (decode) or on a seeded token sample chosen to cover both expert
paths (prefill), since each output row depends only on its own token.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceExperts, GATE_ATOL, assert_close, oracle_rows, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


def _to_dev(inp):
    return {k: v.cuda() for k, v in inp.items()}


def _forward(moe, shape, d, profiled=False):
    T, k = shape.T, shape.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.Workspace(moe.workspace_size(shape))
    if profiled:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(moe.PROFILE_EVENTS)]
        out = moe.moe_forward_profiled(shape, d["logits"], d["x"], d["Wg"], d["Wu"], d["Wd"],
                                       ev, topk_idx=idx, gates=gates, ws=ws)
    else:
        out = moe.moe_forward(shape, d["logits"], d["x"], d["Wg"], d["Wu"], d["Wd"],
                              topk_idx=idx, gates=gates, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return out, idx, gates


# thin_mma_min values: 1 = every thin expert on the tensor-core streaming
# kernel, 33 = every thin expert on the CUDA-core one (0 = chosen by shape).
MMA_ALL, MMA_NONE = 1, 33
# Widths at which a self-routed batch on the CUDA-core streaming kernel runs
# the whole layer in one cooperative launch (two launches elsewhere).
ONE_LAUNCH_WIDTHS = {(4096, 2048), (2048, 1024), (512, 256)}


def self_routed_launches(H, I, mma_min):
    return 1 if mma_min == MMA_NONE and (H, I) in ONE_LAUNCH_WIDTHS else 2


def _full_check(moe, s, thr, inp, d=None, mma_min=0):
    d = d or _to_dev(inp)
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I, fat_threshold=thr, thin_mma_min=mma_min)
    out, idx, gates = _forward(moe, shape, d)
    experts = DeviceExperts(d["Wg"], d["Wu"], d["Wd"])
    ref, ridx, rgates = oracle_rows(synth.bf16_bits(inp["x"]), inp["logits"].numpy(), s.k,
                                    experts, np.arange(s.T))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(gates.cpu().numpy(), rgates, rtol=0, atol=GATE_ATOL)
    return assert_close(out, ref, f"forward {s} thr={thr} mma_min={mma_min}")


# ---------------------------------------------------------------- tiny layer

@pytest.mark.parametrize("mma_min", [MMA_ALL, 7, MMA_NONE])
@pytest.mark.parametrize("thr", [0, 1, 8, 32, 33])
def test_forward_tiny(moe, thr, mma_min):
    """T=64, E=16, top-2, H=512, I=256 (seed 0).  thr=0 sends every expert to
    the tcgen05 GEMM, thr=32/33 every expert to the weight-streaming path;
    mma_min splits the thin experts (5..13 slots here) between the two
    streaming kernels."""
    inp = synth.make_layer(synth.TINY, seed=0)
    _full_check(moe, synth.TINY, thr, inp, mma_min=mma_min)


def test_expert_ffn_and_combine_entry_points(moe):
    """route -> permute -> expert_ffn -> combine through the separate entry
    points; y_sorted row by row and out against the oracle."""
    s = synth.Shape(T=96, E=8, k=3, H=256, I=512)
    inp = synth.make_layer(s, seed=4, zipf_s=1.1)
    d = _to_dev(inp)
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I, fat_threshold=32)
    idx, gates = moe.moe_route(d["logits"], s.k)
    counts, offsets, perm, inv = moe.moe_permute(idx, s.E)
    y = moe.moe_expert_ffn(shape, d["x"], perm, offsets, counts, d["Wg"], d["Wu"], d["Wd"])
    out = moe.moe_combine(y, inv, gates, s.T, s.k, s.H)
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    assert (c >= 32).any() and ((c > 0) & (c < 32)).any(), c   # both paths ran
    xb = synth.bf16_bits(inp["x"])
    experts = DeviceExperts(d["Wg"], d["Wu"], d["Wd"])
    p_perm = perm.cpu().numpy()
    p_off = offsets.cpu().numpy()
    y_ref = np.empty((s.P, s.H))
    for e in range(s.E):
        for p in range(p_off[e], p_off[e + 1]):
            _, y_ref[p] = oracle.expert_ffn(xb[p_perm[p] // s.k], *experts(e))
    assert_close(y, y_ref, "y_sorted")
    out_ref = oracle.combine(y_ref, inv.cpu().numpy(), gates.cpu().numpy().astype(np.float64))
    assert_close(out, out_ref, "combine")


def test_combine_matches_oracle(moe):
    T, k, H = 300, 8, 1024
    g = torch.Generator().manual_seed(9)
    y = torch.randn((T * k, H), generator=g).to(torch.bfloat16)
    inv = torch.randperm(T * k, generator=g).to(torch.int32)
    gates = torch.rand((T, k), generator=g)
    gates = gates / gates.sum(1, keepdim=True)
    out = moe.moe_combine(y.cuda(), inv.cuda(), gates.cuda(), T, k, H)
    torch.cuda.synchronize()
    ref = oracle.combine(oracle.bf16_bits_to_f64(synth.bf16_bits(y)), inv.numpy(),
                         gates.numpy().astype(np.float64))
    assert_close(out, ref, "combine")


def _assigned_logits(counts, E):
    """Logits that send exactly counts[e] tokens to expert e (top-1)."""
    tok = np.repeat(np.arange(E), counts)
    rng = np.random.default_rng(0)
    rng.shuffle(tok)
    lg = rng.standard_normal((len(tok), E)).astype(np.float32)
    lg[np.arange(len(tok)), tok] = 10.0
    return torch.from_numpy(lg)


@pytest.mark.parametrize("mma_min", [MMA_ALL, 31, MMA_NONE])
def test_forward_threshold_edges(moe, mma_min):
    """Experts with exactly 0, 1, 31, 32, 33, 128, 129 and 255 slots: the
    fat-threshold boundary and ragged GEMM tiles (mma_min=31: only the
    31-slot expert streams on the tensor cores)."""
    counts = [31, 32, 33, 0, 1, 128, 129, 255]
    E = len(counts)
    lg = _assigned_logits(counts, E)
    s = synth.Shape(T=lg.shape[0], E=E, k=1, H=256, I=256)
    inp = synth.make_layer(s, seed=6)
    inp["logits"] = lg
    _full_check(moe, s, 32, inp, mma_min=mma_min)
    # k = 2 on the same tokens
    s2 = synth.Shape(T=lg.shape[0], E=E, k=2, H=256, I=256)
    inp["logits"] = lg
    _full_check(moe, s2, 32, inp, mma_min=mma_min)


# Small batches route themselves inside the streaming kernels and combine in
# the down kernel (two launches, or one at the one-launch widths on the
# CUDA-core kernel): T*k <= 32, T below the fat threshold, all
# touched experts on the tensor-core kernel or all on the CUDA-core kernel
# within one streaming unit.
SELF_ROUTED = [
    # T, E, k, H, I
    (1, 16, 2, 512, 256),
    (3, 16, 2, 512, 256),
    (16, 64, 2, 512, 256),     # 32 slots in units of 16
    (4, 1024, 8, 256, 256),    # E = 1024: 32 router candidates per lane
    (5, 3, 2, 768, 512),       # sizes that are not powers of two
    (2, 1, 1, 256, 256),       # a single expert
    (6, 8, 5, 1280, 768),      # 30 slots, k = 5
    (2, 64, 8, 2048, 1024),    # one launch on CUDA cores at this width
]


@pytest.mark.parametrize("mma_min", [MMA_NONE, MMA_ALL])
@pytest.mark.parametrize("T,E,k,H,I", SELF_ROUTED)
def test_forward_self_routed(moe, T, E, k, H, I, mma_min):
    """Routing bit-exact and outputs against the oracle; and bit-identical to
    the same batch through the separate entry points (router, route lists,
    expert FFN on the planner's units or tiles, combine)."""
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    inp = synth.make_layer(s, seed=100 + T, zipf_s=synth.ZIPF_S)
    d = _to_dev(inp)
    shape = moe.Shape(T, E, k, H, I, fat_threshold=32, thin_mma_min=mma_min)
    assert moe.forward_launches(shape) == self_routed_launches(H, I, mma_min)
    _full_check(moe, s, 32, inp, d, mma_min=mma_min)
    out, idx, gates = _forward(moe, shape, d)
    idx2, gates2 = moe.moe_route(d["logits"], k)
    counts, offsets, perm, inv = moe.moe_permute(idx2, E)
    y = moe.moe_expert_ffn(shape, d["x"], perm, offsets, counts, d["Wg"], d["Wu"], d["Wd"])
    out2 = moe.moe_combine(y, inv, gates2, T, k, H)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(gates, gates2)
    assert torch.equal(out, out2)


def test_forward_self_routed_ties_and_reuse(moe):
    """All-equal logits (every token takes experts 0..k-1, gates 1/k: the
    lowest-index tie-break), on a workspace that a routed-and-planned prefill
    batch used before, and that batch again afterwards."""
    s = synth.Shape(T=4, E=16, k=4, H=512, I=256)
    inp = synth.make_layer(s, seed=5)
    inp["logits"] = torch.zeros((s.T, s.E))
    d = _to_dev(inp)
    big = synth.Shape(T=64, E=16, k=4, H=512, I=256)
    binp = synth.make_layer(big, seed=5, zipf_s=synth.ZIPF_S)
    bd = dict(_to_dev(binp), Wg=d["Wg"], Wu=d["Wu"], Wd=d["Wd"])
    bshape = moe.Shape(big.T, big.E, big.k, big.H, big.I, fat_threshold=32,
                       thin_mma_min=MMA_NONE)
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I, fat_threshold=32, thin_mma_min=MMA_NONE)
    ws = moe.Workspace(max(moe.workspace_size(bshape), moe.workspace_size(shape)))
    first = moe.moe_forward(bshape, bd["logits"], bd["x"], bd["Wg"], bd["Wu"], bd["Wd"], ws=ws)
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    out = moe.moe_forward(shape, d["logits"], d["x"], d["Wg"], d["Wu"], d["Wd"],
                          topk_idx=idx, gates=gates, ws=ws)
    again = moe.moe_forward(bshape, bd["logits"], bd["x"], bd["Wg"], bd["Wu"], bd["Wd"], ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(first, again)
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(s.k, dtype=np.int32), (s.T, 1)))
    assert np.allclose(gates.cpu().numpy(), 1.0 / s.k, rtol=0, atol=GATE_ATOL)
    experts = DeviceExperts(d["Wg"], d["Wu"], d["Wd"])
    ref, _, _ = oracle_rows(synth.bf16_bits(inp["x"]), inp["logits"].numpy(), s.k, experts,
                            np.arange(s.T))
    assert_close(out, ref, "self-routed ties")


@pytest.mark.parametrize("H,I,mma_min", [(1024, 512, MMA_NONE), (1024, 512, MMA_ALL),
                                         (512, 256, MMA_NONE)])
def test_forward_self_routed_back_to_back(moe, H, I, mma_min):
    """Self-routed decode steps of batch 1, 2 and 4 enqueued back to back on
    one workspace with no synchronisation between them (programmatic
    dependent launch on): every step's fused combine counts its down CTAs on
    the same ticket word, so a ticket left behind by one step would make the
    next step combine early or not at all; the one-launch layer (H=512,
    I=256) also counts its CTAs between the gate/up and down phases on one
    word, which a step must leave at a multiple of the grid.  Each step
    against the oracle."""
    E, k = 64, 8
    Wg, Wu, Wd = synth.make_weights(E, H, I, seed=21, layer=0, device="cuda")
    experts = DeviceExperts(Wg, Wu, Wd)
    batches = [1, 2, 4, 4, 1, 2, 1, 4]
    shapes = {B: moe.Shape(B, E, k, H, I, fat_threshold=32, thin_mma_min=mma_min)
              for B in set(batches)}
    for sh in shapes.values():
        assert moe.forward_launches(sh) == self_routed_launches(H, I, mma_min)
    ws = moe.Workspace(max(moe.workspace_size(sh) for sh in shapes.values()))
    steps = []
    for r, B in enumerate(batches):
        x = synth.make_x(B, H, seed=200 + r)
        lg = synth.make_logits(B, E, seed=200 + r, zipf_s=synth.ZIPF_S)
        out = moe.moe_forward(shapes[B], lg.cuda(), x.cuda(), Wg, Wu, Wd, ws=ws)
        steps.append((x, lg, out))
    torch.cuda.synchronize()
    assert ws.status() == 0
    for r, (x, lg, out) in enumerate(steps):
        ref, _, _ = oracle_rows(synth.bf16_bits(x), lg.numpy(), k, experts,
                                np.arange(x.shape[0]))
        assert_close(out, ref, f"step {r} (B={x.shape[0]})")


def test_forward_gemm_pair_boundaries(moe):
    """The grouped GEMM runs an expert's 128-row tiles in pairs (256 rows per
    CTA pair): slot counts on either side of pair and tile boundaries, so
    pairs whose second tile is partial or empty."""
    counts = [129, 255, 256, 257, 383, 384, 385, 512, 40]
    E = len(counts)
    lg = _assigned_logits(counts, E)
    s = synth.Shape(T=lg.shape[0], E=E, k=1, H=256, I=256)
    inp = synth.make_layer(s, seed=11)
    inp["logits"] = lg
    _full_check(moe, s, 32, inp)


def test_forward_one_expert_takes_all(moe):
    s = synth.Shape(T=700, E=4, k=1, H=512, I=256)
    inp = synth.make_layer(s, seed=7)
    inp["logits"] = torch.zeros((s.T, s.E))
    inp["logits"][:, 2] = 1.0
    _full_check(moe, s, 32, inp)


def test_forward_T0_is_noop(moe):
    shape = moe.Shape(0, 16, 2, 512, 256)
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    W = torch.empty((16, 256, 512), dtype=torch.bfloat16, device="cuda")
    Wd = torch.empty((16, 512, 256), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(shape, torch.empty((0, 16), device="cuda"), x, W, W, Wd,
                    out=torch.empty((1, 512), dtype=torch.bfloat16, device="cuda"))


def test_forward_rejects_small_workspace(moe):
    s = synth.TINY
    d = _to_dev(synth.make_layer(s, seed=0))
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I)
    ws = moe.Workspace(1024)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward(shape, d["logits"], d["x"], d["Wg"], d["Wu"], d["Wd"], ws=ws)
    assert ei.value.status == 3


# ------------------------------------------------------ full-size layer (E=384)

@pytest.fixture(scope="module")
def big_layer():
    """One layer of the full model shape, weights generated on the device:
    384 experts, H=4096, I=2048 (19.3 GB of bf16 weights)."""
    s = synth.PREFILL
    Wg, Wu, Wd = synth.make_weights(s.E, s.H, s.I, seed=0, layer=0, device="cuda")
    yield dict(Wg=Wg, Wu=Wu, Wd=Wd)
    del Wg, Wu, Wd
    torch.cuda.empty_cache()


def _forward_vs_entry_points(moe, s, shape, d, inp, launches):
    """moe_forward on a whole batch: the expected launch count, routing
    bit-exact, every output against the oracle, and bit-identical to router,
    route lists, expert FFN and combine called one by one."""
    assert moe.forward_launches(shape) == launches
    out, idx, gates = _forward(moe, shape, d)
    experts = DeviceExperts(d["Wg"], d["Wu"], d["Wd"])
    ref, ridx, rgates = oracle_rows(synth.bf16_bits(inp["x"]), inp["logits"].numpy(), s.k,
                                    experts, np.arange(s.T))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(gates.cpu().numpy(), rgates, rtol=0, atol=GATE_ATOL)
    assert_close(out, ref, f"self-routed {s}")
    idx2, gates2 = moe.moe_route(d["logits"], s.k)
    counts, offsets, perm, inv = moe.moe_permute(idx2, s.E)
    y = moe.moe_expert_ffn(shape, d["x"], perm, offsets, counts, d["Wg"], d["Wu"], d["Wd"])
    out2 = moe.moe_combine(y, inv, gates2, s.T, s.k, s.H)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(gates, gates2)
    assert torch.equal(out, out2)


# Batches of 33..256 slots on the tensor-core streaming kernel run the
# router, route-list and gather kernels (measured faster than routing inside
# the streaming kernels at these sizes) and combine in the down kernel (a
# cooperative launch): five launches.
PLANNED_MMA = [
    # T, E, k, H, I, fat threshold, launches
    (12, 5, 3, 768, 512, 32, 5),      # 36 slots on 5 experts (up to 12 slots each)
    (20, 1024, 8, 256, 256, 32, 5),   # 160 slots, E = 1024
    (32, 64, 8, 512, 256, 33, 5),     # 256 slots: the plan's capacity
    (9, 40, 6, 1280, 768, 32, 5),     # 54 slots, k = 6, H not a power of two
    (32, 10, 8, 512, 256, 32, 11),    # two 32-slot (fat) experts beside thin ones: GEMMs too
]


@pytest.mark.parametrize("T,E,k,H,I,thr,launches", PLANNED_MMA)
def test_forward_mma_batches_33_to_256_slots(moe, T, E, k, H, I, thr, launches):
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    inp = synth.make_layer(s, seed=300 + T, zipf_s=synth.ZIPF_S)
    shape = moe.Shape(T, E, k, H, I, fat_threshold=thr, thin_mma_min=MMA_ALL)
    _forward_vs_entry_points(moe, s, shape, _to_dev(inp), inp, launches)


@pytest.mark.parametrize("B", [5, 8, 16, 24])
def test_forward_decode_sweep_batches(moe, big_layer, B):
    """Decode batches 5..24 at full size (E=384, top-8, H=4096, I=2048), the
    decode sweep's batches, on the tensor-core streaming kernels (the default
    for these shapes), every output against the oracle."""
    s = synth.Shape(T=B, E=384, k=8, H=4096, I=2048)
    inp = dict(x=synth.make_x(B, s.H, seed=400 + B),
               logits=synth.make_logits(B, s.E, seed=400 + B, zipf_s=synth.ZIPF_S))
    d = dict(_to_dev(inp), **big_layer)
    shape = moe.Shape(B, s.E, s.k, s.H, s.I)
    _forward_vs_entry_points(moe, s, shape, d, inp, 5)


@pytest.mark.parametrize("B,mma_min", [(1, 0), (2, 0), (4, MMA_NONE)])
def test_forward_decode_one_launch(moe, big_layer, B, mma_min):
    """Full-size decode batches on the CUDA-core streaming kernel (batches 1
    and 2 by default, 4 when forced: 32 slots): the whole layer in one
    cooperative launch, every output against the oracle and bit-identical to
    the separate entry points."""
    s = synth.Shape(T=B, E=384, k=8, H=4096, I=2048)
    inp = dict(x=synth.make_x(B, s.H, seed=500 + B),
               logits=synth.make_logits(B, s.E, seed=500 + B, zipf_s=synth.ZIPF_S))
    d = dict(_to_dev(inp), **big_layer)
    shape = moe.Shape(B, s.E, s.k, s.H, s.I, thin_mma_min=mma_min)
    _forward_vs_entry_points(moe, s, shape, d, inp, 1)


@pytest.mark.parametrize("mma_min", [MMA_ALL, MMA_NONE])
@pytest.mark.parametrize("B", [1, 4])
def test_forward_decode(moe, big_layer, B, mma_min):
    s = synth.Shape(T=B, E=384, k=8, H=4096, I=2048)
    inp = dict(x=synth.make_x(B, s.H, seed=0), logits=synth.make_logits(B, s.E, seed=0,
                                                                           zipf_s=synth.ZIPF_S))
    d = dict(_to_dev(inp), **big_layer)
    _full_check(moe, s, 32, inp, d, mma_min=mma_min)


@pytest.mark.parametrize("H,I,mma_min", [(4096, 2048, 0), (4096, 2048, MMA_NONE),
                                         (2048, 1024, 0)])
def test_forward_prefill_sampled(moe, big_layer, H, I, mma_min):
    """16,384-token chunk, Zipf(1.1)-skewed routing.  Routing, counts and the
    permutation are checked on all tokens; outputs on a sample covering random
    tokens, tokens of thin experts and of the smallest and hottest fat expert."""
    s = synth.Shape(T=16384, E=384, k=8, H=H, I=I)
    inp = dict(x=synth.make_x(s.T, H, seed=0),
               logits=synth.make_logits(s.T, s.E, seed=0, zipf_s=synth.ZIPF_S))
    if H == 4096:
        W = big_layer
    else:
        Wg, Wu, Wd = synth.make_weights(s.E, H, I, seed=0, layer=0, device="cuda")
        W = dict(Wg=Wg, Wu=Wu, Wd=Wd)
    d = dict(_to_dev(inp), **W)
    shape = moe.Shape(s.T, s.E, s.k, H, I, fat_threshold=32, thin_mma_min=mma_min)
    out, idx, gates = _forward(moe, shape, d)
    lg = inp["logits"].numpy()
    ridx, rgates = oracle.route(lg, s.k)
    idx_np = idx.cpu().numpy()
    assert np.array_equal(idx_np, ridx)
    assert np.allclose(gates.cpu().numpy(), rgates, rtol=0, atol=GATE_ATOL)
    counts, offsets, perm, inv = moe.moe_permute(idx, s.E)
    rc, ro, rp, ri = oracle.permute(ridx, s.E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)
    assert (rc >= 32).sum() > 0 and ((rc > 0) & (rc < 32)).sum() > 0
    toks = sample_tokens(ridx, rc, 32, np.random.default_rng(1))
    experts = DeviceExperts(W["Wg"], W["Wu"], W["Wd"])
    ref, _, _ = oracle_rows(synth.bf16_bits(inp["x"]), lg, s.k, experts, toks)
    assert_close(out[torch.from_numpy(toks).cuda()], ref, f"prefill H={H} mma_min={mma_min}")


def test_forward_deterministic_and_profiled(moe, big_layer):
    s = synth.Shape(T=2048, E=384, k=8, H=4096, I=2048)
    inp = dict(x=synth.make_x(s.T, s.H, seed=1),
               logits=synth.make_logits(s.T, s.E, seed=1, zipf_s=synth.ZIPF_S))
    d = dict(_to_dev(inp), **big_layer)
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I)
    a, _, _ = _forward(moe, shape, d)
    b, _, _ = _forward(moe, shape, d)
    c, _, _ = _forward(moe, shape, d, profiled=True)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_decode_sweep_four_layers(moe):
    """Decode batch 24 over 4 resident layers (77 GB of weights); two layers
    checked in full against the oracle, all four for routing."""
    s = synth.Shape(T=24, E=384, k=8, H=4096, I=2048)
    layers = [synth.make_weights(s.E, s.H, s.I, seed=0, layer=l, device="cuda")
              for l in range(4)]
    x = synth.make_x(s.T, s.H, seed=0)
    for l, (Wg, Wu, Wd) in enumerate(layers):
        inp = dict(x=x, logits=synth.make_logits(s.T, s.E, seed=0, layer=l,
                                                 zipf_s=synth.ZIPF_S))
        d = dict(_to_dev(inp), Wg=Wg, Wu=Wu, Wd=Wd)
        if l in (0, 3):
            _full_check(moe, s, 32, inp, d)
        else:
            shape = moe.Shape(s.T, s.E, s.k, s.H, s.I)
            _, idx, _ = _forward(moe, shape, d)
            assert np.array_equal(idx.cpu().numpy(), oracle.route(inp["logits"].numpy(), s.k)[0])
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,k,H,I", [(40, 8, 2, 768, 512), (20, 4, 4, 256, 768),
                                       (70, 6, 3, 1280, 256), (33, 33, 1, 2048, 1024)])
@pytest.mark.parametrize("thr,mma_min", [(0, 0), (33, MMA_ALL), (33, MMA_NONE)])
def test_forward_odd_shapes(moe, T, E, k, H, I, thr, mma_min):
    """Hidden sizes that are not powers of two, all three expert kernels."""
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    _full_check(moe, s, thr, synth.make_layer(s, seed=T, zipf_s=synth.ZIPF_S), mma_min=mma_min)


@pytest.mark.parametrize("mma_min", [MMA_NONE, 13, MMA_ALL])
def test_thin_units_split_at_full_width(moe, mma_min):
    """Full-width experts (H=4096, I=2048) with 1..32 slots on the weight-
    streaming path (threshold 33).  On CUDA cores, experts with more slots
    than one unit holds are split into several units, each streaming the
    weights again; on the tensor cores one tile holds up to 32 slots."""
    counts = [1, 12, 13, 24, 25, 31, 32, 2]
    E = len(counts)
    lg = _assigned_logits(counts, E)
    s = synth.Shape(T=lg.shape[0], E=E, k=1, H=4096, I=2048)
    inp = synth.make_layer(s, seed=8)
    inp["logits"] = lg
    _full_check(moe, s, 33, inp, mma_min=mma_min)


@pytest.mark.parametrize("T,E,k,H,I", [(64, 1024, 8, 256, 256),     # most experts, top-8
                                       (40, 4, 2, 16384, 256),      # largest hidden size
                                       (40, 4, 2, 256, 16384)])     # largest intermediate size
@pytest.mark.parametrize("thr,mma_min", [(0, 0), (33, MMA_ALL), (33, MMA_NONE)])
def test_forward_maximum_sizes(moe, T, E, k, H, I, thr, mma_min):
    """The limits moe.h accepts (E = 1024, H or I = 16384) on each expert
    kernel: grouped GEMM (thr=0), tensor-core and CUDA-core weight streaming.
    The max-abs bound was set at the model's magnitudes (H = 4096, I = 2048);
    with the fixed 0.02 weight scale, pre-activations grow with sqrt(H) and
    sqrt(I), so the weights are rescaled to keep that variance (one bf16 ulp
    of an output near 8 is already 0.03).  The oracle reads the same bytes."""
    s = synth.Shape(T=T, E=E, k=k, H=H, I=I)
    inp = synth.make_layer(s, seed=T + E, zipf_s=synth.ZIPF_S)
    gu, d = min(1.0, (4096 / H) ** 0.5), min(1.0, (2048 / I) ** 0.5)
    inp["Wg"] = (inp["Wg"].float() * gu).to(torch.bfloat16)
    inp["Wu"] = (inp["Wu"].float() * gu).to(torch.bfloat16)
    inp["Wd"] = (inp["Wd"].float() * d).to(torch.bfloat16)
    _full_check(moe, s, thr, inp, mma_min=mma_min)


@pytest.mark.parametrize("T", [256, 257])
def test_route_lists_at_the_small_path_boundary(moe, T):
    """T*k = 2048 takes the single-block route-list kernel, 2056 the
    histogram / scan / scatter kernels: both bit-exact, same forward."""
    s = synth.Shape(T=T, E=64, k=8, H=256, I=256)
    inp = synth.make_layer(s, seed=T, zipf_s=synth.ZIPF_S)
    _full_check(moe, s, 32, inp)
    idx, _ = moe.moe_route(inp["logits"].cuda(), s.k)
    counts, offsets, perm, inv = moe.moe_permute(idx, s.E)
    rc, ro, rp, ri = oracle.permute(idx.cpu().numpy(), s.E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp) and np.array_equal(inv.cpu().numpy(), ri)


@pytest.mark.parametrize("thr", [0, 33])
def test_forward_single_expert(moe, thr):
    """E = 1, k = 1: every token's gate is 1 and the layer is one dense
    SwiGLU FFN (GEMM or streaming path)."""
    s = synth.Shape(T=50, E=1, k=1, H=512, I=256)
    _full_check(moe, s, thr, synth.make_layer(s, seed=3))
