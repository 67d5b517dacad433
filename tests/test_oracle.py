"""Pins for the oracle: each test checks it against something other than
itself -- brute force, library routines, closed forms, invariants.

The pages print no worked tensors, so nothing here is a printed value; the
hand-worked example in tests/golden/hand_worked_layer.json is checked against
its closed form written out in this file.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_round_special_values():
    f = oracle.to_bf16_bits
    # exact values
    assert f(np.array([1.0]))[0] == 0x3F80
    assert f(np.array([-2.0]))[0] == 0xC000
    assert f(np.array([0.0]))[0] == 0x0000
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert f(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1+2^-7 (odd) and 1+2^-6 (even) -> up
    assert f(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above a tie rounds up (a double rounding via fp32 would miss this)
    assert f(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    # overflow to inf, and the largest finite value
    assert f(np.array([1e39]))[0] == 0x7F80
    assert f(np.array([3.3895313892515355e38]))[0] == 0x7F7F


def test_bf16_round_matches_torch_on_fp32_values():
    # For inputs that are fp32 values there is only one rounding, so the
    # result must equal torch's fp32 -> bf16 round-to-nearest-even.
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    mine = oracle.to_bf16_bits(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_widening_exact():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    back = oracle.to_bf16_bits(vals[finite])
    # -0.0 maps back to 0x8000 and every finite pattern round-trips
    assert np.array_equal(back, bits[finite])


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

def brute_force_topk(l, k):
    """Definition by counting: expert e sits at output position
    #{f : l_f > l_e or (l_f == l_e and f < e)}; it is selected iff that is < k."""
    E = len(l)
    out = [None] * k
    for e in range(E):
        pos = sum(1 for f in range(E) if l[f] > l[e] or (l[f] == l[e] and f < e))
        if pos < k:
            out[pos] = e
    return out


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8, 16])
def test_route_matches_brute_force(E):
    rng = np.random.default_rng(E)
    for trial in range(4):
        T = 64
        if trial % 2 == 0:
            logits = rng.standard_normal((T, E)).astype(np.float32)
        else:  # heavy ties
            logits = rng.integers(0, 3, (T, E)).astype(np.float32)
        if trial == 3:
            logits[:, ::2] = -np.inf
            logits[:, 0] = 0.5  # the largest logit must stay finite
        for k in sorted(set([1, max(1, E // 2), E])):
            idx, gates = oracle.route(logits, k)
            for t in range(T):
                assert list(idx[t]) == brute_force_topk(list(logits[t]), k)


def test_route_tie_break_lower_index():
    logits = np.array([[0.0, 1.0, 1.0, 0.5, 1.0]], dtype=np.float32)
    idx, gates = oracle.route(logits, 3)
    assert list(idx[0]) == [1, 2, 4]
    assert np.allclose(gates[0], 1.0 / 3.0, rtol=0, atol=1e-15)
    # -0.0 and +0.0 are equal logits: the lower index wins
    logits = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)
    idx, _ = oracle.route(logits, 1)
    assert idx[0, 0] == 0


def test_gates_properties():
    rng = np.random.default_rng(7)
    logits = (rng.standard_normal((200, 40)) * 3).astype(np.float32)
    for k in (1, 2, 8, 40):
        idx, g = oracle.route(logits, k)
        assert np.allclose(g.sum(1), 1.0, rtol=0, atol=1e-12)
        assert np.all(np.diff(g, axis=1) <= 0)          # selection order
        sel = np.take_along_axis(logits.astype(np.float64), idx, axis=1)
        # softmax ratio law: g_i / g_j = exp(l_i - l_j)
        assert np.allclose(g / g[:, :1], np.exp(sel - sel[:, :1]), rtol=1e-12, atol=0)
        if k == 1:
            assert np.all(g == 1.0)
        if k == 40:
            # all experts selected: the gates are the full softmax
            full = scipy.special.softmax(logits.astype(np.float64), axis=1)
            assert np.allclose(np.take_along_axis(full, idx, axis=1), g,
                               rtol=1e-12, atol=1e-15)


def test_route_rejects_bad_logits():
    with pytest.raises(oracle.OracleError):
        oracle.route(np.array([[0.0, np.nan]], dtype=np.float32), 1)
    with pytest.raises(oracle.OracleError):
        oracle.route(np.array([[0.0, np.inf]], dtype=np.float32), 1)
    with pytest.raises(oracle.OracleError):
        oracle.route(np.array([[-np.inf, -np.inf]], dtype=np.float32), 1)
    with pytest.raises(oracle.OracleError):
        oracle.route(np.zeros((1, 3), dtype=np.float32), 4)


# --------------------------------------------------------------------------
# Route lists (stable counting sort)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(0, 4, 2), (1, 384, 8), (64, 16, 2), (3000, 384, 8), (500, 3, 3)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if T:
        logits += synth.zipf_bias(E, 1.1).numpy()
    idx, _ = oracle.route(logits, k)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    flat = idx.reshape(-1)
    P = T * k
    assert counts.sum() == P
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == P
    assert np.array_equal(offsets[1:], np.cumsum(counts))
    assert np.array_equal(np.sort(perm), np.arange(P))               # bijection
    assert np.array_equal(inv[perm], np.arange(P))                   # inverse
    # a stable sort of the slots by expert is exactly numpy's stable argsort
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                              # ascending slots


def test_permute_rejects_out_of_range():
    with pytest.raises(oracle.OracleError):
        oracle.permute(np.array([[0, 4]], dtype=np.int32), 4)


# --------------------------------------------------------------------------
# Expert FFN and the whole layer
# --------------------------------------------------------------------------

def _bf16_random(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(shape, generator=g) * std).to(torch.bfloat16)
    return t


def test_single_expert_equals_dense_swiglu():
    # E = 1, k = 1: the gate is 1 and the layer is a dense SwiGLU FFN,
    # computed here independently with torch fp64 library routines.
    T, H, I = 12, 48, 32  # H != I so a transposed operand cannot pass
    x = _bf16_random((T, H), 1.0, 1)
    Wg = _bf16_random((1, I, H), 0.2, 2)
    Wu = _bf16_random((1, I, H), 0.2, 3)
    Wd = _bf16_random((1, H, I), 0.2, 4)
    logits = np.zeros((T, 1), dtype=np.float32)
    out, idx, gates = oracle.moe_tokens(
        synth.bf16_bits(x), logits, 1,
        [(synth.bf16_bits(Wg[0]), synth.bf16_bits(Wu[0]), synth.bf16_bits(Wd[0]))])
    xd, Wgd, Wud, Wdd = (t.double() for t in (x, Wg[0], Wu[0], Wd[0]))
    ref = (torch.nn.functional.silu(xd @ Wgd.T) * (xd @ Wud.T)) @ Wdd.T
    assert np.all(gates == 1.0) and np.all(idx == 0)
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_expert_ffn_intermediate_matches_torch():
    H, I = 40, 24
    x = _bf16_random((H,), 1.0, 5)
    Wg, Wu = _bf16_random((I, H), 0.3, 6), _bf16_random((I, H), 0.3, 7)
    Wd = _bf16_random((H, I), 0.3, 8)
    h, y = oracle.expert_ffn(*(synth.bf16_bits(t) for t in (x, Wg, Wu, Wd)))
    a, b = Wg.double() @ x.double(), Wu.double() @ x.double()
    assert np.allclose(h, (a * torch.sigmoid(a) * b).numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(y, (Wd.double() @ (a * torch.sigmoid(a) * b)).numpy(),
                       rtol=1e-12, atol=1e-14)


def test_combine_closed_form_two_experts():
    # Experts 0 and 1 share W_gate and W_up; expert 1's W_down is exactly
    # twice expert 0's (doubling is exact in bf16), so y_1 = 2 y_0 and
    # out = (g_0 + 2 g_1) y_0 = (1 + g_1) y_0 with g_1 = sigmoid(l_1 - l_0).
    H, I, T = 32, 16, 5
    x = _bf16_random((T, H), 1.0, 11)
    Wg, Wu = _bf16_random((I, H), 0.3, 12), _bf16_random((I, H), 0.3, 13)
    Wd0 = _bf16_random((H, I), 0.3, 14)
    Wd1 = (Wd0.float() * 2).to(torch.bfloat16)
    junk = tuple(synth.bf16_bits(_bf16_random(s, 5.0, 15)) for s in ((I, H), (I, H), (H, I)))
    experts = [tuple(synth.bf16_bits(t) for t in (Wg, Wu, Wd0)),
               tuple(synth.bf16_bits(t) for t in (Wg, Wu, Wd1)), junk]
    logits = np.array([[0.75, -0.5, -3.0], [0.0, 0.0, -1.0], [2.0, 1.5, -9.0],
                       [-1.0, 3.0, -2.0], [0.25, 0.125, -0.25]], dtype=np.float32)
    out, idx, gates = oracle.moe_tokens(synth.bf16_bits(x), logits, 2, experts)
    g1 = scipy.special.expit(logits[:, 1].astype(np.float64) - logits[:, 0])
    for t in range(T):
        _, y0 = oracle.expert_ffn(synth.bf16_bits(x[t]), *experts[0])
        assert np.allclose(out[t], (1.0 + g1[t]) * y0, rtol=1e-12, atol=1e-14)


def test_token_order_permutation_invariance():
    shape = synth.Shape(T=24, E=8, k=3, H=64, I=32)
    inp = synth.make_layer(shape, seed=3, zipf_s=1.1)
    xb = synth.bf16_bits(inp["x"])
    lg = inp["logits"].numpy()
    W = [tuple(synth.bf16_bits(w[e]) for w in (inp["Wg"], inp["Wu"], inp["Wd"]))
         for e in range(shape.E)]
    out, idx, gates = oracle.moe_tokens(xb, lg, shape.k, W)
    sigma = np.random.default_rng(0).permutation(shape.T)
    out2, idx2, gates2 = oracle.moe_tokens(xb[sigma], lg[sigma], shape.k, W)
    assert np.array_equal(out2, out[sigma])
    assert np.array_equal(idx2, idx[sigma]) and np.array_equal(gates2, gates[sigma])
    c1, _, p1, _ = oracle.permute(idx, shape.E)
    c2, o2, p2, _ = oracle.permute(idx2, shape.E)
    assert np.array_equal(c1, c2)
    # the sorted lists hold the same (token, j) pairs, re-labelled by sigma
    inv_sigma = np.argsort(sigma)
    for e in range(shape.E):
        seg1 = p1[o2[e]:o2[e + 1]]
        seg2 = p2[o2[e]:o2[e + 1]]
        relabel = sorted(inv_sigma[s // shape.k] * shape.k + s % shape.k for s in seg1)
        assert list(seg2) == relabel


def test_hand_worked_layer():
    """A three-expert, top-2 layer small enough to work by hand; the expected
    output is written below as its closed form."""
    with open(os.path.join(GOLDEN, "hand_worked_layer.json")) as f:
        case = json.load(f)
    to_bits = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)
    x = to_bits([case["x"]])
    experts = [tuple(synth.bf16_bits(to_bits(case["experts"][e][name]))
                     for name in ("W_gate", "W_up", "W_down")) for e in range(3)]
    logits = np.array(case["logits"], dtype=np.float32)
    out, idx, gates = oracle.moe_tokens(synth.bf16_bits(x), logits, 2, experts)
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    # selection [1, 2]; gates sigmoid(1), sigmoid(-1)
    g1, g2 = sig(1.0), sig(-1.0)
    # expert 1: a = 1, b = 1 -> h = silu(1) = sig(1); y = [h, -2h]
    h1 = 1.0 * sig(1.0) * 1.0
    y1 = [h1, -2.0 * h1]
    # expert 2: a = -1, b = 3 -> h = -sig(-1) * 3; y = [0.5 h, 0.25 h]
    h2 = -1.0 * sig(-1.0) * 3.0
    y2 = [0.5 * h2, 0.25 * h2]
    want = [g1 * y1[c] + g2 * y2[c] for c in range(2)]
    assert list(idx[0]) == [1, 2]
    assert np.allclose(gates[0], [g1, g2], rtol=1e-15, atol=0)
    assert np.allclose(out[0], want, rtol=1e-14, atol=0)


def test_synth_is_deterministic():
    a = synth.make_layer(synth.TINY, seed=0, zipf_s=1.1)
    b = synth.make_layer(synth.TINY, seed=0, zipf_s=1.1)
    for key in a:
        assert torch.equal(a[key], b[key])
    c = synth.make_logits(8, 16, seed=0, rep=1)
    assert not torch.equal(c, synth.make_logits(8, 16, seed=0, rep=0))


def test_combine_one_hot_gates_select_rows():
    # With one-hot gates the combine returns the selected sorted rows exactly.
    rng = np.random.default_rng(3)
    T, k, H = 6, 3, 5
    y = rng.standard_normal((T * k, H))
    inv = rng.permutation(T * k).astype(np.int32)
    g = np.zeros((T, k))
    pick = rng.integers(0, k, T)
    g[np.arange(T), pick] = 1.0
    out = oracle.combine(y, inv, g)
    assert np.array_equal(out, y[inv.reshape(T, k)[np.arange(T), pick]])
    # and it is linear in the gates
    g2 = rng.random((T, k))
    a = oracle.combine(y, inv, g2)
    b = oracle.combine(y, inv, 2.0 * g2)
    assert np.allclose(b, 2.0 * a, rtol=1e-15, atol=0)


def test_combine_adds_its_terms():
    # Partition of unity: every sorted row is the constant vector 1 and the
    # gates are a softmax over the selection, so the combine is sum_j g_j = 1
    # for every token.  A combine that kept one term (the largest gate, the
    # first one) or averaged them would give max g < 1 or 1/k instead.
    rng = np.random.default_rng(5)
    T, E, k, H = 40, 12, 4, 7
    lg = rng.standard_normal((T, E)).astype(np.float32)
    _, gates = oracle.route(lg, k)
    assert gates.max(axis=1).max() < 0.99 and np.abs(gates.sum(1) - 1).max() < 1e-12
    inv = rng.permutation(T * k).astype(np.int32)
    out = oracle.combine(np.ones((T * k, H)), inv, gates)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-14)


def test_combine_of_expert_rows_is_the_layer():
    # The combine, fed the sorted expert outputs of a routed layer (each slot's
    # row from the expert FFN, placed by the route lists), gives the layer
    # output that oracle.moe_tokens computes token by token -- the function
    # pinned above by the dense SwiGLU (E=1), the two-expert closed form and
    # the hand-worked layer.  A combine that dropped, maxed or reordered
    # terms, or read the wrong sorted row, would miss it.
    shape = synth.Shape(T=16, E=6, k=3, H=64, I=32)
    inp = synth.make_layer(shape, seed=9, zipf_s=1.1)
    xb = synth.bf16_bits(inp["x"])
    lg = inp["logits"].numpy()
    W = [tuple(synth.bf16_bits(w[e]) for w in (inp["Wg"], inp["Wu"], inp["Wd"]))
         for e in range(shape.E)]
    ref, idx, gates = oracle.moe_tokens(xb, lg, shape.k, W)
    counts, offsets, perm, inv = oracle.permute(idx, shape.E)
    y_sorted = np.empty((shape.P, shape.H))
    for p, s in enumerate(perm):
        t, j = divmod(int(s), shape.k)
        y_sorted[p] = oracle.expert_ffn(xb[t], *W[idx[t, j]])[1]
    out = oracle.combine(y_sorted, inv, gates)
    assert np.allclose(out, ref, rtol=0, atol=1e-13 * np.abs(ref).max())


def test_workload_expert_mix():
    """The seeded prefill chunk (16,384 tokens, 384 experts, top-8, Zipf(1.1)
    router bias) routes to 233 experts: 81 fat ones (>= 32 slots) holding
    130,162 slots and 152 thin ones holding 910; the decode sweep's 4 layers x
    4 logit sets touch 8 / 12.19 / 17.63 / 24.63 / 32.81 / 38.5 experts on
    average at batch 1 / 2 / 4 / 8 / 16 / 24 (the figures the benchmark and
    its roofline bytes quote)."""
    s = synth.PREFILL
    idx, _ = oracle.route(synth.make_logits(s.T, s.E, seed=0, zipf_s=synth.ZIPF_S).numpy(), s.k)
    c = np.bincount(idx.reshape(-1), minlength=s.E)
    fat, thin = c >= 32, (c > 0) & (c < 32)
    assert (c > 0).sum() == 233 and fat.sum() == 81 and thin.sum() == 152
    assert c[fat].sum() == 130162 and c[thin].sum() == 910
    expect = {1: 8.0, 2: 12.1875, 4: 17.625, 8: 24.625, 16: 32.8125, 24: 38.5}
    for B in synth.DECODE_SWEEP_BATCHES:
        touched = [len(np.unique(oracle.route(
            synth.make_logits(B, s.E, seed=0, layer=l, rep=r, zipf_s=synth.ZIPF_S).numpy(),
            s.k)[0])) for l in range(4) for r in range(4)]
        assert np.mean(touched) == expect[B], B
