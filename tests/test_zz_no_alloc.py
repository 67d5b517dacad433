"""moe_permute_noalloc: the route-list entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside libmoe).

Checked through the C ABI against moe_permute, bit-exact, on two calls in a
row with different inputs -- the shared array keeps the previous call's
contents, so a stale byte would show -- on both the single-block and the
multi-chunk kernels.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routed_expert_ffn_02_gb300 as m
    return m


def _outs(T, E, k):
    P = T * k
    return (torch.empty(E, dtype=torch.int32, device="cuda"),
            torch.empty(E + 1, dtype=torch.int32, device="cuda"),
            torch.empty(max(P, 1), dtype=torch.int32, device="cuda")[:P],
            torch.empty(max(P, 1), dtype=torch.int32, device="cuda")[:P])


def _call_noalloc(moe, idx, E, out, status):
    lib = moe.binding.raw_lib()
    T, k = idx.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.moe_permute_noalloc(p(idx), T, E, k, p(out[0]), p(out[1]), p(out[2]), p(out[3]),
                                 p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.moe_last_error()


@pytest.mark.parametrize("T,E,k", [(4, 384, 8), (16384, 384, 8), (3000, 1024, 3),
                                   (32768, 1024, 8)])   # the last fills the array
def test_noalloc_matches_moe_permute_twice(moe, T, E, k):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        lg = synth.make_logits(T, E, seed=50 + call, zipf_s=synth.ZIPF_S).cuda()
        idx, _ = moe.moe_route(lg, k)
        ref = moe.moe_permute(idx, E)
        got = _outs(T, E, k)
        _call_noalloc(moe, idx, E, got, status)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert status.item() == 0


def test_noalloc_reports_bad_index_then_recovers(moe):
    T, E, k = 5000, 16, 2
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx = torch.randint(0, E, (T, k), dtype=torch.int32, device="cuda")
    bad = idx.clone()
    bad[7, 1] = E
    _call_noalloc(moe, bad, E, _outs(T, E, k), status)
    torch.cuda.synchronize()
    assert status.item() == 6          # MOE_ERR_BAD_INDEX
    got = _outs(T, E, k)
    _call_noalloc(moe, idx, E, got, status)
    torch.cuda.synchronize()
    assert status.item() == 0          # the status is cleared by each call
    for a, b in zip(got, moe.moe_permute(idx, E)):
        assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    lib = moe.binding.raw_lib()
    st = lib.moe_permute_noalloc(None, 262144 // 8 + 1, 384, 8, None, None, None, None, None,
                                 None)
    assert st == 2 and b"262144" in lib.moe_last_error()


def test_noalloc_shape_changes_between_calls(moe):
    """A call over the whole array (128 chunks of 2048 slots, E = 1024) and
    then smaller multi-chunk calls with other E and chunk counts: each result
    is bit-exact, so nothing of the previous call's histograms leaks in."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for i, (T, E, k) in enumerate([(32768, 1024, 8), (5000, 48, 4), (20000, 700, 6),
                                   (1, 1, 1), (9000, 1024, 2)]):
        lg = synth.make_logits(T, E, seed=70 + i, zipf_s=synth.ZIPF_S).cuda()
        idx, _ = moe.moe_route(lg, k)
        ref = moe.moe_permute(idx, E)
        got = _outs(T, E, k)
        _call_noalloc(moe, idx, E, got, status)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), (T, E, k)
        assert status.item() == 0
