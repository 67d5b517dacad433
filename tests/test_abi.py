"""C ABI checks that need no GPU: the library loads, exports every function
include/moe.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_ffn_02_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s+(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_functions():
    names = declared_functions()
    assert "moe_forward" in names and "moe_route" in names and len(names) >= 12


def test_library_exports_every_declared_function(moe):
    lib = moe.binding.raw_lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(moe.EXPORTED) == declared_functions()


def test_version(moe):
    assert "sm_103a" in moe.version()


def test_workspace_sizes(moe):
    s = moe.Shape(16384, 384, 8, 4096, 2048)
    n = moe.workspace_size(s)
    P = s.P
    # sorted activations (reused for the sorted outputs) and the intermediate dominate
    assert P * (4096 + 2048) * 2 < n < P * (4096 + 2048) * 2 + 64 * 2 ** 20
    assert moe.expert_ffn_workspace_size(s) < n
    assert moe.permute_workspace_size(16384, 384, 8) >= 256
    small = moe.workspace_size(moe.Shape(1, 384, 8, 4096, 2048))
    assert small < 4 * 2 ** 20


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(E=0), dict(E=1025), dict(k=0), dict(k=9), dict(E=4, k=5),
    dict(H=100), dict(H=0), dict(I=128), dict(fat_threshold=-1), dict(fat_threshold=34),
    dict(thin_mma_min=-1), dict(thin_mma_min=34),
])
def test_bad_shapes_rejected(moe, bad):
    base = dict(T=16, E=16, k=2, H=512, I=256, fat_threshold=32)
    base.update(bad)
    shape = moe.binding.MoeShape(**base)
    lib = moe.binding.raw_lib()
    assert lib.moe_workspace_size(ctypes.byref(shape)) == 0
    st = lib.moe_forward(ctypes.byref(shape), None, None, None, None, None, None, None, None,
                         None, 0, None)
    assert st == 1
    assert lib.moe_last_error()


def test_hidden_size_limit(moe):
    lib = moe.binding.raw_lib()
    shape = moe.binding.MoeShape(16, 16, 2, 16640, 256, 32)
    assert lib.moe_workspace_size(ctypes.byref(shape)) == 0
    st = lib.moe_forward(ctypes.byref(shape), None, None, None, None, None, None, None, None,
                         None, 0, None)
    assert st == 2


def test_route_argument_errors(moe):
    lib = moe.binding.raw_lib()
    assert lib.moe_route(None, 4, 3, 4, None, None, None) == 1       # k > E
    assert lib.moe_route(None, 4, 3, 2, None, None, None) == 1       # NULL logits
    assert lib.moe_route(None, 0, 3, 2, None, None, None) == 0       # T == 0: no-op
    assert lib.moe_permute_workspace_size(4, 3, 9) == 0


def test_pointer_and_workspace_errors(moe):
    lib = moe.binding.raw_lib()
    shape = moe.binding.MoeShape(16, 16, 2, 512, 256, 32)
    good = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)   # 8-byte aligned only
    # misaligned activation pointer
    st = lib.moe_forward(ctypes.byref(shape), good, odd, good, good, good, good, None, None,
                         good, 1 << 30, None)
    assert st == 1 and b"aligned" in lib.moe_last_error()
    # missing / small / misaligned workspace
    st = lib.moe_forward(ctypes.byref(shape), good, good, good, good, good, good, None, None,
                         None, 0, None)
    assert st == 3
    st = lib.moe_forward(ctypes.byref(shape), good, good, good, good, good, good, None, None,
                         good, 100, None)
    assert st == 3
    st = lib.moe_forward(ctypes.byref(shape), good, good, good, good, good, good, None, None,
                         ctypes.c_void_p(0x10010), 1 << 30, None)
    assert st == 3
    st = lib.moe_permute(good, 16, 16, 2, good, good, good, good, None, 0, None)
    assert st == 3
    assert lib.moe_combine(good, good, good, 4, 9, 512, good, None) == 1
    assert lib.moe_combine(good, good, good, 4, 2, 12, good, None) == 1


def test_product_path_does_not_import_oracle():
    """The library package and its binding never reference the oracle."""
    pkg = os.path.join(ROOT, "routed_expert_ffn_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "moe_oracle" not in src, f


def test_stager_argument_errors(moe):
    lib = moe.binding.raw_lib()
    shape = moe.binding.MoeShape(16, 16, 2, 512, 256, 32)
    assert lib.moe_layer_weight_bytes(ctypes.byref(shape)) == 3 * 16 * 512 * 256 * 2
    h = ctypes.c_void_p()
    assert lib.moe_stager_create(None, 2, 1 << 20, ctypes.byref(h)) == 1
    assert lib.moe_stager_create(ctypes.c_void_p(0x10000), 0, 1 << 20, ctypes.byref(h)) == 1
    assert lib.moe_stager_create(ctypes.c_void_p(0x10010), 2, 1 << 20, ctypes.byref(h)) == 1
    assert lib.moe_forward_offload(None, ctypes.byref(shape), 1, None, None, None, None, None, 0,
                                   None, None) == 1


def test_forward_launch_count(moe):
    """Kernels one moe_forward launches: route, route lists (1 or 3), then
    only the expert kernels that can have work, then combine (fused into the
    tensor-core down kernel when that is the only expert kernel).  Small batches
    on one streaming kernel route inside it and combine in the down kernel:
    gate/up, down; on the CUDA-core kernel at H=4096, I=2048, H=2048,
    I=1024 or H=512, I=256, one cooperative launch for the whole layer."""
    S = moe.Shape
    # decode: 8 or 16 touched experts x 16 blocks < 384 items -> CUDA cores,
    # from 24 x 16 = 384 on tensor cores; up to 32 slots the batch is routed
    # inside the streaming kernels either way
    assert moe.forward_launches(S(1, 384, 8, 4096, 2048)) == 1
    assert moe.forward_launches(S(2, 384, 8, 4096, 2048)) == 1
    assert moe.forward_launches(S(3, 384, 8, 4096, 2048)) == 2
    assert moe.forward_launches(S(4, 384, 8, 4096, 2048)) == 2
    assert moe.forward_launches(S(1, 384, 8, 4096, 2048, thin_mma_min=1)) == 2
    assert moe.forward_launches(S(4, 384, 8, 4096, 2048, thin_mma_min=33)) == 1
    assert moe.forward_launches(S(2, 384, 8, 2048, 1024)) == 1
    assert moe.forward_launches(S(2, 384, 8, 1024, 512)) == 2     # no one-launch build
    assert moe.forward_launches(S(4, 384, 8, 4096, 2048, thin_mma_min=3)) == 8   # split kernels
    for B in (5, 8, 16, 24):                                 # decode sweep: > 32 slots
        assert moe.forward_launches(S(B, 384, 8, 4096, 2048)) == 5
    assert moe.forward_launches(S(32, 64, 8, 512, 256, 33, 1)) == 5   # 256 slots
    assert moe.forward_launches(S(32, 64, 8, 512, 256, 32, 1)) == 11  # T = 32 may be fat
    # CUDA-core self-routing limits: 32 slots, below the fat threshold, one
    # unit per expert
    assert moe.forward_launches(S(5, 384, 8, 4096, 2048, thin_mma_min=33)) == 5   # 40 slots
    assert moe.forward_launches(S(32, 64, 1, 512, 256, thin_mma_min=33)) == 11    # T = 32 may be fat
    assert moe.forward_launches(S(16, 64, 2, 512, 256, thin_mma_min=33)) == 1     # unit of 16
    assert moe.forward_launches(S(13, 64, 2, 4096, 2048, thin_mma_min=33)) == 5   # units of 12
    assert moe.forward_launches(S(2, 64, 2, 512, 256, fat_threshold=0)) == 9     # every expert fat
    # fat experts: pair GEMMs (gate/up in two launches) and solo-tile GEMMs
    assert moe.forward_launches(S(16384, 384, 8, 4096, 2048)) == 13
    assert moe.forward_launches(S(16384, 384, 8, 4096, 2048, thin_mma_min=8)) == 15
    assert moe.forward_launches(S(16384, 384, 8, 4096, 2048, fat_threshold=0)) == 11
    assert moe.forward_launches(S(0, 384, 8, 4096, 2048)) == 0


def test_pipe_argument_errors(moe):
    """moe_forward_host rejects a NULL pipe, equal streams and a small
    workspace before touching the GPU; the pipe workspace adds two staging
    slots to the forward workspace."""
    lib = moe.binding.raw_lib()
    shape = moe.binding.MoeShape(16, 16, 2, 512, 256, 32)
    fwd = lib.moe_workspace_size(ctypes.byref(shape))
    slot = 16 * 512 * 2 + 16 * 16 * 4 + 16 * 512 * 2   # x, logits, out (each 256-aligned here)
    assert lib.moe_pipe_workspace_size(ctypes.byref(shape)) == fwd + 2 * slot
    bad = moe.binding.MoeShape(16, 16, 2, 100, 256, 32)
    assert lib.moe_pipe_workspace_size(ctypes.byref(bad)) == 0
    s1, s2, s3 = ctypes.c_void_p(1), ctypes.c_void_p(2), ctypes.c_void_p(3)
    args = [None] * 7 + [0]          # logits, x, 3 weights, out, ws, ws_bytes
    assert lib.moe_forward_host(None, ctypes.byref(shape), *args, s1, s2, s3) == 1
    fake = ctypes.c_void_p(8)   # never dereferenced: the stream check comes first
    assert lib.moe_forward_host(fake, ctypes.byref(shape), *args, s1, s1, s3) == 1
    assert b"different streams" in lib.moe_last_error()
    assert lib.moe_forward_host(fake, ctypes.byref(bad), *args, s1, s2, s3) == 1
    assert lib.moe_pipe_create(None) == 1


def test_cache_argument_errors(moe):
    """moe_cache_bytes sizing and argument checks made before any CUDA call."""
    lib = moe.binding.raw_lib()
    shape = moe.binding.MoeShape(16, 32, 4, 512, 256, 32)
    per_expert = 512 * 256 * 2
    tables = (3 * 32 * 4 + 255) // 256 * 256
    assert lib.moe_cache_bytes(ctypes.byref(shape), 10, 3) == 3 * 10 * per_expert + tables
    assert lib.moe_cache_bytes(ctypes.byref(shape), 0, 3) == 0
    assert lib.moe_cache_bytes(ctypes.byref(shape), 10, 0) == 0
    out = ctypes.c_void_p()
    assert lib.moe_cache_create(ctypes.byref(shape), 10, 3, None, 0, ctypes.byref(out)) == 1
    assert lib.moe_cache_create(ctypes.byref(shape), 10, 3, ctypes.c_void_p(256), 16,
                                ctypes.byref(out)) == 1     # below moe_cache_bytes
    assert lib.moe_forward_cached(None, ctypes.byref(shape), 0, None, None, None, None, None,
                                  None, 0, None, None) == 1
    h, m = ctypes.c_int64(), ctypes.c_int64()
    assert lib.moe_cache_stats(None, ctypes.byref(h), ctypes.byref(m)) == 1
