"""CPU: the benchmark's algorithmic work per stage and its roofline
arithmetic, against values worked out by hand from the formulas (bytes and
flops per stage as the kernel table states them)."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
bench = pytest.importorskip("bench")


class _Shape:
    def __init__(self, T, E, k, H, I, fat_threshold, thin_mma_min):
        self.T, self.E, self.k, self.H, self.I = T, E, k, H, I
        self.fat_threshold, self.thin_mma_min = fat_threshold, thin_mma_min


def test_stage_work_by_hand():
    # T=4 tokens, top-2: 8 slots over 8 experts; threshold 3 makes expert 0
    # (3 slots) fat, experts 1, 3, 4 (2, 1, 2 slots) thin; thin_mma_min 2 puts
    # experts 1 and 4 on the tensor-core kernel (their rows are gathered).
    sh = _Shape(T=4, E=8, k=2, H=256, I=128, fat_threshold=3, thin_mma_min=2)
    counts = np.array([3, 2, 0, 1, 2, 0, 0, 0])
    w = bench.stage_work(sh, counts)
    H, I = 256, 128
    assert w["route"]["bytes"] == 4 * 8 * 4 + 8 * 8
    assert w["permute"]["bytes"] == 8 * 16 + 8 * 8
    # no pair tiles (expert 0 is a single-tile solo expert): the gather
    # kernel copies nothing, the gate/up GEMM's first launch copies all 7 rows
    assert w["gather"]["bytes"] == 0
    assert w["gemm_gate_up"]["flops"] == 2 * 3 * H * 2 * I
    assert w["gemm_gate_up"]["bytes"] == (1 * (2 * I * H * 2) + 3 * (H + I) * 2
                                          + (3 + 4) * H * 4)
    assert w["gemm_down"]["flops"] == 2 * 3 * I * H
    assert w["gemm_down"]["bytes"] == 1 * (H * I * 2) + 3 * (H + I) * 2
    assert w["thin_gate_up"]["bytes"] == 3 * (2 * I * H * 2) + 5 * (H + I) * 2
    assert w["thin_down"]["bytes"] == 3 * (H * I * 2) + 5 * (H + I) * 2
    assert w["combine"]["bytes"] == 8 * H * 2 + 4 * H * 2 + 8 * 8
    assert w["_info"] == dict(fat_experts=1, thin_experts=3, fat_rows=3, thin_rows=5,
                              touched=4)


def test_stage_work_gather_parts():
    # Experts 0 and 1 are fat with 600 and 300 slots: pair tiles of 256 rows
    # (expert 0: 256, 256, 88; expert 1: 256, 44), five pairs; the gather
    # kernel copies the first ceil(5 / 3) = 2 pairs' rows (512), the first
    # gate/up GEMM launch the other 388 rows and expert 2's 100 (a solo tile).
    sh = _Shape(T=1000, E=4, k=1, H=256, I=128, fat_threshold=32, thin_mma_min=0)
    counts = np.array([600, 300, 100, 0])
    w = bench.stage_work(sh, counts)
    H, I = 256, 128
    assert w["gather"]["bytes"] == 512 * H * 4
    assert w["gemm_gate_up"]["bytes"] == (3 * (2 * I * H * 2) + 1000 * (H + I) * 2
                                          + (1000 - 512) * H * 4)


def test_stage_work_self_routed_batch_has_no_gather():
    # 4 tokens, top-8 over 384 experts, H=4096, I=2048: 32 slots, all thin,
    # on the tensor-core kernel by the shape rule, routed inside the kernels.
    sh = _Shape(T=4, E=384, k=8, H=4096, I=2048, fat_threshold=32, thin_mma_min=0)
    counts = np.zeros(384, dtype=np.int64)
    counts[:16] = 2
    w = bench.stage_work(sh, counts)
    assert w["gather"]["bytes"] == 0
    assert w["thin_gate_up"]["bytes"] == 16 * (2 * 2048 * 4096 * 2) + 32 * (4096 + 2048) * 2


def test_roofline_arithmetic():
    peaks = dict(hbm_gbs=6787.2, bf16_tflops=1919.3, bf16_tflops_sustained=1712.5,
                 source="measured")
    work = {"gemm_gate_up": dict(flops=1919.3e9, bytes=0),
            "combine": dict(bytes=6787.2e6, flops=0)}
    r = bench.roofline_for("gemm_gate_up", work, 1.0, peaks)    # 1 ms
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1919.3, rel=1e-4) and r["frac"] == pytest.approx(1.0)
    r = bench.roofline_for("combine", work, 2.0, peaks)         # 2 ms: half the peak
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(3393.6, rel=1e-4) and r["frac"] == pytest.approx(0.5)


def test_clock_sampler_window_and_reasons():
    """The clock summary takes the median SM clock of the samples inside the
    marked window, the throttle reasons active there, and the whole run's
    minimum beside them (synthetic nvidia-smi lines; no subprocess)."""
    clk = bench.ClockSampler(0)
    line = "{sm}, 2070, 900.5, {hw}, Not Active, Not Active, {pc}"
    clk.samples = [
        (0.0, line.format(sm=1500, hw="Not Active", pc="Active")),      # before the window
        (1.0, line.format(sm=2070, hw="Not Active", pc="Not Active")),
        (1.1, line.format(sm=2040, hw="Not Active", pc="Active")),
        (1.2, line.format(sm=2070, hw="Not Active", pc="Not Active")),
        (3.0, line.format(sm=1200, hw="Active", pc="Not Active")),      # after it
        (3.1, "garbled"),
    ]
    clk.mark(0.9, 1.3)
    s = clk.summary()
    assert s["sm_mhz"] == 2070.0 and s["samples"] == 3 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["run"]["sm_mhz_min"] == 1200.0 and s["run"]["samples"] == 5
    assert s["run"]["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unsampled"]
