#!/usr/bin/env python
"""Benchmark of the routed MoE FFN layer on GB300.

Headline workload: one MoE layer over a 16,384-token prefill chunk (384
experts, top-8, H=4096, I=2048, bf16, Zipf(1.1)-skewed router logits, fat
threshold 32).  A step is one moe_forward: route, route lists, both expert
paths and the combine.  Reported beside it: decode batches 1 and 4 on the
same layer, the decode batch sweep 1..24 over 4 resident layers, and (unless
--no-offload) the 12-layer prefill streamed from pinned host memory with the
host link's own copy bandwidth beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line.  --impl reference times the CPU oracle on a bounded
token sample of the same workload on the host cores.  Under torchrun
(N > 1) every rank runs its own replica of the layer (no data exchange).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "routed MoE-layer tokens/s (16k prefill chunk; decode batch 1-24) + % roofline"
PREFILL = synth.PREFILL
FAT_THRESHOLD = 32
L2_BYTES = 129 * 2 ** 20


def measured_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from a committed ncu capture under
    profiles/, or None if there is none or the kernel's sources changed since."""
    import glob
    import hashlib
    for path in glob.glob(os.path.join(ROOT, "profiles", "traffic_*.json")):
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel") != kernel:
            continue
        h = hashlib.sha256()
        for src in rec["source_files"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] == rec["source_sha256_16"]:
            return rec["bytes_per_launch"]
    return None


def receipts(moe, layer):
    """sha256 (first 16 hex digits) of the library that ran and of the step's
    inputs, so a result can be matched to the exact build and data."""
    import hashlib
    with open(moe.LIB_PATH, "rb") as f:
        lib = hashlib.sha256(f.read()).hexdigest()[:16]
    h = hashlib.sha256()
    h.update(layer.x_cpu.view(torch.int16).numpy().tobytes())
    h.update(layer.logits_cpu[0].numpy().tobytes())
    return {"libmoe_sha256_16": lib, "inputs_sha256_16": h.hexdigest()[:16]}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 20 ms while
    running; each sample carries its host time so a timed window can be
    picked out (mark() brackets it)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []          # (host time, line)
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t_end = time.monotonic() + 5.0          # sampling is live before timing
            while not self.samples and time.monotonic() < t_end:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The timed window, in time.monotonic() seconds."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _parse(self, lines):
        sm, mx, reasons = [], [], set()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return sm, mx, reasons

    def summary(self):
        lines = [l for _, l in self.samples]
        if self.window:
            t0, t1 = self.window
            inside = [l for t, l in self.samples if t0 <= t <= t1]
        else:
            inside = lines
        sm, mx, reasons = self._parse(inside)
        all_sm, all_mx, all_reasons = self._parse(lines)
        if not all_sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else max(all_mx),
               "reasons": sorted(reasons), "samples": len(sm),
               "run": {"sm_mhz_median": statistics.median(all_sm), "sm_mhz_min": min(all_sm),
                       "reasons": sorted(all_reasons), "samples": len(all_sm)}}
        return out


# --------------------------------------------------------------- workload

def stage_work(shape, counts_np):
    """Algorithmic flops and bytes per stage for one step (used for rooflines).
    Fat experts: counts >= threshold; thin: 0 < counts < threshold."""
    T, E, k, H, I = shape.T, shape.E, shape.k, shape.H, shape.I
    P = T * k
    thr = shape.fat_threshold
    fat = counts_np >= max(thr, 1)
    thin = (counts_np > 0) & (counts_np < thr)
    fat_rows = int(counts_np[fat].sum())
    thin_rows = int(counts_np[thin].sum())
    # x_sorted holds the rows of fat experts and of thin experts on the
    # tensor-core streaming kernel (the library's rule when thin_mma_min is 0)
    mma_min = shape.thin_mma_min or (1 if min(E, P) * (I // 128) >= 384 else 33)
    mma_rows = int(counts_np[thin & (counts_np >= mma_min)].sum())
    # batches of <= 32 slots below the fat threshold on the tensor-core kernel
    # route themselves and load x rows directly: no gather
    if P <= 32 and T < thr and mma_min <= 1:
        mma_rows = 0
    n_fat, n_thin = int(fat.sum()), int(thin.sum())
    w_gu = 2 * I * H * 2      # gate + up bytes per expert
    w_d = H * I * 2
    # With fat experts the gather kernel copies the rows of the first third of
    # the pair tiles (256-row tiles of experts with more than one 128-row
    # tile, in expert order); the gate/up GEMM's first launch copies the rest.
    pair_rows = []
    for c in counts_np:
        c = int(c)
        if c >= max(thr, 1) and c > 128:
            pair_rows += [min(256, c - 256 * q) for q in range((c + 255) // 256)]
    gathered = fat_rows + mma_rows
    first = sum(pair_rows[:(len(pair_rows) + 2) // 3]) if n_fat else gathered
    return {
        "route": dict(bytes=T * E * 4 + P * 8, flops=0),
        "permute": dict(bytes=P * 4 * 4 + E * 8, flops=0),
        "gather": dict(bytes=first * H * 2 * 2, flops=0),
        "gemm_gate_up": dict(flops=2 * fat_rows * H * 2 * I,
                             bytes=n_fat * w_gu + fat_rows * (H + I) * 2
                             + (gathered - first) * H * 2 * 2),
        "thin_gate_up": dict(bytes=n_thin * w_gu + thin_rows * (H + I) * 2,
                             flops=2 * thin_rows * H * 2 * I),
        "gemm_down": dict(flops=2 * fat_rows * I * H,
                          bytes=n_fat * w_d + fat_rows * (H + I) * 2),
        "thin_down": dict(bytes=n_thin * w_d + thin_rows * (H + I) * 2,
                          flops=2 * thin_rows * I * H),
        "combine": dict(bytes=P * H * 2 + T * H * 2 + P * 8, flops=0),
        "_info": dict(fat_experts=n_fat, thin_experts=n_thin, fat_rows=fat_rows,
                      thin_rows=thin_rows, touched=int((counts_np > 0).sum())),
    }


# Nominal GB300 figures (dense bf16 tensor rate, HBM3e bandwidth): the
# targets are stated against these, so every fraction of the measured peaks
# is reported beside its fraction of the nominal ones.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0


def roofline_for(stage, work, ms, peaks):
    w = work[stage]
    if stage.startswith("gemm"):
        # The timed loop is short (well under a second, SM clock at its
        # maximum), so the burst figure is the comparable peak.
        ach = w["flops"] / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "peak_note": f"bf16 dense burst (cuBLAS), {peaks['source']}",
                "frac_nominal": round(ach / NOMINAL_BF16_TFLOPS, 4)}
    ach = w["bytes"] / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(ach / peak, 4), "peak_note": f"HBM copy, {peaks['source']}",
            "frac_nominal": round(ach / NOMINAL_HBM_GBS, 4)}


class Layer:
    def __init__(self, moe, shape, device, n_logit_sets=1, zipf=synth.ZIPF_S, weights=None):
        self.moe = moe
        self.shape = shape
        self.device = device
        if weights is None:
            weights = synth.make_weights(shape.E, shape.H, shape.I, seed=0, layer=0,
                                         device=device)
        self.Wg, self.Wu, self.Wd = weights
        self.x_cpu = synth.make_x(shape.T, shape.H, seed=0)
        self.logits_cpu = [synth.make_logits(shape.T, shape.E, seed=0, rep=r, zipf_s=zipf)
                           for r in range(n_logit_sets)]
        self.x = self.x_cpu.to(device)
        self.logits = [l.to(device) for l in self.logits_cpu]
        self.out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((shape.T, shape.k), dtype=torch.int32, device=device)
        self.gates = torch.empty((shape.T, shape.k), dtype=torch.float32, device=device)
        self.ws = moe.Workspace(moe.workspace_size(shape), device)

    def forward(self, i=0, events=None, logits=None, x=None, out=None):
        lg = logits if logits is not None else self.logits[i % len(self.logits)]
        args = (self.shape, lg, x if x is not None else self.x, self.Wg, self.Wu, self.Wd)
        kw = dict(out=out if out is not None else self.out, topk_idx=self.idx,
                  gates=self.gates, ws=self.ws)
        if events is not None:
            return self.moe.moe_forward_profiled(*args, events, **kw)
        return self.moe.moe_forward(*args, **kw)

    def counts(self, i=0):
        self.forward(i)
        c, _, _, _ = self.moe.moe_permute(self.idx, self.shape.E)
        torch.cuda.synchronize()
        return c.cpu().numpy()


def time_steps(layer, steps, warmup, profiled=True, rotate=True, clk=None):
    moe = layer.moe
    for i in range(warmup):
        layer.forward(i)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.PROFILE_EVENTS)]
          for _ in range(steps)] if profiled else None
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    t0 = time.monotonic()
    start.record()
    for i in range(steps):
        layer.forward(i if rotate else 0, events=ev[i] if profiled else None)
    end.record()
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    if clk is not None:
        clk.mark(t0, t1)
    total_ms = start.elapsed_time(end)
    stage_ms = None
    if profiled:
        stage_ms = {}
        for j, name in enumerate(moe.PROFILE_STAGES):
            stage_ms[name] = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev)
    return total_ms, stage_ms


def time_graph_steps(layer, steps, warmup, n_graphs=8, clk=None):
    """Times `steps` decode steps replayed through the library's DecodeGraph
    (one captured step per logits set, its static inputs filled once);
    returns total ms.  clk: a running ClockSampler, told the timed window."""
    moe = layer.moe
    graphs = []
    for i in range(n_graphs):
        g = moe.DecodeGraph(layer.shape, layer.Wg, layer.Wu, layer.Wd)
        g.logits.copy_(layer.logits[i % len(layer.logits)])
        g.x.copy_(layer.x)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(warmup):
        graphs[i % n_graphs].replay()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    t0 = time.monotonic()
    start.record()
    for i in range(steps):
        graphs[i % n_graphs].replay()
    end.record()
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark(t0, time.monotonic())
    barrier()
    for g in graphs:
        assert g.ws.status() == 0
    return start.elapsed_time(end)


# -------------------------------------------------------- distributed glue

_DIST = {"on": False}


def init_dist():
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        _DIST["on"] = True
        return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def barrier():
    if _DIST["on"]:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float) -> float:
    if not _DIST["on"]:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------- CPU oracle legs

def oracle_sample(n_tokens, expert_source, logits_np, x_bits, k, seed=123):
    """Times the oracle on n_tokens sampled tokens of the workload.
    expert_source(e) -> bf16 bit arrays of expert e (fetched before timing)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(logits_np.shape[0], size=n_tokens, replace=False))
    idx, _ = oracle.route(logits_np[toks], k)
    need = sorted(set(idx.reshape(-1).tolist()))
    weights = {e: expert_source(e) for e in need}
    t0 = time.perf_counter()
    oracle.moe_tokens(x_bits[toks], logits_np[toks], k, weights.__getitem__)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt, len(need)


def prefill_config(T, E, info, thin_mma_min, world):
    """The bench line's config (both arms print the same one)."""
    return {
        "workload": f"prefill chunk: 1 MoE layer, T={T} tokens, E={E} experts, top-8, "
                    "H=4096, I=2048, bf16, Zipf(1.1) router bias, fat threshold 32",
        "parallelism": "replicas only" if world > 1 else "single GPU",
        "l2": f"inputs larger than L2 ({E * 3 * 4096 * 2048 * 2 / 1e9:.1f} GB of expert "
              "weights per layer)",
        "fat_experts": info["fat_experts"],
        "thin_experts": info["thin_experts"],
        "touched_experts": info["touched"],
        "thin_mma_min": thin_mma_min or "default",
    }


def run_reference(args):
    """--impl reference: the oracle as it stands, on the host cores, each step
    a bounded token sample of the prefill workload."""
    rank, world, _ = init_dist()
    if rank != 0:
        return
    shape = PREFILL
    x_bits = synth.bf16_bits(synth.make_x(shape.T, shape.H, seed=0))
    logits_np = synth.make_logits(shape.T, shape.E, seed=0, zipf_s=synth.ZIPF_S).numpy()
    tokens_per_step = 2
    cache = {}

    def expert(e):
        if e not in cache:
            cache[e] = tuple(synth.bf16_bits(w) for w in synth.make_expert(e, shape.H, shape.I))
        return cache[e]

    # the workload's expert mix, as the GPU arm's config states it
    import oracle
    oracle.build()
    idx, _ = oracle.route(logits_np, shape.k)
    counts = np.bincount(idx.reshape(-1), minlength=shape.E)
    fat, thin = counts >= FAT_THRESHOLD, (counts > 0) & (counts < FAT_THRESHOLD)
    info = dict(fat_experts=int(fat.sum()), thin_experts=int(thin.sum()),
                touched=int((counts > 0).sum()))
    times = []
    for i in range(args.warmup + args.steps):
        tps, dt, _ = oracle_sample(tokens_per_step, expert, logits_np, x_bits, shape.k, seed=i)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = tokens_per_step * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(shape.T, shape.E, info, 0, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1,
                         "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{tokens_per_step} tokens per step of the 16,384-token "
                                   "chunk, all of their 8 experts each, single-threaded fp64"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------- decode sweep

def run_sweep(moe, dev, base_weights, peaks, thin_mma_min=0, reps=40, warmup=5, n_layers=4,
              n_sets=4):
    """Decode batches 1..24 through 4 resident MoE layers (384 experts,
    H=4096, I=2048, bf16; 77 GB of weights so L2 cannot hold them).  A step is
    one batch through all 4 layers, replayed from a CUDA graph; n_sets logit
    sets rotate so the touched experts change from step to step."""
    E, H, I, k = PREFILL.E, PREFILL.H, PREFILL.I, PREFILL.k
    layers = [base_weights] + [synth.make_weights(E, H, I, seed=0, layer=l, device=dev)
                               for l in range(1, n_layers)]
    expert_bytes = 3 * H * I * 2
    out = {}
    for B in synth.DECODE_SWEEP_BATCHES:
        shape = moe.Shape(B, E, k, H, I, FAT_THRESHOLD, thin_mma_min)
        ws = moe.Workspace(moe.workspace_size(shape), dev)
        x = synth.make_x(B, H, seed=0).to(dev)
        lg = [[synth.make_logits(B, E, seed=0, layer=l, rep=r, zipf_s=synth.ZIPF_S).to(dev)
               for l in range(n_layers)] for r in range(n_sets)]
        outs = [torch.empty((B, H), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
        touched = []
        for r in range(n_sets):
            for l in range(n_layers):
                idx, _ = moe.moe_route(lg[r][l], k)
                touched.append(int(torch.unique(idx).numel()))
        stream = torch.cuda.Stream()
        graphs = []
        with torch.cuda.stream(stream):
            for r in range(n_sets):
                for l in range(n_layers):
                    moe.moe_forward(shape, lg[r][l], x, *layers[l], out=outs[l], ws=ws)
            torch.cuda.synchronize()
            for r in range(n_sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for l in range(n_layers):
                        moe.moe_forward(shape, lg[r][l], x, *layers[l], out=outs[l], ws=ws)
                graphs.append(g)
        for i in range(warmup):
            graphs[i % n_sets].replay()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record()
        for i in range(reps):
            graphs[i % n_sets].replay()
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / reps
        bytes_step = sum(touched) / n_sets * expert_bytes
        out[f"B{B}"] = {
            "tokens_per_s": round(B / (ms * 1e-3), 1),
            "us_per_step": round(1e3 * ms, 2),
            "touched_experts_per_layer": round(sum(touched) / len(touched), 2),
            "frac_of_hbm_roofline": round(bytes_step / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "frac_of_nominal_hbm": round(bytes_step / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        }
        del graphs, ws
    del layers[1:]
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------- offload

def measure_h2d_link(dev, nbytes=1 << 31, reps=5):
    """Host-to-device copy bandwidth of this box's link (GB/s): one copy of
    nbytes from pinned host memory, best of reps, CUDA events on a side
    stream (what the stager's copies can reach at most)."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    src.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    best = float("inf")
    with torch.cuda.stream(st):
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            dst.copy_(src, non_blocking=True)
            b.record(st)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
    del src, dst
    return nbytes / (best * 1e-3) / 1e9


def run_offload(args, moe, dev, n_layers=12, n_slots=8):
    """Offload prefill: 12 layers x 384 experts (H=2048, I=1024, bf16, 58 GB)
    in pinned host memory, streamed through 8 HBM staging slots on a side copy
    stream while the layers run on a 16,384-token chunk.  A step is the whole
    chunk through all 12 layers."""
    s = synth.OFFLOAD
    shape = moe.Shape(s.T, s.E, s.k, s.H, s.I, FAT_THRESHOLD, args.thin_mma_min)
    host = []
    for l in range(n_layers):
        W = synth.make_weights(s.E, s.H, s.I, seed=0, layer=l, device=dev)
        host.append(moe.pack_layer_weights(*W))
        del W
    torch.cuda.empty_cache()
    x = synth.make_x(s.T, s.H, seed=0).to(dev)
    logits = [synth.make_logits(s.T, s.E, seed=0, layer=l, zipf_s=synth.ZIPF_S).to(dev)
              for l in range(n_layers)]
    outs = [torch.empty((s.T, s.H), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    st = moe.Stager(shape, n_slots, dev)
    ws = moe.Workspace(moe.workspace_size(shape), dev)
    copy = torch.cuda.Stream(device=dev)
    compute = torch.cuda.current_stream()
    steps = max(1, min(args.steps, 5))
    for _ in range(max(1, min(args.warmup, 2))):
        st.forward(shape, logits, x, host, outs, ws, compute, copy)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        st.forward(shape, logits, x, host, outs, ws, compute, copy)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    # compute alone on resident copies of two layers, for the overlap check
    W0 = synth.make_weights(s.E, s.H, s.I, seed=0, layer=0, device=dev)
    for _ in range(3):
        moe.moe_forward(shape, logits[0], x, *W0, out=outs[0], ws=ws)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(5):
        moe.moe_forward(shape, logits[0], x, *W0, out=outs[0], ws=ws)
    c1.record()
    torch.cuda.synchronize()
    layer_ms = c0.elapsed_time(c1) / 5
    st.close()
    del st
    torch.cuda.empty_cache()
    cached = run_offload_decode_cache(moe, dev, host, s, n_layers)
    # the stager copies only the experts each layer's tokens are routed to
    touched = []
    for l in range(n_layers):
        idx, _ = moe.moe_route(logits[l], s.k)
        touched.append(int(torch.unique(idx).numel()))
    per_expert = moe.layer_weight_bytes(shape) // s.E
    copied = sum(touched) * per_expert
    link = measure_h2d_link(dev)
    h2d = copied / (ms * 1e-3) / 1e9
    return {
        "workload": "12 MoE layers x 384 experts, H=2048, I=1024, bf16 (58 GB pinned host), "
                    "8 HBM staging slots, T=16384, top-8, Zipf(1.1)",
        "tokens_per_s": round(s.T / (ms * 1e-3), 1),
        "ms_per_chunk": round(ms, 3),
        "touched_experts_per_layer": round(sum(touched) / n_layers, 1),
        "h2d_bytes_per_chunk": copied,
        "h2d_gbs": round(h2d, 1),
        "link_h2d_gbs": round(link, 1),
        "frac_of_link": round(h2d / link, 4),
        "link_note": "one 2 GiB pinned-host-to-device copy, best of 5, CUDA events",
        "compute_ms_per_layer_resident": round(layer_ms, 3),
        "bound": "host-to-device copy" if ms > n_layers * layer_ms * 1.2 else "compute",
        "decode_with_expert_cache": cached,
    }


def run_offload_decode_cache(moe, dev, host, s, n_layers, B=4, n_slots=1536, warm=16, steps=16):
    """Decode batch B through the same offloaded layers (experts in pinned
    host memory): one step is B tokens through all layers.  With an HBM
    expert cache of n_slots experts (least recently used evicted) against the
    stager, which copies every touched expert of every layer at every step.
    Each step draws new logits (same Zipf(1.1) expert popularity per layer)."""
    shape = moe.Shape(B, s.E, s.k, s.H, s.I, FAT_THRESHOLD)
    x = synth.make_x(B, s.H, seed=0).to(dev)
    n_sets = warm + steps
    lg = [[synth.make_logits(B, s.E, seed=0, layer=l, rep=r, zipf_s=synth.ZIPF_S).to(dev)
           for l in range(n_layers)] for r in range(n_sets)]
    outs = [torch.empty((B, s.H), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    ws = moe.Workspace(moe.workspace_size(shape), dev)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev)
    ids = list(range(n_layers))

    cache = moe.ExpertCache(shape, n_slots, n_layers, dev)
    for r in range(warm):
        cache.forward(ids, lg[r], x, host, outs, ws, compute, copy)
    torch.cuda.synchronize()
    h0, m0 = cache.stats()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for r in range(warm, n_sets):
        cache.forward(ids, lg[r], x, host, outs, ws, compute, copy)
    t1.record()
    torch.cuda.synchronize()
    ms_cache = t0.elapsed_time(t1) / steps
    h1, m1 = cache.stats()
    cache.close()
    del cache
    torch.cuda.empty_cache()

    st = moe.Stager(shape, 8, dev)
    for r in range(2):
        st.forward(shape, lg[r], x, host, outs, ws, compute, copy)
    torch.cuda.synchronize()
    n_st = 4
    t0.record()
    for r in range(warm, warm + n_st):
        st.forward(shape, lg[r], x, host, outs, ws, compute, copy)
    t1.record()
    torch.cuda.synchronize()
    ms_stream = t0.elapsed_time(t1) / n_st
    st.close()
    del st
    torch.cuda.empty_cache()
    hits, misses = h1 - h0, m1 - m0
    return {
        "workload": f"decode batch {B} through {n_layers} offloaded layers (384 experts, H=2048, "
                    f"I=1024), HBM cache of {n_slots} experts "
                    f"({n_slots * moe.layer_weight_bytes(shape) // s.E / 1e9:.1f} GB)",
        "ms_per_step_cached": round(ms_cache, 3),
        "tokens_per_s_cached": round(B / (ms_cache * 1e-3), 1),
        "hit_rate": round(hits / max(hits + misses, 1), 4),
        "misses_per_step": round(misses / steps, 1),
        "ms_per_step_streamed": round(ms_stream, 3),
        "tokens_per_s_streamed": round(B / (ms_stream * 1e-3), 1),
    }


# -------------------------------------------------------------- GPU bench

def run_gpu(args):
    rank, world, local = init_dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import routed_expert_ffn_02_gb300 as moe
    peaks = load_peaks()

    T = args.tokens or PREFILL.T
    E = args.experts or PREFILL.E
    shape = moe.Shape(T, E, PREFILL.k, PREFILL.H, PREFILL.I, FAT_THRESHOLD, args.thin_mma_min)
    layer = Layer(moe, shape, dev, n_logit_sets=1)
    counts = layer.counts()
    work = stage_work(shape, counts)

    with ClockSampler(local) as clk:
        total_ms, stage_ms = time_steps(layer, args.steps, args.warmup, clk=clk)
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    value = world * shape.T * args.steps / (total_ms * 1e-3)
    if args.tokens or args.experts:
        print(f"# small case T={T} E={E}: {total_ms / args.steps:.4f} ms/step; stages "
              + json.dumps({k2: round(v2, 4) for k2, v2 in stage_ms.items()}), flush=True)

    dominant = max(stage_ms, key=stage_ms.get)
    roof = roofline_for(dominant, work, stage_ms[dominant], peaks)
    roof["kernel"] = dominant
    if work["_info"]["fat_experts"]:
        roof["note"] = ("the stage's first GEMM launch also copies two thirds of the row "
                        "gather (the later pair tiles', solo and tensor-core tiles' x rows) "
                        "with otherwise idle warps")
    roof["traffic"] = args.traffic if args.traffic is not None else (
        measured_traffic(dominant) if not (args.tokens or args.experts) else None)
    stages = {s: {"ms": round(stage_ms[s], 4), **{k2: v2 for k2, v2 in
                                                 roofline_for(s, work, max(stage_ms[s], 1e-6),
                                                              peaks).items()
                                                 if k2 in ("achieved", "unit", "frac", "frac_nominal")}}
              for s in stage_ms}
    layer_ideal_ms = max(
        (work["gemm_gate_up"]["flops"] + work["gemm_down"]["flops"]
         + work["thin_gate_up"]["flops"] + work["thin_down"]["flops"])
        / (peaks["bf16_tflops_sustained"] * 1e12),
        sum(w["bytes"] for n, w in work.items() if not n.startswith("_"))
        / (peaks["hbm_gbs"] * 1e9)) * 1e3
    # No-overlap bound: each touched expert alone at whichever of the tensor
    # or HBM roofline binds it (weights once, its rows of x in and y out),
    # summed over experts, so memory-bound medium and thin experts show.
    per_expert_ms = 0.0
    for n_e in counts[counts > 0]:
        f = 6.0 * int(n_e) * shape.H * shape.I
        b = 3.0 * shape.H * shape.I * 2 + int(n_e) * shape.H * 2 * 2
        per_expert_ms += max(f / (peaks["bf16_tflops_sustained"] * 1e12),
                             b / (peaks["hbm_gbs"] * 1e9)) * 1e3

    # end to end through the C ABI with host buffers (moe_forward_host): every
    # step copies its logits and x in from pinned host memory and its output
    # back; successive steps overlap one step's copies with another's compute.
    # The timed region opens before the first input copy and closes after the
    # last output copy.
    e2e = None
    if not args.no_e2e:
        x_h = layer.x_cpu.pin_memory()
        lg_h = layer.logits_cpu[0].pin_memory()
        out_h = torch.empty((shape.T, shape.H), dtype=torch.bfloat16).pin_memory()
        pipe = moe.Pipe(shape, dev)

        def e2e_step():
            pipe.forward(lg_h, x_h, layer.Wg, layer.Wu, layer.Wd, out_h)

        for _ in range(args.warmup):
            e2e_step()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        done = torch.cuda.Event()
        torch.cuda.synchronize()
        barrier()
        s0.record(pipe.compute)
        pipe.h2d.wait_event(s0)
        pipe.d2h.wait_event(s0)
        for _ in range(args.steps):
            e2e_step()
        done.record(pipe.d2h)
        pipe.compute.wait_event(done)
        s1.record(pipe.compute)
        torch.cuda.synchronize()
        barrier()
        assert pipe.ws.status() == 0
        e2e_ms = max_over_ranks(s0.elapsed_time(s1))
        e2e = {"value": round(world * shape.T * args.steps / (e2e_ms * 1e-3), 1),
               "unit": "tokens/s",
               "h2d_bytes_per_step": x_h.numel() * 2 + lg_h.numel() * 4,
               "d2h_bytes_per_step": out_h.numel() * 2,
               "ms_per_step": round(e2e_ms / args.steps, 4),
               "api": "moe_forward_host (pinned host buffers, copies overlapped across steps)"}
        pipe.close()

    # decode batches on the same resident layer (secondary lines): each step is
    # one forward captured in a CUDA graph (as a serving engine runs decode),
    # rotating 8 logit sets so the touched experts change from step to step.
    decode = {}
    if not args.no_decode:
        for B in (1, 4):
            dshape = moe.Shape(B, PREFILL.E, PREFILL.k, PREFILL.H, PREFILL.I, FAT_THRESHOLD,
                               args.thin_mma_min)
            dl = Layer(moe, dshape, dev, n_logit_sets=8, weights=(layer.Wg, layer.Wu, layer.Wd))
            dcounts = dl.counts()
            dwork = stage_work(dshape, dcounts)
            # a few hundred replays (tens of ms) so that the clock sampler
            # sees the timed window
            reps = max(args.steps, 500)
            with ClockSampler(local) as dclk:
                dt, dst = time_steps(dl, reps, max(args.warmup, 5))
                gt = time_graph_steps(dl, reps, max(args.warmup, 5), clk=dclk)
            dclocks = dclk.summary()
            dt, gt = max_over_ranks(dt), max_over_ranks(gt)
            bytes_step = sum(w["bytes"] for n, w in dwork.items() if not n.startswith("_"))
            decode[f"B{B}"] = {
                "tokens_per_s": round(world * B * reps / (gt * 1e-3), 1),
                "us_per_step": round(1e3 * gt / reps, 2),
                "us_per_step_eager": round(1e3 * dt / reps, 2),
                "touched_experts": dwork["_info"]["touched"],
                "layer_frac_of_hbm_roofline": round(
                    bytes_step / (gt / reps * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "layer_frac_of_nominal_hbm": round(
                    bytes_step / (gt / reps * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                "stage_us_eager": {s: round(1e3 * v, 2) for s, v in dst.items()},
                "clocks": {"sm_mhz": dclocks.get("sm_mhz"), "samples": dclocks.get("samples"),
                           "reasons": dclocks.get("reasons"),
                           "leg_sm_mhz_min": dclocks.get("run", {}).get("sm_mhz_min")},
            }
            del dl

    # CPU baseline: the oracle on a bounded token sample of this workload
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        def expert(e):
            return tuple(synth.bf16_bits(w[e]) for w in (layer.Wg, layer.Wu, layer.Wd))
        n = args.cpu_tokens
        tps, dt, n_exp = oracle_sample(n, expert, layer.logits_cpu[0].numpy(),
                                       synth.bf16_bits(layer.x_cpu), shape.k)
        cpu = {"value": round(tps, 4), "unit": "tokens/s", "cores": 1,
               "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n} tokens of the 16,384-token chunk with all their experts "
                         f"({n * shape.k} token-expert pairs, {n_exp} experts), "
                         f"single-threaded fp64, {dt:.1f} s"}

    sweep = None
    if not args.no_sweep:
        sweep = run_sweep(moe, dev, (layer.Wg, layer.Wu, layer.Wd), peaks, args.thin_mma_min)
    # One replica's offload leg pins 58 GB of host memory, so it runs at N=1 only.
    offload = None
    if not (args.no_offload or args.tokens or args.experts):
        offload = run_offload(args, moe, dev) if world == 1 else {
            "skipped": "runs at N=1 only (58 GB of pinned host memory per replica)"}

    launches = moe.forward_launches(shape) * args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": prefill_config(T, E, work["_info"], shape.thin_mma_min, world),
            "roofline": roof,
            "layer_roofline": {"ideal_ms": round(layer_ideal_ms, 4),
                               "frac": round(layer_ideal_ms / ms_per_step, 4),
                               "note": "max(all flops / bf16 sustained peak, all algorithmic "
                                       "bytes / HBM peak) over the whole layer",
                               "per_expert_ideal_ms": round(per_expert_ms, 4),
                               "per_expert_frac": round(per_expert_ms / ms_per_step, 4),
                               "per_expert_note": "sum over touched experts of max(flops / "
                                                  "bf16 sustained peak, bytes / HBM peak): no "
                                                  "overlap between experts"},
            "stages": stages,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "decode": decode,
            "decode_sweep_4_layers": sweep,
            "offload": offload,
            "peaks": peaks,
            "receipts": receipts(moe, layer),
        }
        print(json.dumps(line), flush=True)


def run_decode_profile(args):
    """A few eager decode forwards at batch B on a layer of E experts (384 by
    default, --experts to shrink it for profilers), H=4096, I=2048, 8 logit
    sets rotated (so each forward touches new experts); prints mean stage
    times.  For ncu."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import routed_expert_ffn_02_gb300 as moe
    B = args.decode_profile
    shape = moe.Shape(B, args.experts or PREFILL.E, PREFILL.k, PREFILL.H, PREFILL.I,
                      FAT_THRESHOLD, args.thin_mma_min)
    layer = Layer(moe, shape, dev, n_logit_sets=8)
    _, stage_ms = time_steps(layer, 8, 3)
    print(json.dumps({"decode_profile": f"B{B}",
                      "stage_us": {k: round(1e3 * v, 2) for k, v in stage_ms.items()}}),
          flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=48)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T of the layer (small cases for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E of the layer (small cases for profiling)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the decode batch sweep over 4 resident layers")
    ap.add_argument("--no-offload", action="store_true",
                    help="skip the offload prefill (58 GB of experts in pinned host memory)")
    ap.add_argument("--thin-mma-min", type=int, default=0,
                    help="slots from which a thin expert streams on the tensor cores "
                         "(0: library default; 33: CUDA cores only)")
    ap.add_argument("--decode-profile", type=int, default=None, metavar="B",
                    help="only run 8 eager decode forwards at batch B on the full layer "
                         "(for profilers) and print their stage times")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode_profile:
        run_decode_profile(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
