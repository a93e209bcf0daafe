"""Benchmark of the block-quantized integer GEMM/GEMV library on GB300.

Headline workload: decode GEMV at M = 1 over the four Q8_0 projections
N x K = 4096x4096, 12288x4096, 4096x12288, 151936x4096 (weights ~ N(0, 0.02),
activations ~ N(0, 1) with 1% of entries x20).  One step = quantize the four
activation rows + four GEMVs.  value = algorithmic GB/s of the whole step:
  bytes = sum over projections of N*K*(1 + 2/32) + M*K*(1 + 4/32) + M*N*4,
the same accounting for every arm.  The per-step working set (787 MB of
weights) is larger than L2, so no flush runs between steps.

Extra sections measure the other rows of the hot path: the decode workload at
M = 4, the prefill GEMM (M = 2048) in int8-equivalent TOPS, and the grouped
W4A8 MoE GEMM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica (weak scaling: the path has no
exchange step); rank 0 prints one JSON line.  --impl reference times the CPU
oracle on the host cores as the reference arm.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill int8 TOPS (% tensor peak); decode GEMV GB/s (% of HBM) on 1 GB300"
DECODE_WORKLOAD = ("decode GEMV M=1, Q8_0 W8A8, N x K = 4096x4096, 12288x4096, 4096x12288, "
                   "151936x4096; activation quantization + GEMV per projection")


def decode_bytes(M, shapes):
    return sum(N * K * (1 + 2 / 32) + M * K * (1 + 4 / 32) + M * N * 4 for N, K in shapes)


# DRAM bytes (read + write) of one lm-head GEMV launch, from the ncu capture
# summarised in profiles/gemv_q8_lmhead_151936x4096_m1.md (same kernel build).
LM_HEAD_TRAFFIC_BYTES = 661.244928e6 + 3.205376e6


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def host_cpu():
    """(logical cores, CPU model) of the host the oracle runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform
    return os.cpu_count() or 1, model or platform.machine()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def sampled(index, fn):
    """Run fn() under a clock sampler; returns (fn's result, clock record)."""
    smp = ClockSampler(index)
    smp.start()
    time.sleep(0.2)
    try:
        out = fn()
    finally:
        clk = smp.stop()
    return out, clk


def event_median_ms(fn, flush, min_reps, min_s=1.0):
    """Median CUDA-event time of fn() with flush() (an L2 scrub) before every
    call, outside the timed pair.  The calls are queued back to back, with one
    synchronize at the end, for at least min_reps calls and about min_s seconds,
    so that the GPU stays under load while its clocks are sampled."""
    import torch
    for _ in range(3):
        flush()
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    flush()
    fn()
    b.record()
    torch.cuda.synchronize()
    per = max(a.elapsed_time(b), 1e-3) * 1e-3
    reps = max(min_reps, min(int(min_s / per), 20000))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for x, y in evs:
        flush()
        x.record()
        fn()
        y.record()
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in evs), reps


# --------------------------------------------------------------------------- oracle arm

def oracle_decode(shapes, M, budget_s, steps_hint):
    """Time the CPU oracle on a bounded sample of the decode workload.

    Each sample step quantizes the activation rows and computes the first R
    output rows of every projection (R chosen so the whole run stays within
    budget_s).  Returns (GB/s, seconds per sample step, cores, description)."""
    import oracle
    from block_quantized_integer_gb300 import inputs
    cases = []
    for i, (N, K) in enumerate(shapes):
        rng = inputs.rng_for(inputs.DECODE, 100 + i)
        R = min(N, 4096)
        w = inputs.normal(rng, (R, K), 0.02)
        x = inputs.normal(rng, (M, K))
        inputs.with_entry_outliers(rng, x, 0.01, 20.0)
        qw, dw = oracle.quantize_w_q8_0(w)
        cases.append((N, K, x, qw, dw))

    def one(rows_frac):
        nbytes = 0.0
        t0 = time.perf_counter()
        for N, K, x, qw, dw in cases:
            R = max(1, int(qw.shape[0] * rows_frac))
            qx, dx = oracle.quantize_act_q8(x)
            oracle.qgemm(qx, dx, qw[:R], dw[:R], 8, want_mag=False)
            nbytes += R * K * (1 + 2 / 32) + M * K * (1 + 4 / 32) + M * R * 4
        return nbytes, time.perf_counter() - t0

    nb, dt = one(1.0)
    per_step = max(budget_s / max(steps_hint, 1), 0.02)
    frac = min(1.0, per_step / max(dt, 1e-6))
    return cases, one, frac, nb / dt / 1e9


# --------------------------------------------------------------------------- GPU arm

def make_decode(dev, M, seed_sub=0):
    """The four decode projections.  Their activations live in one device buffer
    (and one pinned host buffer), their outputs likewise, each projection's x and
    y being views: the end-to-end step moves the inputs in and the outputs out
    with one copy each (the keys x_all, x_all_host, y_all, y_all_host)."""
    import torch
    import block_quantized_integer_gb300 as qg
    from block_quantized_integer_gb300 import inputs
    shapes = inputs.DECODE_SHAPES
    nx, ny = sum(M * K for _, K in shapes), sum(M * N for N, _ in shapes)
    x_all = torch.empty(nx, dtype=torch.float32, device=dev)
    y_all = torch.empty(ny, dtype=torch.float32, device=dev)
    x_all_host = torch.empty(nx, dtype=torch.float32).pin_memory()
    y_all_host = torch.empty(ny, dtype=torch.float32).pin_memory()
    projs, ox, oy = [], 0, 0
    for i, (N, K) in enumerate(shapes):
        w, x = inputs.decode_case(N, K, M=M, sub=i + seed_sub)
        wt = torch.from_numpy(w).to(dev)
        qw, dw = qg.quantize_weight_q8_0(wt)
        del wt
        xt = x_all[ox:ox + M * K].view(M, K)
        xt.copy_(torch.from_numpy(x))
        x_all_host[ox:ox + M * K].copy_(torch.from_numpy(x).reshape(-1))
        qx = torch.empty((M, K), dtype=torch.int8, device=dev)
        dx = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
        y = y_all[oy:oy + M * N].view(M, N)
        projs.append(dict(N=N, K=K, x=xt, qx=qx, dx=dx, qw=qw, dw=dw, y=y, x_all=x_all,
                          y_all=y_all, x_all_host=x_all_host, y_all_host=y_all_host))
        ox += M * K
        oy += M * N
    torch.cuda.synchronize()
    return projs


class DecodeGraphs:
    """The decode step captured in CUDA graphs (the launch sequence is fixed,
    so graph replay removes per-launch host overhead from the small GEMVs):
    graph `full` = the whole step (four activation quantizations, four GEMVs)
    in one graph, so programmatic dependent launch reaches every kernel
    boundary, the lm-head GEMV's included;
    graphs `head` (quantizations + the three small GEMVs) and `lm` (the
    lm-head GEMV alone) replay the same launches split in two, so that CUDA
    events can time the lm-head GEMV by itself;
    graph `e2e` = the inputs in from pinned host memory (one copy), the whole
    step, the outputs out to pinned host memory (one copy)."""

    def __init__(self, projs):
        import torch
        import block_quantized_integer_gb300 as qg
        self.projs = projs
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):                      # warm up (allocations, attributes)
                self._head(qg)
                self._lm(qg)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.g_head, self.g_lm, self.g_e2e = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                              torch.cuda.CUDAGraph())
        self.g_full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_full):
            self._head(qg)
            self._lm(qg)
        with torch.cuda.graph(self.g_head):
            self._head(qg)
        with torch.cuda.graph(self.g_lm):
            self._lm(qg)
        pk = projs[0]
        with torch.cuda.graph(self.g_e2e):
            pk["x_all"].copy_(pk["x_all_host"], non_blocking=True)
            self._head(qg)
            self._lm(qg)
            pk["y_all_host"].copy_(pk["y_all"], non_blocking=True)
        torch.cuda.synchronize()

    def _head(self, qg):
        # projection by projection: quantize, then its GEMV; the lm-head's
        # quantization closes the head so that its GEMV can stand alone
        for p in self.projs[:-1]:
            qg.quantize_act_q8(p["x"], p["qx"], p["dx"])
            qg.qgemm_q8_0(p["qx"], p["dx"], p["qw"], p["dw"], y=p["y"])
        p = self.projs[-1]
        qg.quantize_act_q8(p["x"], p["qx"], p["dx"])

    def _lm(self, qg):
        p = self.projs[-1]
        qg.qgemm_q8_0(p["qx"], p["dx"], p["qw"], p["dw"], y=p["y"])

    def step_full(self, timer=None):
        self.g_full.replay()

    def step(self, timer=None):
        self.g_head.replay()
        if timer is not None:
            timer[0].record()
        self.g_lm.replay()
        if timer is not None:
            timer[1].record()

    def step_e2e(self, timer=None):
        self.g_e2e.replay()


def max_over_ranks(ms, dist=None, device="cuda"):
    """The slowest rank's time: every rank contributes its own, all receive the max
    (NCCL needs a device tensor, gloo a host one)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world, bytes_per_step, steps, ms):
    """Whole-job GB/s of `world` replicas, each moving bytes_per_step per step, timed by
    the slowest rank over `steps` steps."""
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


def timed(fn, steps, warmup, dist=None, per_kernel=None):
    """Run fn warmup times, then time `steps` calls with CUDA events on the
    current stream, barrier + synchronize on both sides; max over ranks."""
    import torch
    for _ in range(warmup):
        fn(None)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    timers = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)] if per_kernel else [None] * steps
    start.record()
    for i in range(steps):
        fn(timers[i])
    end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist)
    kms = None
    if per_kernel:
        kms = statistics.mean(a.elapsed_time(b) for a, b in timers)
    return ms, kms


def prefill_section(dev, peaks, reps=20, long_ctx=False):
    """Prefill GEMM M=2048 (both shapes), or the M=18432 long-context shapes:
    int8-equivalent TOPS = 2MNK / t."""
    import torch
    import block_quantized_integer_gb300 as qg
    from block_quantized_integer_gb300 import inputs
    out = []
    shapes = inputs.LONGCTX_SHAPES if long_ctx else inputs.PREFILL_SHAPES
    for i, (M, N, K) in enumerate(shapes):
        w, x = (inputs.longctx_case(M, N, K, sub=i) if long_ctx
                else inputs.prefill_case(M, N, K, sub=i))
        qw, dw = qg.quantize_weight_q8_0(torch.from_numpy(w).to(dev))
        qx, dx = qg.quantize_act_q8(torch.from_numpy(x).to(dev))
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws = torch.empty(qg.workspace_size(qg.OP_QGEMM_Q8_0, M, N, K), dtype=torch.uint8,
                         device=dev)
        scrub = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
        # flush L2 (256 MB > 129 MB) before every call
        ms, n = event_median_ms(lambda: qg.qgemm_q8_0(qx, dx, qw, dw, y=y, workspace=ws),
                                lambda: scrub.fill_(1.0), reps)
        tops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out.append({"M": M, "N": N, "K": K, "ms": ms, "tops": tops, "reps": n,
                    "frac_of_bf16_peak": tops / peaks["bf16_tflops"]})
        del qw, dw, qx, dx, y, scrub
    return {"unit": "TOPS (int8-equivalent, 2MNK/t)", "shapes": out,
            "peak_tflops": peaks["bf16_tflops"],
            "peak_note": "bf16 dense tensor peak (" + peaks["source"] + "); the kernel issues "
                         "integer-valued f16 or s8 MMA, no int8 tcgen05 form exists on sm_103a",
            "l2": "flushed before every timed call"}


def moe_section(dev, peaks, reps=20):
    import torch
    import block_quantized_integer_gb300 as qg
    from block_quantized_integer_gb300 import inputs
    d = inputs.moe_case()
    ids = torch.from_numpy(d["topk_ids"]).to(dev)
    res = {}
    total_ms, total_bytes, total_ops = 0.0, 0.0, 0.0
    for which, key, xkey, mode in (("gate_up", "w_gate_up", "x_tok", 0),
                                   ("down", "w_down", "x_pair", 1)):
        w = d[key]
        E, N, K = w.shape
        qw4, dw = qg.quantize_weight_q4_0(torch.from_numpy(w.reshape(E * N, K)).to(dev))
        qw4, dw = qw4.view(E, N, K // 2), dw.view(E, N, K // 32)
        qx, dx = qg.quantize_act_q8(torch.from_numpy(d[xkey]).to(dev))
        P = ids.numel()
        y = torch.empty((P, N), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(qg.workspace_size(qg.OP_GROUPED_MOE, 0, N, K, ids.shape[0],
                                           ids.shape[1], E), dtype=torch.uint8, device=dev)
        scrub = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
        ms, _ = event_median_ms(
            lambda: qg.grouped_qgemm_moe(qx, dx, ids, mode, qw4, dw, y=y, d_err=err, workspace=ws),
            lambda: scrub.fill_(1.0), reps)
        used = np.unique(d["topk_ids"]).size
        nbytes = used * N * K * (0.5 + 2 / 32) + qx.shape[0] * K * (1 + 4 / 32) + P * N * 4
        ops = 2.0 * P * N * K
        res[which] = {"E": E, "N": N, "K": K, "pairs": P, "ms": ms,
                      "gbs": nbytes / (ms * 1e-3) / 1e9, "tops": ops / (ms * 1e-3) / 1e12}
        total_ms += ms
        total_bytes += nbytes
        total_ops += ops
        del qw4, dw, qx, dx, y, scrub
    res["total"] = {"ms": total_ms, "gbs": total_bytes / (total_ms * 1e-3) / 1e9,
                    "tops": total_ops / (total_ms * 1e-3) / 1e12,
                    "frac_of_hbm": total_bytes / (total_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    res["workload"] = ("grouped W4A8 MoE, 128 experts, gate/up N=2048 (fused) K=2048 and "
                       "down N=2048 K=1024, 947 tokens top-8 Zipf(1.1); routing included")
    res["l2"] = "flushed before every timed call"
    return res


def moe_layer_section(dev, peaks, reps=20):
    """The whole MoE layer on the MoE workload: gate/up grouped GEMM -> SwiGLU +
    re-quantization -> down grouped GEMM (one activation row per pair) ->
    router-weighted combine, every step through the C ABI on one stream."""
    import torch
    import block_quantized_integer_gb300 as qg
    from block_quantized_integer_gb300 import inputs
    d = inputs.moe_case()
    ids = torch.from_numpy(d["topk_ids"]).to(dev)
    rw = torch.from_numpy(d["route_w"]).to(dev)
    T, topk = ids.shape
    P = T * topk
    w1, w2 = d["w_gate_up"], d["w_down"]
    E, N1, K1 = w1.shape
    _, N2, K2 = w2.shape
    F = N1 // 2
    q1, d1 = qg.quantize_weight_q4_0(torch.from_numpy(w1.reshape(E * N1, K1)).to(dev))
    q2, d2 = qg.quantize_weight_q4_0(torch.from_numpy(w2.reshape(E * N2, K2)).to(dev))
    q1, d1 = q1.view(E, N1, K1 // 2), d1.view(E, N1, K1 // 32)
    q2, d2 = q2.view(E, N2, K2 // 2), d2.view(E, N2, K2 // 32)
    qx, dx = qg.quantize_act_q8(torch.from_numpy(d["x_tok"]).to(dev))
    gu = torch.empty((P, N1), dtype=torch.float32, device=dev)
    yd = torch.empty((P, N2), dtype=torch.float32, device=dev)
    out = torch.empty((T, N2), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws1 = torch.empty(qg.workspace_size(qg.OP_GROUPED_MOE, 0, N1, K1, T, topk, E), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(qg.workspace_size(qg.OP_GROUPED_MOE, 0, N2, K2, T, topk, E), dtype=torch.uint8, device=dev)
    scrub = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)

    def layer(ev=None):
        if ev: ev[0].record()
        qg.grouped_qgemm_moe(qx, dx, ids, 0, q1, d1, y=gu, d_err=err, workspace=ws1)
        if ev: ev[1].record()
        qh, dh = qg.moe_swiglu_quant(gu, F)
        if ev: ev[2].record()
        qg.grouped_qgemm_moe(qh, dh, ids, 1, q2, d2, y=yd, d_err=err, workspace=ws2)
        if ev: ev[3].record()
        qg.moe_combine(yd, rw, out=out)
        if ev: ev[4].record()

    for _ in range(3):
        layer()
    steps = {k: [] for k in ("gate_up", "swiglu_quant", "down", "combine", "total")}
    for _ in range(reps):
        scrub.fill_(1.0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        layer(ev)
        torch.cuda.synchronize()
        t = [ev[i].elapsed_time(ev[i + 1]) for i in range(4)]
        for k, v in zip(("gate_up", "swiglu_quant", "down", "combine"), t):
            steps[k].append(v)
        steps["total"].append(ev[0].elapsed_time(ev[4]))
    res = {k + "_ms": statistics.median(v) for k, v in steps.items()}
    wbytes = (np.unique(d["topk_ids"]).size * (N1 * K1 + N2 * K2) * (0.5 + 2 / 32))
    res["weight_gbs"] = wbytes / (res["total_ms"] * 1e-3) / 1e9
    res["frac_of_hbm_weights"] = res["weight_gbs"] / peaks["hbm_gbs"]
    res["workload"] = ("MoE layer: 947 tokens top-8 Zipf(1.1) over 128 experts; gate/up N=2048 K=2048, "
                       "SwiGLU + int8 re-quantization F=1024, down N=2048 K=1024, router-weighted combine")
    res["l2"] = "flushed before every timed layer"
    del scrub
    return res


def decode_shapes_section(dev, peaks, reps=50):
    """Each decode projection on its own at M = 1 and M = 4, L2 flushed before every
    timed call (the 17.8 MB projection would otherwise be served from L2); median of
    reps.  Keys M{M}_{N}x{K}: activation quantization + GEMV, two launches;
    fused_M{M}_{N}x{K}: the one-launch GEMV that quantizes x itself."""
    import torch
    import block_quantized_integer_gb300 as qg
    scrub = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
    out = {}

    def median_ms(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            scrub.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    for M in (1, 4):
        projs = make_decode(dev, M)
        for p in projs:
            def two():
                qg.quantize_act_q8(p["x"], p["qx"], p["dx"])
                qg.qgemm_q8_0(p["qx"], p["dx"], p["qw"], p["dw"], y=p["y"])

            def fused():
                qg.qgemv_q8_0_f32(p["x"], p["qw"], p["dw"], y=p["y"])
            nb = decode_bytes(M, [(p["N"], p["K"])])
            for key, fn in ((f"M{M}_{p['N']}x{p['K']}", two),
                            (f"fused_M{M}_{p['N']}x{p['K']}", fused)):
                ms = median_ms(fn)
                out[key] = {"us": ms * 1e3, "gbs": nb / (ms * 1e-3) / 1e9,
                            "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del projs
        torch.cuda.empty_cache()
    out["l2"] = "flushed before every timed call"
    del scrub
    return out


def next_rows_section(dev, peaks, reps=20):
    """The HBM-bound kernels of the rows beyond the hot path, each on a
    representative size, as algorithmic GB/s against the measured HBM peak
    (L2 flushed before every timed call)."""
    import torch
    import block_quantized_integer_gb300 as qg
    g = torch.Generator(device="cpu").manual_seed(20261202 + 7)
    scrub = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)

    def timeit(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            scrub.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    out = {}
    # activation quantization (hot-path row a1) at its largest workload: the
    # long-context prefill activations, 18432 x 17408 binary32 (1.28 GB in)
    Mq, Kq = 18432, 17408
    xq = torch.randn((Mq, Kq), generator=g).to(dev)
    qxq = torch.empty((Mq, Kq), dtype=torch.int8, device=dev)
    dxq = torch.empty((Mq, Kq // 32), dtype=torch.float32, device=dev)
    ms = timeit(lambda: qg.quantize_act_q8(xq, qxq, dxq))
    nb = Mq * Kq * (4 + 1 + 4 / 32)
    out["quantize_act_q8"] = {"shape": f"{Mq}x{Kq}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    del xq, qxq, dxq
    # SwiGLU + re-quantization on the MoE workload's gate/up output (7576 x 2048 -> 7576 x 1024)
    P, F = 7576, 1024
    gu = torch.randn((P, 2 * F), generator=g).to(dev)
    ms = timeit(lambda: qg.moe_swiglu_quant(gu, F))
    nb = P * 2 * F * 4 + P * F * (1 + 4 / 32)
    out["swiglu_quant"] = {"shape": f"{P}x{2 * F} -> {P}x{F}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    # router-weighted combine: 947 tokens x top-8 rows of 2048
    T, topk, N = 947, 8, 2048
    y = torch.randn((T * topk, N), generator=g).to(dev)
    w = torch.rand((T, topk), generator=g).to(dev)
    o = torch.empty((T, N), device=dev)
    ms = timeit(lambda: qg.moe_combine(y, w, out=o))
    nb = T * topk * N * 4 + T * topk * 4 + T * N * 4
    out["moe_combine"] = {"shape": f"{T}x{topk}x{N}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    # GGUF Q8_0 import of a 12288 x 4096 matrix (34-byte blocks -> planes)
    Nw, K = 12288, 4096
    blocks = torch.randint(0, 256, (Nw * (K // 32) * 34,), dtype=torch.uint8, generator=g).to(dev)
    ms = timeit(lambda: qg.import_gguf_q8_0(blocks, Nw, K))
    nb = 2 * Nw * (K // 32) * 34
    out["import_gguf_q8_0"] = {"shape": f"{Nw}x{K}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    # split-K attention merge: 16 splits x 32 heads x 2048 queries x D 128
    S, R, D = 16, 32 * 2048, 128
    mm = torch.randn((S, R), generator=g).to(dev)
    ll = (torch.rand((S, R), generator=g) + 1.0).to(dev)
    acc = torch.randn((S, R, D), generator=g).to(dev)
    ms = timeit(lambda: qg.attn_splitk_merge(mm, ll, acc))
    nb = S * R * (D + 2) * 4 + R * (D + 1) * 4
    out["attn_splitk_merge"] = {"shape": f"S={S} R={R} D={D}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    # 3-bit KV codec: one head's keys over a 256 K context, D = 128
    Tk, Dk = 262144, 128
    xk = torch.randn((Tk, Dk), generator=g).to(dev)
    ck, sk = qg.kv3_encode(xk)
    ms = timeit(lambda: qg.kv3_encode(xk))
    nb = Tk * Dk * 4 + Tk * (3 * Dk // 8 + 4)
    out["kv3_encode"] = {"shape": f"T={Tk} D={Dk}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    ms = timeit(lambda: qg.kv3_decode(ck, sk, Dk))
    out["kv3_decode"] = {"shape": f"T={Tk} D={Dk}", "ms": ms, "gbs": nb / (ms * 1e-3) / 1e9}
    del xk, ck, sk
    # The same byte count moved by a plain device copy (half read, half written),
    # timed the same way: at 70-150 MB a call, launch and ramp take a visible part
    # of any kernel, so this is the bound a streaming kernel of that size meets.
    for v in out.values():
        half = (int(v["gbs"] * 1e9 * v["ms"] * 1e-3) // 2 + 15) // 16 * 16
        src = torch.empty(half, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        v["copy_ms"] = timeit(lambda: dst.copy_(src))
        v["frac_of_copy"] = v["copy_ms"] / v["ms"]
        v["frac_of_hbm"] = v["gbs"] / peaks["hbm_gbs"]
        del src, dst
    out["l2"] = "flushed before every timed call"
    out["copy"] = ("frac_of_copy: a device-to-device copy of the same bytes (half read, half "
                   "written), timed the same way, divided by the kernel's time")
    del scrub
    return out


def flatten_sections(line, peaks, clocks):
    """Copy every configured workload's figure to flat scalar keys, at the top
    level and in the `prefill` dict (a record that keeps only scalars still
    holds them), with each timed section's clock record beside it."""
    flat = {}
    for key, sec in (("prefill", "prefill"), ("longctx", "prefill_long_context")):
        for r in line[sec]["shapes"]:
            tag = f"{key}_{r['M']}x{r['N']}x{r['K']}"
            flat[tag + "_tops"] = r["tops"]
            flat[tag + "_frac"] = r["frac_of_bf16_peak"]
            flat[tag + "_ms"] = r["ms"]
    moe = line["moe"]
    flat["moe_total_ms"] = moe["total"]["ms"]
    flat["moe_total_frac_of_hbm"] = moe["total"]["frac_of_hbm"]
    flat["moe_gate_up_ms"] = moe["gate_up"]["ms"]
    flat["moe_down_ms"] = moe["down"]["ms"]
    flat["moe_layer_total_ms"] = line["moe_layer"]["total_ms"]
    flat["moe_layer_frac_of_hbm"] = line["moe_layer"]["frac_of_hbm_weights"]
    flat["decode_m4_gbs"] = line["decode_m4"]["gbs"]
    flat["decode_m4_frac"] = line["decode_m4"]["gbs"] / peaks["hbm_gbs"]
    for k, v in line["next_rows"].items():
        if isinstance(v, dict):
            flat[f"next_{k}_frac"] = v["frac_of_hbm"]
            flat[f"next_{k}_frac_of_copy"] = v["frac_of_copy"]
    for sec, clk in clocks.items():
        flat[f"{sec}_sm_mhz"] = clk.get("sm_mhz")
        flat[f"{sec}_clock_samples"] = clk.get("samples", 0)
        flat[f"{sec}_throttle"] = ",".join(clk.get("reasons", [])) or "none"
        line["clocks"][f"{sec}_sm_mhz"] = clk.get("sm_mhz")
        line["clocks"][f"{sec}_reasons"] = ",".join(clk.get("reasons", [])) or "none"
    line.update(flat)
    line["prefill"].update(flat)


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip prefill/MoE/M=4 sections")
    ap.add_argument("--only", choices=["prefill", "longctx", "moe", "moe_layer", "next", "decode",
                                       "decode_shapes"],
                    default=None,
                    help="run one section only (for profiling); prints its JSON")
    ap.add_argument("--reps", type=int, default=50, help="timed calls per prefill/MoE shape")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.only is not None:
        import torch
        dev = torch.device("cuda", 0)
        peaks = load_peaks()
        if args.only == "prefill":
            out = prefill_section(dev, peaks, reps=args.reps)
        elif args.only == "longctx":
            out = prefill_section(dev, peaks, reps=args.reps, long_ctx=True)
        elif args.only == "moe":
            out = moe_section(dev, peaks, reps=args.reps)
        elif args.only == "moe_layer":
            out = moe_layer_section(dev, peaks, reps=args.reps)
        elif args.only == "next":
            out = next_rows_section(dev, peaks, reps=args.reps)
        elif args.only == "decode_shapes":
            out = decode_shapes_section(dev, peaks, reps=args.reps)
        else:
            projs = make_decode(dev, 1)
            graphs = DecodeGraphs(projs)
            ms, _ = timed(graphs.step_full, args.steps, args.warmup, None)
            _, kms = timed(graphs.step, args.steps, args.warmup, None, per_kernel=True)
            from block_quantized_integer_gb300 import inputs as _in
            out = {"gbs": decode_bytes(1, _in.DECODE_SHAPES) * args.steps / (ms * 1e-3) / 1e9,
                   "lm_head_ms": kms}
        print(json.dumps(out), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from block_quantized_integer_gb300 import inputs
    shapes = inputs.DECODE_SHAPES
    bytes_step = decode_bytes(1, shapes)

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 60.0
        cases, one, frac, _ = oracle_decode(shapes, 1, budget, args.steps + args.warmup)
        for _ in range(args.warmup):
            one(frac)
        tot_b, tot_t = 0.0, 0.0
        for _ in range(args.steps):
            b, t = one(frac)
            tot_b += b
            tot_t += t
        import oracle
        v = tot_b / tot_t / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
                "config": {"workload": DECODE_WORKLOAD, "parallelism": "replicas"},
                "cpu_baseline": {"value": v, "unit": "GB/s",
                                 "cores": oracle.num_threads(), "nproc": host_cpu()[0],
                                 "cpu_model": host_cpu()[1], "kind": "oracle",
                                 "sample": f"first {frac:.4f} of the rows of each projection "
                                           f"(at most 4096 rows), M=1, per step"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import block_quantized_integer_gb300 as qg
    peaks = load_peaks()

    projs = make_decode(dev, 1)
    graphs = DecodeGraphs(projs)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms, _ = timed(graphs.step_full, args.steps, args.warmup, dist)
    # the lm-head GEMV alone, for the roofline: the same launches with the step
    # split into two graphs and CUDA events around the second
    _, kms = timed(graphs.step, args.steps, args.warmup, dist, per_kernel=True)
    clocks = sampler.stop()
    value = replica_value(world, bytes_step, args.steps, ms)

    # end to end: pinned host x in, y out, every step
    ms_e2e, _ = timed(graphs.step_e2e, max(args.steps // 4, 10), 3, dist)
    e2e = replica_value(world, bytes_step, max(args.steps // 4, 10), ms_e2e)
    h2d = projs[0]["x_all_host"].numel() * 4
    d2h = projs[0]["y_all_host"].numel() * 4

    N_lm, K_lm = shapes[-1]
    lm_bytes = decode_bytes(1, [(N_lm, K_lm)])
    achieved = lm_bytes / (kms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "M": 1, "parallelism": "replicas" if world > 1
                   else "single GPU", "l2": "inputs larger than L2: 787 MB of weights per step, "
                                            "no flush"},
        "frac_of_hbm": value / world / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": LM_HEAD_TRAFFIC_BYTES, "algorithmic_bytes": lm_bytes,
                     "kernel": "gemv_kernel (151936x4096 Q8_0, M=1)",
                     "peak_source": peaks["source"] + " STREAM-style copy"},
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * len(projs) * args.steps,
        "launch": "one CUDA graph per step (quantize x4, four GEMVs, programmatic dependent "
                  "launch between kernels); the lm-head GEMV timed alone in a second loop that "
                  "splits the step into two graphs",
        "clocks": clocks,
    }
    del graphs, projs
    torch.cuda.empty_cache()

    if not args.no_extra and rank == 0:
        def m4():
            projs4 = make_decode(dev, 4)
            g4 = DecodeGraphs(projs4)
            n4 = max(args.steps // 2, 10)
            ms4, _ = timed(g4.step_full, n4, 5)
            del g4, projs4
            return decode_bytes(4, shapes) * n4 / (ms4 * 1e-3) / 1e9, ms4 / n4
        (gbs4, ms4), clk4 = sampled(local, m4)
        line["decode_m4"] = {"gbs": gbs4, "ms_per_step": ms4}
        torch.cuda.empty_cache()
        line["decode_shapes"] = decode_shapes_section(dev, peaks, reps=args.reps)
        torch.cuda.empty_cache()
        line["prefill"], clk_pf = sampled(local, lambda: prefill_section(dev, peaks, reps=args.reps))
        torch.cuda.empty_cache()
        line["prefill_long_context"], clk_lc = sampled(
            local, lambda: prefill_section(dev, peaks, reps=max(args.reps // 4, 3), long_ctx=True))
        torch.cuda.empty_cache()
        line["moe"], clk_moe = sampled(local, lambda: moe_section(dev, peaks, reps=args.reps))
        line["moe_layer"] = moe_layer_section(dev, peaks, reps=args.reps)
        line["next_rows"] = next_rows_section(dev, peaks, reps=args.reps)
        torch.cuda.empty_cache()
        flatten_sections(line, peaks, {"decode_m4": clk4, "prefill": clk_pf, "longctx": clk_lc,
                                       "moe": clk_moe})

    if rank == 0:
        _, one, frac, _ = oracle_decode(shapes, 1, 15.0, 1)
        one(frac)
        b, t = one(frac)
        import oracle
        nproc, model = host_cpu()
        # the oracle splits its output rows into column chunks over OpenMP threads
        line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s",
                                "cores": oracle.num_threads(), "nproc": nproc, "cpu_model": model,
                                "kind": "oracle",
                                "sample": f"first {frac:.4f} of the rows of each projection "
                                          f"(at most 4096 rows), M=1, one step"}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
