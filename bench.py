#!/usr/bin/env python3
"""Benchmark of the GB300 W4A16 dequantise-GEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_int4|prefill_mxfp4|large_nvfp4|tiny_nvfp4|layer_sweep]

Default workload (decode_int4): the decode GEMV of the 3B int4-g128 model's
gate/up projection, N=8192, K=3072, bf16 activations, bf16 output.  One STEP
is the whole hot path over one batch: three wq_gemm calls, at M = 1, 4 and
16, each on its own weight set.  R distinct device copies of the weights
(more than twice the L2 size in total) are rotated, so every call streams its
weights from HBM.  The timed steps are replayed from CUDA graphs, K steps
exactly, bracketed by a barrier and cudaDeviceSynchronize, timed with CUDA
events on the launching stream, max over ranks.  The metric is the effective
weight bandwidth (packed codes + scales + zeros per call / time).

Prints ONE JSON line on rank 0 (keys described in the design notes):
metric, value, unit, roofline (dominant kernel, live CUDA-event timing),
cpu_baseline (the oracle on the host cores, bounded sample), e2e (through the
public Python API with pinned host buffers), clocks (nvidia-smi sampled
during the timed region), gpu_launches.

--workload layer_sweep: one step is every projection of the 3B decoder (q,
k, v, o, gate, up, down) and the tied LM head, int4 g128, at M = 1, 16, 128
and 2048 (32 chained calls); the value is the step's fraction of the roofline
(sum over the calls of max(bytes / HBM, flops / bf16 tensor peak) over the
measured step time), with every (shape, M) also timed alone in "per_shape".

--impl reference times the oracle (the fp64 CPU implementation under
oracle/) on the same workload and prints the same line with
"impl": "reference".  Under torchrun every rank runs an independent replica
(the path has no exchange step); value is the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

BENCH_WORKLOADS = {
    "decode_int4": dict(fmt="int4", group=128, Ms=(1, 4, 16), N=8192, K=3072, out="bf16",
                        bound="hbm", metric="weight HBM GB/s (M≤16)", unit="GB/s"),
    "prefill_mxfp4": dict(fmt="mxfp4", group=32, Ms=(2048,), N=3072, K=3072, out="bf16",
                          bound="tensor", metric="dequant-GEMM TFLOP/s (large M)", unit="TFLOP/s"),
    "large_nvfp4": dict(fmt="nvfp4", group=16, Ms=(8192,), N=8192, K=8192, out="bf16", scale_mult=1.0,
                        bound="tensor", metric="dequant-GEMM TFLOP/s (large M)", unit="TFLOP/s"),
    "tiny_nvfp4": dict(fmt="nvfp4", group=16, Ms=(16,), N=256, K=512, out="fp32",
                       bound="hbm", metric="weight HBM GB/s (M≤16)", unit="GB/s"),
    # every projection of the 3B decoder (k and v, gate and up: two calls of
    # one shape, distinct weights) and the tied LM head, at M = 1, 16, 128,
    # 2048; one step is all 32 calls, chained; the value is the step's
    # fraction of the roofline: sum over calls of max(bytes / HBM, flops /
    # tensor peak), over the measured step time
    "layer_sweep": dict(fmt="int4", group=128, Ms=(1, 16, 128, 2048), out="bf16", bound="roofline",
                        calls=(("q", "q"), ("k", "kv"), ("v", "kv"), ("o", "o"), ("gate", "gate_up"),
                               ("up", "gate_up"), ("down", "down"), ("lm_head", "lm_head")),
                        metric="% of roofline (decoder-layer sweep)", unit="% of roofline"),
}
DEFAULT_STEPS = {"layer_sweep": (300, 10)}   # (steps, warm-up) when not given: one step is ~2 ms

# launch modes of the small-M calls (include/wq.h); the tensor-core path
# ignores both bits
LAUNCH_FLAGS = {
    "ready": lambda wq: wq.WQ_LAUNCH_INPUTS_READY,
    "overlap": lambda wq: wq.WQ_LAUNCH_OVERLAP,
    "plain": lambda wq: 0,
}
LAUNCH_DESC = {
    "ready": "WQ_LAUNCH_INPUTS_READY (programmatic dependent launch; the activations were written before the "
             "chain, so each call reads them at once and waits for its predecessor only before storing C)",
    "overlap": "WQ_LAUNCH_OVERLAP (programmatic dependent launch; each call reads A after its predecessor "
               "completes: a dependent chain)",
    "plain": "plain launches",
}
SPIN_CYCLES = 100000   # ~50 us spin ahead of a start event (device clock cycles)


def bench_config(workload: str, ws: int) -> dict:
    """The workload a line measures: identical in both arms (how our arm
    launches and lays out its weights is under the line's "setup")."""
    w = BENCH_WORKLOADS[workload]
    cfg = {"workload": workload, "format": w["fmt"], "group": w["group"], "M": list(w["Ms"]), "out": w["out"]}
    if workload == "layer_sweep":
        from weight_only_bit_w4a16_gb300 import synth
        cfg["calls"] = {c: list(synth.LAYER_SHAPES[fam]) for c, fam in w["calls"]}
        cfg["calls_per_step"] = len(w["Ms"]) * len(w["calls"])
    else:
        cfg.update(N=w["N"], K=w["K"], calls_per_step=len(w["Ms"]))
    cfg["parallelism"] = f"replicas x{ws}"
    return cfg

KERNEL_SOURCES = {  # files whose content defines the dominant kernel of a workload (and layout)
    "decode_int4": ["wq_gemv_tma.cu", "wq_gemv.cuh", "wq_common.cuh"],
    "decode_int4:prepacked": ["wq_gemv_pre.cu", "wq_gemv.cuh", "wq_common.cuh", "wq_tc.cuh"],
    "tiny_nvfp4": ["wq_gemv_tma.cu", "wq_gemv.cuh", "wq_common.cuh"],
    "tiny_nvfp4:prepacked": ["wq_gemv_pre.cu", "wq_gemv.cuh", "wq_common.cuh"],
    "prefill_mxfp4": ["wq_tc.cu", "wq_tc.cuh", "wq_common.cuh"],
    "prefill_mxfp4:prepacked": ["wq_tc.cu", "wq_tc.cuh", "wq_common.cuh"],
    "large_nvfp4": ["wq_tc.cu", "wq_tc.cuh", "wq_common.cuh"],
    "large_nvfp4:prepacked": ["wq_tc.cu", "wq_tc.cuh", "wq_common.cuh"],
}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; timing max over ranks)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(use_cuda: bool):
    ws, rank, _ = dist_env()
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [r for r, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.monotonic(), sm, smax, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if not inside:   # timed region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest to timed region"
        sm = sorted(s[1] for s in inside)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted({r for s in inside for r in s[3]}), "samples": len(inside),
                "window": window}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_hash(workload: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[workload]:
        p = os.path.join(ROOT, "weight_only_bit_w4a16_gb300", "csrc", f)
        if os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (profiles/traffic.txt: workload hash bytes)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_hash(workload)
    with open(p) as f:
        for line in f:
            parts = line.split("#")[0].split()
            if len(parts) >= 3 and parts[0] == workload and parts[1] == want:
                return float(parts[2])
    return None


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def oracle_step_sample(w, cols_per_call: int, A_by_M, weights, seed=0):
    """Run the oracle on a column sample of every call of one step; returns
    (seconds, weight bytes covered)."""
    import oracle
    from weight_only_bit_w4a16_gb300 import metrics
    packed, scales, zeros = weights
    rng = np.random.default_rng(seed)
    t = time.perf_counter()
    covered = 0
    for M in w["Ms"]:
        cols = np.sort(rng.choice(w["N"], size=cols_per_call, replace=False))
        oracle.gemm(A_by_M[M], packed, scales, zeros, w["fmt"], w["group"], cols=cols)
        covered += metrics.weight_bytes(w["fmt"], cols_per_call, w["K"], w["group"])
    return time.perf_counter() - t, covered


def oracle_rate(w, A_by_M, weights, budget_s: float):
    """Calibrate a column sample to about budget_s of oracle work per step."""
    cols = min(w["N"], 64)
    dt, _ = oracle_step_sample(w, cols, A_by_M, weights)
    cols = int(max(1, min(w["N"], cols * budget_s / max(dt, 1e-6))))
    return cols


def host_inputs(w, seed=0):
    from weight_only_bit_w4a16_gb300 import synth
    weights = synth.make_weights(w["fmt"], w["N"], w["K"], w["group"], seed=seed,
                                 scale_mult=w.get("scale_mult", 0.5))
    A_by_M = {M: synth.draw_A(np.random.default_rng(seed + 1000 + M), M, w["K"]) for M in w["Ms"]}
    return A_by_M, weights


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def one_core(measure, budget_s):
    """measure(budget) -> dict on one oracle thread; the thread count is restored."""
    import oracle
    n = oracle.max_threads()
    oracle.set_threads(1)
    try:
        return measure(budget_s)
    finally:
        oracle.set_threads(n)


def cpu_baseline(w, A_by_M, weights, budget_s=15.0):
    import oracle
    from weight_only_bit_w4a16_gb300 import metrics

    def measure(budget):
        cols = oracle_rate(w, A_by_M, weights, budget)
        dt, covered = oracle_step_sample(w, cols, A_by_M, weights, seed=1)
        flops = sum(metrics.call_flops(M, cols, w["K"]) for M in w["Ms"])
        value = covered / dt / 1e9 if w["unit"] == "GB/s" else flops / dt / 1e12
        return {"value": value, "sample": f"{cols} of {w['N']} output columns of each call of one step "
                                          f"(M={list(w['Ms'])}, K={w['K']}), {dt:.1f} s"}

    res = measure(budget_s)
    single = one_core(measure, max(0.05, budget_s / 4))
    return {"value": res["value"], "unit": w["unit"], "cores": oracle.max_threads(), "kind": "oracle",
            "sample": res["sample"], "cpu": cpu_model(),
            "one_core": {"value": single["value"], "unit": w["unit"], "sample": single["sample"]}}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import weight_only_bit_w4a16_gb300 as wq
    from weight_only_bit_w4a16_gb300 import metrics

    ws, rank = dist_init(use_cuda=True)
    _, _, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wq.lib()   # fails loudly without the built library
    w = BENCH_WORKLOADS[args.workload]
    fmt, group, Ms, N, K, out = w["fmt"], w["group"], w["Ms"], w["N"], w["K"], w["out"]
    fcode = wq.FORMATS[fmt] | (wq.WQ_OUT_F32 if out == "fp32" else 0)
    odt = torch.float32 if out == "fp32" else torch.bfloat16

    A_by_M, weights = host_inputs(w)
    packed_h, scales_h, zeros_h = weights
    wb = metrics.weight_bytes(fmt, N, K, group)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 * 1024 * 1024)
    per_step_w = wb * len(Ms)
    R = max(2 * len(Ms), math.ceil(2.0 * l2 / wb))
    R = int(math.ceil(R / len(Ms)) * len(Ms))

    def up(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    packed0 = up(packed_h)
    scales0 = up(scales_h.view(np.int16) if fmt == "int4" else scales_h)
    zeros0 = up(zeros_h)
    pool = [(packed0.clone(), scales0.clone(), None if zeros0 is None else zeros0.clone()) for _ in range(R)]
    del packed0, scales0, zeros0
    # prepacked layout (wq_prepack, an untimed build step like the weight
    # upload): one repacked buffer per weight set
    prepacked = args.layout == "prepacked"
    traffic_key = args.workload + (":prepacked" if prepacked and args.workload + ":prepacked" in KERNEL_SOURCES
                                   else "")
    pre_pool = [wq.prepack(pk, sc, zr, fmt, group) for pk, sc, zr in pool] if prepacked else None
    torch.cuda.synchronize()
    A_d = {M: up(A_by_M[M].view(np.int16)) for M in Ms}
    C_d = {M: torch.empty((M, N), dtype=odt, device=dev) for M in Ms}
    s = torch.cuda.Stream(dev)

    # Launch mode of the timed calls.  The weights are never written by the
    # kernels of the step and the activations are written before the step,
    # so every call may declare its inputs ready (WQ_LAUNCH_INPUTS_READY:
    # the calls overlap end to end and still complete in stream order);
    # "overlap" times the dependent chain (WQ_LAUNCH_OVERLAP: A read after
    # the preceding call completes), "plain" ordinary launches.  The modes
    # not timed as the value are reported beside it.
    overlap = LAUNCH_FLAGS[args.launch](wq)

    def call(M, slot, stream_handle, flags=None):
        fl = overlap if flags is None else flags
        if prepacked:
            st = wq.wq_gemm_prepacked(A_d[M].data_ptr(), pre_pool[slot].buf.data_ptr(), C_d[M].data_ptr(), M, N,
                                      K, fcode, group, None, None, 0, stream_handle, wq.WQ_PATH_AUTO | fl)
            if st != wq.WQ_OK:
                raise wq.WQError(st, "wq_gemm_prepacked")
            return
        pk, sc, zr = pool[slot]
        st = wq.wq_gemm_ex(A_d[M].data_ptr(), pk.data_ptr(), sc.data_ptr(),
                           None if zr is None else zr.data_ptr(), C_d[M].data_ptr(), M, N, K, fcode, group,
                           stream_handle, wq.WQ_PATH_AUTO | fl)
        if st != wq.WQ_OK:
            raise wq.WQError(st, "wq_gemm_ex")

    def capture(nsteps, Ms_used, flags=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                h = torch.cuda.current_stream().cuda_stream
                for i in range(nsteps):
                    for j, M in enumerate(Ms_used):
                        call(M, (i * len(Ms_used) + j) % R, h, flags)
        return g

    # graphs of G steps; G * len(Ms) is a multiple of R so replays rotate seamlessly
    G = R // len(Ms)
    G *= max(1, math.ceil(64 / G))
    with torch.cuda.stream(s):
        for i in range(2):   # eager warm-up outside capture (module load, attributes)
            for j, M in enumerate(Ms):
                call(M, j, s.cuda_stream)
    torch.cuda.synchronize()
    g_full = capture(G, Ms) if args.steps >= G else None
    rem = args.steps % G
    g_rem = capture(rem, Ms) if rem else None

    # warm-up (untimed): at least W steps, and every graph the timed region
    # replays has been replayed before it (a graph's first replay uploads it)
    warm = 0
    while warm < max(1, args.warmup) or warm == 0:
        for g_ in (g_full, g_rem):
            if g_ is not None:
                g_.replay()
                warm += G if g_ is g_full else rem
    torch.cuda.synchronize()

    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    with torch.cuda.stream(s):
        # a short spin ahead of the start event: the graph launches are queued
        # behind it, so host-side submission is not inside the timed window
        torch.cuda._sleep(SPIN_CYCLES)
        ev0.record(s)
        for _ in range(args.steps // G):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    time.sleep(0.15)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, dev)
    launches = args.steps * len(Ms)
    clocks = sampler.summary(t0, t1)

    peaks = measured_peaks()
    avg_launch_s = ms / 1e3 / launches
    if w["bound"] == "hbm":
        value = ws * args.steps * per_step_w / (ms_max / 1e3) / 1e9
        algo = sum(metrics.call_bytes(fmt, M, N, K, group, out) for M in Ms) / len(Ms)
        achieved = algo / avg_launch_s / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(traffic_key),
                "algorithmic_bytes_per_launch": algo, "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        flops = sum(metrics.call_flops(M, N, K) for M in Ms)
        value = ws * args.steps * flops / (ms_max / 1e3) / 1e12
        algo = flops / len(Ms)
        achieved = algo / avg_launch_s / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(traffic_key),
                "algorithmic_flops_per_launch": algo, "peak_source": peaks["source"] + " bf16_tflops (burst)"}

    def replay_ms(g_, n_steps, reps):
        """Milliseconds per step of `reps` replays of a warmed graph of
        n_steps steps (spin kernel ahead of the start event)."""
        g_.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            torch.cuda._sleep(SPIN_CYCLES)
            e0.record(s)
            for _ in range(reps):
                g_.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * n_steps)

    def step_value(ms_step):
        return ws * (per_step_w if w["bound"] == "hbm" else sum(metrics.call_flops(M, N, K) for M in Ms)) / \
            (ms_step / 1e3) / (1e9 if w["bound"] == "hbm" else 1e12)

    # the same steps in the other launch modes, not part of the value
    other_modes = {}
    for mode in LAUNCH_FLAGS:
        if mode == args.launch:
            continue
        g_m = capture(G, Ms, flags=LAUNCH_FLAGS[mode](wq))
        ms_m = replay_ms(g_m, G, max(1, min(args.steps, 2000) // G))
        other_modes[mode] = {"ms_per_step": ms_m, "value": step_value(ms_m), "launch": LAUNCH_DESC[mode]}
        del g_m

    # per-M launch time (separate graphs of one M; not part of the timed steps)
    per_m = {}
    if w["bound"] == "hbm" and len(Ms) > 1:
        for M in Ms:
            entry = {}
            # back-to-back calls of one M over the rotated weights, enough of
            # them per graph that the pipeline's fill at a replay's start is
            # a small share
            n_m = R * max(1, math.ceil(96 / R))
            for mode in ([args.launch] + [m for m in LAUNCH_FLAGS if m != args.launch and m != "plain"]):
                gm = capture(n_m, (M,), flags=LAUNCH_FLAGS[mode](wq))
                us = replay_ms(gm, n_m, max(1, 2000 // n_m)) * 1e3
                del gm
                cb = metrics.call_bytes(fmt, M, N, K, group, out)
                d = {"us_per_call": us, "weight_GBps": wb / us / 1e3, "roofline_frac": cb / us / 1e3 / peaks["hbm_gbs"]}
                if mode == args.launch:
                    entry.update(d)
                else:
                    entry[mode] = d
            per_m[str(M)] = entry

    e2e = run_e2e(args, w, A_by_M, weights, pool, dev, ws, pre_pool)
    fused = fused_gate_up(w, dev, l2) if (w["bound"] == "hbm" and fmt == "int4" and args.launch != "plain") else None
    tensor_core = None
    if args.workload == "decode_int4" and not args.no_tensor_core:
        del pool, pre_pool
        torch.cuda.empty_cache()
        tensor_core = tensor_core_block(args, dev, gpu_id, peaks)

    result = {
        "metric": w["metric"], "value": value, "unit": w["unit"], "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": bench_config(args.workload, ws),
        "setup": {"l2": f"inputs larger than L2: {R} weight sets of {wb / 1e6:.2f} MB rotated "
                        f"({R * wb / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
                  "timing": "CUDA graphs of the timed steps (each replayed once before timing), CUDA events on "
                            "the launching stream, a short spin kernel ahead of the start event",
                  "launch": LAUNCH_DESC[args.launch],
                  "layout": ("prepacked (wq_prepack, untimed build step)" if prepacked else
                             "as given (packed, scales, zeros)")},
        "roofline": roof, "clocks": clocks, "gpu_launches": launches, "e2e": e2e,
        "other_launch_modes": other_modes,
    }
    if per_m:
        result["per_m"] = per_m
    if fused:
        result["fused_gate_up"] = fused
    if tensor_core:
        result["tensor_core"] = tensor_core
    if rank == 0 and ws == 1:
        result["cpu_baseline"] = cpu_baseline(w, A_by_M, weights, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)


def fused_gate_up(w, dev, l2):
    """The decoder's gate/up projection pair (two N x K int4 weights) with the
    SiLU-gated product, per call: one fused call (wq_gemm_fused over the
    interleaved 2N-row weight) against two GEMV calls plus torch's silu and
    multiply.  Graph-timed, chained launches, weights rotated past L2.  Not
    part of the value."""
    import torch
    import weight_only_bit_w4a16_gb300 as wq
    from weight_only_bit_w4a16_gb300 import metrics, synth
    N, K, group, Ms = w["N"], w["K"], w["group"], w["Ms"]
    gate = synth.make_weights("int4", N, K, group, seed=101)
    up = synth.make_weights("int4", N, K, group, seed=102)
    # interleave in groups of 8 rows: 16b..16b+7 gate rows 8b.., 16b+8.. up rows 8b..
    order = np.empty(2 * N, dtype=np.int64)
    o = np.arange(N)
    order[16 * (o // 8) + (o % 8)] = o
    order[16 * (o // 8) + 8 + (o % 8)] = N + o
    fused_h = [np.ascontiguousarray(np.concatenate([g, u])[order]) for g, u in zip(gate, up)]
    wb2 = 2 * metrics.weight_bytes("int4", N, K, group)
    R = max(2, math.ceil(2.0 * l2 / wb2))

    def dev_set(pk, sc, zr):
        return (torch.from_numpy(pk).to(dev), torch.from_numpy(sc.view(np.int16)).to(dev),
                torch.from_numpy(zr).to(dev))
    fused_d = [dev_set(*fused_h) for _ in range(R)]
    gate_d = [dev_set(*gate) for _ in range(R)]
    up_d = [dev_set(*up) for _ in range(R)]
    s = torch.cuda.Stream(dev)
    out = {}
    for M in Ms:
        A = torch.randn(M, K, device=dev).to(torch.bfloat16)
        H = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        G = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        U = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        epi = wq.wq_epilogue(None, None, 1)
        flags = wq.WQ_PATH_AUTO | wq.WQ_LAUNCH_OVERLAP

        def fused_call(i, h):
            pk, sc, zr = fused_d[i % R]
            st = wq.wq_gemm_fused(A.data_ptr(), pk.data_ptr(), sc.data_ptr(), zr.data_ptr(), H.data_ptr(), M,
                                  2 * N, K, wq.WQ_INT4, group, ctypes.byref(epi), None, 0, h, flags)
            if st != wq.WQ_OK:
                raise wq.WQError(st, "wq_gemm_fused")

        def unfused_call(i, h):
            for wset, dst in ((gate_d, G), (up_d, U)):
                pk, sc, zr = wset[i % R]
                st = wq.wq_gemm_ex(A.data_ptr(), pk.data_ptr(), sc.data_ptr(), zr.data_ptr(), dst.data_ptr(), M, N,
                                   K, wq.WQ_INT4, group, h, flags)
                if st != wq.WQ_OK:
                    raise wq.WQError(st, "wq_gemm_ex")
            torch.mul(torch.nn.functional.silu(G), U, out=H)

        res = {}
        for name, fn in (("fused_us", fused_call), ("unfused_us", unfused_call)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                for i in range(2):
                    fn(i, s.cuda_stream)
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s):
                    for i in range(4 * R):
                        fn(i, torch.cuda.current_stream().cuda_stream)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 20
            with torch.cuda.stream(s):
                e0.record(s)
                for _ in range(reps):
                    g.replay()
                e1.record(s)
            torch.cuda.synchronize()
            res[name] = e0.elapsed_time(e1) * 1e3 / (reps * 4 * R)
        res["speedup"] = res["unfused_us"] / res["fused_us"]
        res["fused_weight_GBps"] = wb2 / res["fused_us"] / 1e3
        out[str(M)] = res
    return {"shape": f"gate + up {N} x {K} int4 g{group} each (fused: one {2 * N}-row call, SiLU-gated "
                     f"epilogue; unfused: two calls + torch silu and mul)", "per_m": out}


# ---------------------------------------------------------------------------
# the tensor-core configurations, timed in the default run
# ---------------------------------------------------------------------------
def tensor_core_block(args, dev, gpu_id, peaks):
    """The large-M configurations beside the decode line: the MXFP4 prefill
    (2048 x 3072 x 3072) and the NVFP4 8192^3 GEMM on prepacked weights, and
    one step of the decoder-layer sweep (every projection and the LM head at
    M = 1, 16, 128, 2048).  Each: a warmed CUDA graph of back-to-back calls
    (weight copies rotated past L2), CUDA events with a spin kernel ahead of
    the start, its own clock samples.  Not part of the value."""
    import torch
    import weight_only_bit_w4a16_gb300 as wq
    from weight_only_bit_w4a16_gb300 import metrics
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 * 1024 * 1024)
    s = torch.cuda.Stream(dev)
    out = {}
    # the calls chained as the decode line's are (--launch); the tensor-core
    # kernel takes programmatic dependent launch for launches of up to two
    # waves of tiles
    launch_flags = LAUNCH_FLAGS[args.launch](wq)

    def timed(g_, n_calls, reps):
        g_.replay()
        torch.cuda.synchronize()
        sampler = ClockSampler(gpu_id)
        time.sleep(0.2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.monotonic()
        with torch.cuda.stream(s):
            torch.cuda._sleep(SPIN_CYCLES)
            e0.record(s)
            for _ in range(reps):
                g_.replay()
            e1.record(s)
        torch.cuda.synchronize()
        t1 = time.monotonic()
        time.sleep(0.1)
        sampler.stop()
        return e0.elapsed_time(e1) / (reps * n_calls), sampler.summary(t0, t1)

    for name in ("prefill_mxfp4", "large_nvfp4"):
        w = BENCH_WORKLOADS[name]
        fmt, group, N, K, M = w["fmt"], w["group"], w["N"], w["K"], w["Ms"][0]
        A_by_M, (pk_h, sc_h, zr_h) = host_inputs(w)
        wb = metrics.weight_bytes(fmt, N, K, group)
        R = max(2, math.ceil(2.0 * l2 / wb))
        pk = torch.from_numpy(pk_h).to(dev)
        sc = torch.from_numpy(sc_h).to(dev)
        pres = [wq.prepack(pk, sc, None, fmt, group) for _ in range(R)]
        torch.cuda.synchronize()
        del pk, sc
        A = torch.from_numpy(A_by_M[M].view(np.int16)).view(torch.bfloat16).to(dev)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsb = wq.wq_gemm_workspace_size(M, N, K, wq.FORMATS[fmt], group)
        work = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
        n_calls = R * max(1, math.ceil(8 / R))
        with torch.cuda.stream(s):
            def go(i, h):
                st = wq.wq_gemm_prepacked(A.data_ptr(), pres[i % R].buf.data_ptr(), C.data_ptr(), M, N, K,
                                          wq.FORMATS[fmt], group, None, work.data_ptr(), wsb, h,
                                          wq.WQ_PATH_AUTO | launch_flags)
                if st != wq.WQ_OK:
                    raise wq.WQError(st, name)
            go(0, s.cuda_stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(n_calls):
                    go(i, torch.cuda.current_stream().cuda_stream)
        reps = max(1, math.ceil(0.1 / max(1e-6, n_calls * 2.0 * M * N * K / 1.5e15)))
        ms, clk = timed(g, n_calls, reps)
        flops = 2.0 * M * N * K
        tf = flops / (ms / 1e3) / 1e12
        out[name] = {"M": M, "N": N, "K": K, "format": fmt, "ms_per_call": ms, "tflops": tf, "calls": n_calls * reps,
                     "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                  "frac": tf / peaks["bf16_tflops"], "traffic": profiled_traffic(name + ":prepacked"),
                                  "algorithmic_bytes_per_launch": metrics.call_bytes(fmt, M, N, K, group, "bf16"),
                                  "peak_source": peaks["source"] + " bf16_tflops (burst)"},
                     "clocks": clk, "layout": "prepacked", "rotation": f"{R} weight copies",
                     "launch": LAUNCH_DESC[args.launch] + " (tensor-core kernel: up to two waves of tiles)"}
        del g, pres, A, C, work
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    # one step of the decoder-layer sweep: every projection and the LM head
    # at every M, chained (the small-M calls with their inputs ready)
    w = BENCH_WORKLOADS["layer_sweep"]
    shapes = sweep_shapes(w)
    weights_h, A_h = sweep_inputs(w, shapes)
    pres = {c: wq.prepack(torch.from_numpy(pk).to(dev), torch.from_numpy(sc.view(np.int16)).to(dev),
                          torch.from_numpy(zr).to(dev), "int4", 128) for c, (pk, sc, zr) in weights_h.items()}
    torch.cuda.synchronize()
    A_d = {k: torch.from_numpy(a.view(np.int16)).to(dev) for k, a in A_h.items()}
    C_d = {(M, c): torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in w["Ms"] for c, (N, K) in shapes.items()}
    wsb = max(wq.wq_gemm_workspace_size(M, N, K, wq.WQ_INT4, 128) for M in w["Ms"] for N, K in shapes.values())
    work = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
    flags = LAUNCH_FLAGS[args.launch](wq)

    def step(h):
        for M in w["Ms"]:
            for c, (N, K) in shapes.items():
                st = wq.wq_gemm_prepacked(A_d[(M, K)].data_ptr(), pres[c].buf.data_ptr(), C_d[(M, c)].data_ptr(), M,
                                          N, K, wq.WQ_INT4, 128, None, work.data_ptr(), wsb, h,
                                          wq.WQ_PATH_AUTO | flags)
                if st != wq.WQ_OK:
                    raise wq.WQError(st, f"{c} M={M}")

    with torch.cuda.stream(s):
        step(s.cuda_stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(torch.cuda.current_stream().cuda_stream)
    ms, clk = timed(g, 1, 20)
    bound = sum(roofline_time(M, N, K, peaks)[0] for M in w["Ms"] for N, K in shapes.values())
    flops = sum(2.0 * M * N * K for M in w["Ms"] for N, K in shapes.values())
    out["layer_sweep_step"] = {"calls": len(w["Ms"]) * len(shapes), "ms_per_step": ms,
                               "roofline_ms": bound * 1e3, "pct_of_roofline": 100.0 * bound / (ms / 1e3),
                               "tflops": flops / (ms / 1e3) / 1e12, "steps": 20, "clocks": clk,
                               "launch": LAUNCH_DESC[args.launch] + " for the small-M calls"}
    del g, pres, A_d, C_d, work
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# end-to-end timing: copies in, calls, copies out, pipelined over the steps
# ---------------------------------------------------------------------------
def e2e_pipeline_ms(dev, nsteps, h2d, compute, d2h, nbuf=2, group=16):
    """Milliseconds for nsteps end-to-end steps, max over ranks.  Step i
    copies its inputs in on a copy stream (h2d(i, b)), runs its calls on the
    compute stream (compute(i, b)) and copies its results out on a second
    copy stream (d2h(i, b)), with device buffers b = i mod nbuf: step i's
    copies overlap the neighbouring steps' calls, as a serving loop
    double-buffers them.  Events order each buffer's reuse (step i + nbuf
    writes buffer b only after step i has read its inputs and its results
    are on the host).  Groups of `group` steps are captured in one CUDA graph
    (the three streams forked from and joined to the capturing one) and
    replayed; each replay fills and drains the pipeline once.  Returns the
    milliseconds, the steps timed and the buffer of a replay's last step."""
    import torch
    s_c, s_in, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    group = max(1, min(group, nsteps))

    def body(n):
        fork = torch.cuda.Event()
        fork.record(s_c)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_c = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]
        for i in range(n):
            b = i % nbuf
            if i >= nbuf:
                s_in.wait_event(ev_c[b])      # step i - nbuf has read buffer b's inputs
            with torch.cuda.stream(s_in):
                h2d(i, b)
            ev_in[b].record(s_in)
            s_c.wait_event(ev_in[b])
            if i >= nbuf:
                s_c.wait_event(ev_out[b])     # ... and its results are on the host
            with torch.cuda.stream(s_c):
                compute(i, b)
            ev_c[b].record(s_c)
            s_out.wait_event(ev_c[b])
            with torch.cuda.stream(s_out):
                d2h(i, b)
            ev_out[b].record(s_out)
        for st in (s_in, s_out):
            join = torch.cuda.Event()
            join.record(st)
            s_c.wait_event(join)

    with torch.cuda.stream(s_c):
        body(min(nsteps, 2 * nbuf))      # eager warm-up (module load, first-call work)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_c):
        body(group)
    reps = max(1, nsteps // group)
    with torch.cuda.stream(s_c):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_c):
        e0.record(s_c)
        for _ in range(reps):
            g.replay()
        e1.record(s_c)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1), dev), reps * group, (group - 1) % nbuf


def run_e2e(args, w, A_by_M, weights, pool, dev, ws, pre_pool=None):
    """The same metric through the public API (weight_only_bit_w4a16_gb300.gemm,
    or gemm_prepacked on prepacked weights) from pinned host memory.  Per
    step: one H2D copy of the step's activations (all its calls' A, packed
    in one pinned buffer), the calls chained on device-resident weights
    (uploaded -- and repacked -- once, as a model's weights are), one D2H
    copy of all the step's results -- pipelined over the steps
    (e2e_pipeline_ms).  "serial" reports the same steps issued one after
    another on one stream, and "with_weight_upload" serial steps that also
    upload (and repack) every weight."""
    import torch
    import weight_only_bit_w4a16_gb300 as wq
    from weight_only_bit_w4a16_gb300 import metrics
    fmt, group, Ms, N, K, out = w["fmt"], w["group"], w["Ms"], w["N"], w["K"], w["out"]
    odt = torch.float32 if out == "fp32" else torch.bfloat16
    # one pinned host buffer and one device buffer for all of a step's
    # activations, and likewise for its results; per-call views into them
    a_rows, c_rows = sum(Ms), sum(Ms)
    A_h_all = torch.empty((a_rows, K), dtype=torch.bfloat16).pin_memory()
    C_h_all = torch.empty((c_rows, N), dtype=odt).pin_memory()
    A_d_all = torch.empty((a_rows, K), dtype=torch.bfloat16, device=dev)
    C_d_all = torch.empty((c_rows, N), dtype=odt, device=dev)
    A_d, C_d, r0 = {}, {}, 0
    for M in Ms:
        A_h_all[r0:r0 + M].copy_(torch.from_numpy(A_by_M[M].view(np.int16)).view(torch.bfloat16))
        A_d[M], C_d[M] = A_d_all[r0:r0 + M], C_d_all[r0:r0 + M]
        r0 += M
    s = torch.cuda.Stream(dev)
    R = len(pool)
    steps = max(1, min(args.steps, 2000))
    # Every call is launched as a dependent chain (WQ_LAUNCH_OVERLAP): the
    # step's first call follows the copy of its activations through a full
    # dependency and overlaps only the previous step's last call; the staged
    # kernel serves such chains.  Same GPU, 1000 pipelined steps: 1674 GB/s,
    # against 1484 with every call's inputs declared ready, 1325 with the
    # later two calls of a step ready, and 1079 with the first call plain and
    # the later two ready.
    kw_later = {"overlap": args.launch != "plain"}

    def one(i, upload_weights=None):
        if upload_weights is not None:
            for j, M in enumerate(Ms):
                slot = (i * len(Ms) + j) % R
                pk, sc, zr = pool[slot]
                pk.copy_(upload_weights[0], non_blocking=True)
                sc.copy_(upload_weights[1], non_blocking=True)
                if zr is not None:
                    zr.copy_(upload_weights[2], non_blocking=True)
                if pre_pool is not None:
                    wq.prepack(pk, sc, zr, fmt, group, out=pre_pool[slot].buf)
        A_d_all.copy_(A_h_all, non_blocking=True)
        for j, M in enumerate(Ms):
            slot = (i * len(Ms) + j) % R
            kw = kw_later
            if pre_pool is not None:
                wq.gemm_prepacked(A_d[M], pre_pool[slot], out_dtype=out, out=C_d[M], **kw)
            else:
                pk, sc, zr = pool[slot]
                wq.gemm(A_d[M], pk, sc, zr, fmt, group, out_dtype=out, out=C_d[M], **kw)
        C_h_all.copy_(C_d_all, non_blocking=True)

    def timed(nsteps, upload=None):
        with torch.cuda.stream(s):
            for i in range(3):
                one(i, upload)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for i in range(nsteps):
                one(i, upload)
            e1.record(s)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    h2d = A_h_all.numel() * 2
    d2h = C_h_all.numel() * C_h_all.element_size()
    wbytes = metrics.weight_bytes(fmt, N, K, group)

    def rate(ms_, n_):
        if w["unit"] == "GB/s":
            return ws * n_ * wbytes * len(Ms) / (ms_ / 1e3) / 1e9
        return ws * n_ * sum(metrics.call_flops(M, N, K) for M in Ms) / (ms_ / 1e3) / 1e12

    # pipelined: double-buffered device inputs and outputs, one pinned host
    # output buffer per device one
    A_buf = [A_d_all, torch.empty_like(A_d_all)]
    C_buf = [C_d_all, torch.empty_like(C_d_all)]
    C_hb = [C_h_all, torch.empty(C_h_all.shape, dtype=odt).pin_memory()]
    views = []
    for b_ in range(2):
        vA, vC, r0 = {}, {}, 0
        for M in Ms:
            vA[M], vC[M] = A_buf[b_][r0:r0 + M], C_buf[b_][r0:r0 + M]
            r0 += M
        views.append((vA, vC))

    def p_h2d(i, b_):
        A_buf[b_].copy_(A_h_all, non_blocking=True)

    def p_compute(i, b_):
        vA, vC = views[b_]
        for j, M in enumerate(Ms):
            slot = (i * len(Ms) + j) % R
            kw = kw_later
            if pre_pool is not None:
                wq.gemm_prepacked(vA[M], pre_pool[slot], out_dtype=out, out=vC[M], **kw)
            else:
                pk, sc, zr = pool[slot]
                wq.gemm(vA[M], pk, sc, zr, fmt, group, out_dtype=out, out=vC[M], **kw)

    def p_d2h(i, b_):
        C_hb[b_].copy_(C_buf[b_], non_blocking=True)

    group_steps = R // math.gcd(R, len(Ms)) if R % len(Ms) else R // len(Ms)   # whole weight rotations
    group_steps *= max(1, 16 // group_steps)
    ms_p, n_p, last = e2e_pipeline_ms(dev, steps, p_h2d, p_compute, p_d2h, group=group_steps)
    # the pipeline's last results on the host against the same step run alone
    # (every weight set holds the same weights; the kernels are deterministic)
    with torch.cuda.stream(s):
        A_buf[1 - last].copy_(A_h_all)
        p_compute(0, 1 - last)
    torch.cuda.synchronize()
    checked = bool(torch.equal(C_hb[last].view(torch.int16 if out != "fp32" else torch.int32),
                               C_buf[1 - last].cpu().view(torch.int16 if out != "fp32" else torch.int32)))
    ms = timed(steps)
    res = {"value": rate(ms_p, n_p), "unit": w["unit"], "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": n_p, "pipeline": "copy-in / calls / copy-out streams, double-buffered, "
                                     f"{group_steps} steps per CUDA graph",
           "results_checked": checked,
           "serial": {"value": rate(ms, steps), "steps": steps,
                      "how": "each step's copies and calls in order on one stream, Python-issued"},
           "weights": "device-resident (uploaded once, untimed, as model weights)" +
                      (", prepacked once (untimed)" if pre_pool is not None else ""),
           "launch": ("every call WQ_LAUNCH_OVERLAP (a dependent chain; each step's first call also waits for "
                      "its activations' copy)" if args.launch != "plain" else "plain launches"),
           "api": "gemm_prepacked" if pre_pool is not None else "gemm"}
    # every step also uploads its weights from pinned host memory
    pk_h = torch.from_numpy(weights[0]).pin_memory()
    sc_h = torch.from_numpy(weights[1].view(np.int16) if fmt == "int4" else weights[1]).pin_memory()
    zr_h = None if weights[2] is None else torch.from_numpy(weights[2]).pin_memory()
    steps_w = max(1, min(args.steps, 100))
    ms_w = timed(steps_w, (pk_h, sc_h, zr_h))
    res["with_weight_upload"] = {"value": rate(ms_w, steps_w), "unit": w["unit"],
                                 "h2d_bytes_per_step": h2d + wbytes * len(Ms), "d2h_bytes_per_step": d2h,
                                 "steps": steps_w}
    return res


# ---------------------------------------------------------------------------
# reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = BENCH_WORKLOADS[args.workload]
    A_by_M, weights = host_inputs(w)
    total = args.steps + args.warmup
    cols = oracle_rate(w, A_by_M, weights, budget_s=max(0.01, 90.0 / max(total, 1)))
    for i in range(args.warmup):
        oracle_step_sample(w, cols, A_by_M, weights, seed=100 + i)
    t = 0.0
    covered = 0
    for i in range(args.steps):
        dt, cv = oracle_step_sample(w, cols, A_by_M, weights, seed=i)
        t += dt
        covered += cv
    from weight_only_bit_w4a16_gb300 import metrics
    if w["unit"] == "GB/s":
        value = covered / t / 1e9
    else:
        value = args.steps * sum(metrics.call_flops(M, cols, w["K"]) for M in w["Ms"]) / t / 1e12
    sample = (f"{cols} of {w['N']} output columns of each call of each step "
              f"(M={list(w['Ms'])}, K={w['K']})")
    res = {"impl": "reference", "metric": w["metric"], "value": value, "unit": w["unit"],
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": bench_config(args.workload, ws),
           "cpu_baseline": {"value": value, "unit": w["unit"], "cores": oracle.max_threads(),
                            "kind": "oracle", "sample": sample, "cpu": cpu_model()},
           "e2e": {"value": value, "unit": w["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(res), flush=True)


# ---------------------------------------------------------------------------
# the decoder-layer sweep
# ---------------------------------------------------------------------------
def sweep_shapes(w):
    from weight_only_bit_w4a16_gb300 import synth
    return {c: synth.LAYER_SHAPES[fam] for c, fam in w["calls"]}


def roofline_time(M, N, K, peaks, fmt="int4", group=128, out="bf16"):
    """The roofline bound of one call: max(algorithmic bytes / HBM, flops /
    bf16 tensor peak), in seconds, and which of the two it is."""
    from weight_only_bit_w4a16_gb300 import metrics
    tb = metrics.call_bytes(fmt, M, N, K, group, out) / (peaks["hbm_gbs"] * 1e9)
    tf = metrics.call_flops(M, N, K) / (peaks["bf16_tflops"] * 1e12)
    return (tb, "hbm") if tb >= tf else (tf, "tensor")


def sweep_inputs(w, shapes):
    from weight_only_bit_w4a16_gb300 import synth
    weights = {c: synth.make_weights(w["fmt"], N, K, w["group"], seed=500 + i)
               for i, (c, (N, K)) in enumerate(shapes.items())}
    Ks = sorted({K for _, K in shapes.values()})
    A = {(M, K): synth.draw_A(np.random.default_rng(2000 + M + K), M, K) for M in w["Ms"] for K in Ks}
    return weights, A


def sweep_oracle_sample(w, shapes, weights, A, cols, peaks, seed=0):
    """The oracle on `cols` output columns of every call of one step:
    (seconds, roofline seconds of the sampled work)."""
    import oracle
    rng = np.random.default_rng(seed)
    t = time.perf_counter()
    bound = 0.0
    for M in w["Ms"]:
        for c, (N, K) in shapes.items():
            n = min(cols, N)
            pick = np.sort(rng.choice(N, size=n, replace=False))
            pk, sc, zr = weights[c]
            oracle.gemm(A[(M, K)], pk, sc, zr, w["fmt"], w["group"], cols=pick)
            bound += roofline_time(M, N, K, peaks)[0] * n / N   # the sampled share of the call
    return time.perf_counter() - t, bound


def sweep_oracle_cols(w, shapes, weights, A, peaks, budget_s):
    dt, _ = sweep_oracle_sample(w, shapes, weights, A, 1, peaks)
    return int(max(1, min(64, budget_s / max(dt, 1e-6))))


def run_sweep(args):
    import torch
    import weight_only_bit_w4a16_gb300 as wq

    ws, rank = dist_init(use_cuda=True)
    _, _, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wq.lib()   # fails loudly without the built library
    w = BENCH_WORKLOADS[args.workload]
    fmt, group, Ms = w["fmt"], w["group"], w["Ms"]
    fcode = wq.FORMATS[fmt]
    shapes = sweep_shapes(w)
    peaks = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 * 1024 * 1024)
    prepacked = args.layout == "prepacked"
    overlap = LAUNCH_FLAGS[args.launch](wq)

    weights_h, A_h = sweep_inputs(w, shapes)

    def up(pk, sc, zr):
        return (torch.from_numpy(pk).to(dev), torch.from_numpy(sc.view(np.int16)).to(dev),
                torch.from_numpy(zr).to(dev))

    def weight_set(c):
        d = up(*weights_h[c])
        return wq.prepack(*d, fmt, group) if prepacked else d

    wsets = {c: weight_set(c) for c in shapes}
    A_d = {key: torch.from_numpy(a.view(np.int16)).to(dev) for key, a in A_h.items()}
    C_d = {(M, c): torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in Ms for c, (N, K) in shapes.items()}
    # one workspace serves every call on the stream (completed calls leave its flags zero)
    ws_bytes = max(wq.wq_gemm_workspace_size(M, N, K, fcode, group) for M in Ms for N, K in shapes.values())
    work = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)

    def call(M, c, h, wset, flags=None, C=None):
        N, K = shapes[c]
        fl = wq.WQ_PATH_AUTO | (overlap if flags is None else flags)
        A, Cd = A_d[(M, K)], (C if C is not None else C_d[(M, c)])
        if prepacked:
            st = wq.wq_gemm_prepacked(A.data_ptr(), wset.buf.data_ptr(), Cd.data_ptr(), M, N, K, fcode, group, None,
                                      work.data_ptr(), ws_bytes, h, fl)
        else:
            pk, sc, zr = wset
            st = wq.wq_gemm_ws(A.data_ptr(), pk.data_ptr(), sc.data_ptr(), zr.data_ptr(), Cd.data_ptr(), M, N, K,
                               fcode, group, work.data_ptr(), ws_bytes, h, fl)
        if st != wq.WQ_OK:
            raise wq.WQError(st, f"{c} M={M}")

    def one_step(h, flags=None):
        for M in Ms:
            for c in shapes:
                call(M, c, h, wsets[c], flags)

    def graph_of(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                h = torch.cuda.current_stream().cuda_stream
                for i in range(n):
                    fn(i, h)
        return g

    with torch.cuda.stream(s):
        for _ in range(2):   # eager warm-up outside capture (module load, attributes)
            one_step(s.cuda_stream)
    torch.cuda.synchronize()
    g_step = graph_of(lambda i, h: one_step(h), 1)
    g_plain = graph_of(lambda i, h: one_step(h, 0), 1)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()

    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    with torch.cuda.stream(s):
        ev0.record(s)
        for _ in range(args.steps):
            g_step.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    time.sleep(0.15)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, dev)
    clocks = sampler.summary(t0, t1)
    step_s = ms_max / 1e3 / args.steps
    bound_step = sum(roofline_time(M, N, K, peaks)[0] for M in Ms for N, K in shapes.values())
    value = 100.0 * bound_step / step_s
    flops_step = sum(2 * M * N * K for M in Ms for N, K in shapes.values())

    with torch.cuda.stream(s):
        g_plain.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(max(1, args.steps // 4)):
            g_plain.replay()
        e1.record(s)
    torch.cuda.synchronize()
    plain_step_s = e0.elapsed_time(e1) / 1e3 / max(1, args.steps // 4)

    # each (call shape, M) alone: back-to-back launches over weight copies
    # rotated past L2, graph-timed; k/v and gate/up share a shape
    per_shape = {}
    for c, (N, K) in shapes.items():
        fam = dict(w["calls"])[c]
        if fam in per_shape:
            continue
        wb = sum(a.nbytes for a in weights_h[c])
        R = max(2, math.ceil(2.0 * l2 / wb))
        copies = [wsets[c]] + [weight_set(c) for _ in range(R - 1)]
        n_calls = R * max(1, math.ceil(16 / R))
        per_shape[fam] = {}
        for M in Ms:
            g = graph_of(lambda i, h, M=M: call(M, c, h, copies[i % R]), n_calls)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 3
            with torch.cuda.stream(s):
                e0.record(s)
                for _ in range(reps):
                    g.replay()
                e1.record(s)
            torch.cuda.synchronize()
            t_call = e0.elapsed_time(e1) / 1e3 / (reps * n_calls)
            tb, bound = roofline_time(M, N, K, peaks)
            per_shape[fam][str(M)] = {"N": N, "K": K, "us_per_call": t_call * 1e6,
                                      "tflops": 2 * M * N * K / t_call / 1e12, "weight_GBps": wb / t_call / 1e9,
                                      "bound": bound, "roofline_frac": tb / t_call}
            del g
        del copies
    torch.cuda.synchronize()

    # the dominant kernel of the step: the (shape, M) with the largest time share
    share = {(fam, M): v["us_per_call"] * sum(1 for c2, f2 in w["calls"] if f2 == fam)
             for fam, d in per_shape.items() for M, v in d.items()}
    (dfam, dM), _ = max(share.items(), key=lambda kv: kv[1])
    d = per_shape[dfam][dM]
    M_d = int(dM)
    if d["bound"] == "tensor":
        algo = 2.0 * M_d * d["N"] * d["K"]
        achieved = algo / (d["us_per_call"] * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None, "algorithmic_flops_per_launch": algo,
                "peak_source": peaks["source"] + " bf16_tflops (burst)"}
    else:
        from weight_only_bit_w4a16_gb300 import metrics
        algo = metrics.call_bytes(fmt, M_d, d["N"], d["K"], group, "bf16")
        achieved = algo / (d["us_per_call"] * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_launch": algo,
                "peak_source": peaks["source"] + " hbm_gbs"}
    roof["kernel"] = f"{dfam} {d['N']}x{d['K']} at M={dM}, timed alone (back-to-back launches, weights rotated past L2)"
    roof["step_share"] = share[(dfam, dM)] * 1e-6 / step_s

    e2e = run_sweep_e2e(args, w, shapes, weights_h, A_h, wsets, prepacked, dev, ws, bound_step)

    wbytes_step = sum(a.nbytes for c in shapes for a in weights_h[c])
    result = {
        "metric": w["metric"], "value": value, "unit": w["unit"], "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(args.workload, ws),
        "setup": {"l2": f"inputs larger than L2: a step streams {wbytes_step / 1e6:.0f} MB of weights per M "
                        f"(L2 {l2 / 1e6:.0f} MB); a weight is reused only after all the others",
                  "timing": "CUDA graph of one step, replayed; CUDA events on the launching stream",
                  "launch": LAUNCH_DESC[args.launch] + " (small-M calls; the tensor-core path ignores it)",
                  "layout": ("prepacked (wq_prepack, untimed build step)" if prepacked else
                             "as given (packed, scales, zeros)"),
                  "workspace": f"{ws_bytes} B, shared by the calls (stream-K where the tiles fill the SMs badly)"},
        "roofline": roof, "clocks": clocks, "gpu_launches": args.steps * len(Ms) * len(shapes), "e2e": e2e,
        "step": {"roofline_us": bound_step * 1e6, "measured_us": step_s * 1e6,
                 "tflops": flops_step / step_s / 1e12},
        "plain_launch": {"ms_per_step": plain_step_s * 1e3, "value": 100.0 * bound_step / plain_step_s},
        "per_shape": per_shape,
    }
    if rank == 0 and ws == 1:
        import oracle

        def measure(budget):
            cols = sweep_oracle_cols(w, shapes, weights_h, A_h, peaks, budget)
            dt, bound = sweep_oracle_sample(w, shapes, weights_h, A_h, cols, peaks, seed=1)
            return {"value": 100.0 * bound / dt,
                    "sample": f"{cols} output columns of each of the step's {len(Ms) * len(shapes)} calls, {dt:.1f} s"}

        res = measure(args.cpu_budget)
        single = one_core(measure, max(0.05, args.cpu_budget / 4))
        result["cpu_baseline"] = {"value": res["value"], "unit": w["unit"], "cores": oracle.max_threads(),
                                  "kind": "oracle", "sample": res["sample"], "cpu": cpu_model(),
                                  "one_core": {"value": single["value"], "unit": w["unit"],
                                               "sample": single["sample"]}}
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_sweep_e2e(args, w, shapes, weights_h, A_h, wsets, prepacked, dev, ws, bound_step):
    """The sweep through the public API (gemm_prepacked, or gemm with
    --layout plain) from pinned host memory: per step one H2D copy of all the
    step's activations and one D2H copy of all its results, pipelined over
    the steps (e2e_pipeline_ms); the weights stay device-resident (uploaded,
    and repacked, once)."""
    import torch
    import weight_only_bit_w4a16_gb300 as wq
    Ms = w["Ms"]
    keys = sorted(A_h)
    a_elems = sum(A_h[k].size for k in keys)
    c_elems = sum(M * N for M in Ms for N, _ in shapes.values())
    A_h_all = torch.empty(a_elems, dtype=torch.bfloat16).pin_memory()
    o = 0
    for k in keys:
        n = A_h[k].size
        A_h_all[o:o + n].copy_(torch.from_numpy(A_h[k].view(np.int16).reshape(-1)).view(torch.bfloat16))
        o += n
    nbuf = 2
    A_buf = [torch.empty(a_elems, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    C_buf = [torch.empty(c_elems, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    C_hb = [torch.empty(c_elems, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    views = []
    for b in range(nbuf):
        vA, vC, o = {}, {}, 0
        for k in keys:
            M, K = k
            vA[k] = A_buf[b][o:o + M * K].view(M, K)
            o += M * K
        o = 0
        for M in Ms:
            for c, (N, K) in shapes.items():
                vC[(M, c)] = C_buf[b][o:o + M * N].view(M, N)
                o += M * N
        views.append((vA, vC))
    work = {(M, c): wq.workspace(M, N, K, "int4", device=dev) for M in Ms for c, (N, K) in shapes.items()}
    # wq.workspace grows one cached buffer: take the largest once, for every call
    big = max((t for t in work.values() if t is not None), key=lambda t: t.numel(), default=None)

    def h2d(i, b):
        A_buf[b].copy_(A_h_all, non_blocking=True)

    def compute(i, b):
        vA, vC = views[b]
        j = 0
        for M in Ms:
            for c, (N, K) in shapes.items():
                kw = {"overlap": args.launch != "plain"} if j > 0 else {}   # see run_e2e
                wsp = big if work[(M, c)] is not None else None
                if prepacked:
                    wq.gemm_prepacked(vA[(M, K)], wsets[c], out=vC[(M, c)], workspace=wsp, **kw)
                else:
                    pk, sc, zr = wsets[c]
                    wq.gemm(vA[(M, K)], pk, sc, zr, "int4", out=vC[(M, c)], workspace=wsp, **kw)
                j += 1

    def d2h(i, b):
        C_hb[b].copy_(C_buf[b], non_blocking=True)

    steps = max(1, min(args.steps, 96))
    ms, n, last = e2e_pipeline_ms(dev, steps, h2d, compute, d2h, nbuf=nbuf, group=8)
    # the pipeline's last results on the host against the same step run alone
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        A_buf[1 - last].copy_(A_h_all)
        compute(0, 1 - last)
    torch.cuda.synchronize()
    checked = bool(torch.equal(C_hb[last].view(torch.int16), C_buf[1 - last].cpu().view(torch.int16)))
    return {"value": 100.0 * bound_step / (ms / 1e3 / n), "unit": w["unit"], "results_checked": checked,
            "h2d_bytes_per_step": a_elems * 2, "d2h_bytes_per_step": c_elems * 2, "steps": n,
            "pipeline": "copy-in / calls / copy-out streams, double-buffered, 8 steps per CUDA graph",
            "weights": "device-resident (uploaded once, untimed, as model weights)" +
                       (", prepacked once (untimed)" if prepacked else ""),
            "api": "gemm_prepacked" if prepacked else "gemm"}


def run_reference_sweep(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = BENCH_WORKLOADS[args.workload]
    shapes = sweep_shapes(w)
    peaks = measured_peaks()
    weights_h, A_h = sweep_inputs(w, shapes)
    total = args.steps + args.warmup
    cols = sweep_oracle_cols(w, shapes, weights_h, A_h, peaks, max(0.01, 90.0 / max(total, 1)))
    for i in range(args.warmup):
        sweep_oracle_sample(w, shapes, weights_h, A_h, cols, peaks, seed=100 + i)
    t = bound = 0.0
    for i in range(args.steps):
        dt, b = sweep_oracle_sample(w, shapes, weights_h, A_h, cols, peaks, seed=i)
        t += dt
        bound += b
    value = 100.0 * bound / t
    sample = f"{cols} output columns of each of the step's {len(w['Ms']) * len(shapes)} calls, each step"
    res = {"impl": "reference", "metric": w["metric"], "value": value, "unit": w["unit"],
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": bench_config(args.workload, ws),
           "cpu_baseline": {"value": value, "unit": w["unit"], "cores": oracle.max_threads(),
                            "kind": "oracle", "sample": sample, "cpu": cpu_model()},
           "e2e": {"value": value, "unit": w["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 20000; layer_sweep 300)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 200; layer_sweep 10)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(BENCH_WORKLOADS), default="decode_int4")
    ap.add_argument("--layout", choices=["prepacked", "plain"], default="prepacked",
                    help="weights as given, or repacked once by wq_prepack before timing")
    ap.add_argument("--launch", choices=sorted(LAUNCH_FLAGS), default="ready",
                    help="launch mode of the small-M calls: inputs ready (default), dependent chain, plain")
    ap.add_argument("--no-overlap", action="store_true", help="same as --launch plain")
    ap.add_argument("--no-tensor-core", action="store_true",
                    help="skip the tensor-core block of the default (decode) run")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    args = ap.parse_args(argv)
    if args.no_overlap:
        args.launch = "plain"
    d_steps, d_warm = DEFAULT_STEPS.get(args.workload, (20000, 200))
    args.steps = d_steps if args.steps is None else args.steps
    args.warmup = d_warm if args.warmup is None else args.warmup
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps >= 1 and --warmup >= 0")
    sweep = args.workload == "layer_sweep"
    if args.impl == "reference":
        (run_reference_sweep if sweep else run_reference)(args)
    else:
        (run_sweep if sweep else run_ours)(args)


if __name__ == "__main__":
    main()
