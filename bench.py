#!/usr/bin/env python3
"""Benchmark of the block-quantized int8 MMQ hot path on GB300.

One step = one pass of the whole path over one batch: quantize the f32 activations to
q8_1, then contract them with the block-quantized weights (f32 out).  Default workload:
Q8_0 attention projection, M=512 tokens, N=K=3584 (the configuration the headline
metric is quoted on).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c1|c2|c3|c3q|layer|sweep]

--workload layer: one 7B GQA transformer layer at 2K-token prefill, x28 layers (the four
activation quantizes and the seven Q4_K projections; attention, norms and activations
are not part of the path and are not timed).  --workload sweep: M in {1 .. 8192} on the
3584x3584 Q4_K projection, one JSON line per M.

--impl reference times the CPU oracle (the plain C fp64 definition) on the host cores
on a bounded sample of the same workload.  Multi-GPU runs (torchrun, one rank per GPU)
are independent replicas of the single-GPU step (weak scaling, no collective on the
data path); the timed region is bracketed by barriers and the max over ranks is taken.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
L2_FALLBACK = 129 * 1024 * 1024  # when the device's L2 size cannot be queried
MIN_TIMED_S = 1.0         # every timed region lasts at least this much device time (clock samples)
MIN_REPLAYS, MAX_REPLAYS = 5, 200000
E2E_MAX_STEPS = 20000

WORKLOADS = {
    "c1": dict(index=1, label="q8_0 MMQ attention-proj M=512 N=3584 K=3584 (quantize + GEMM)"),
    "c2": dict(index=2, label="q4_k MMQ ffn-up M=2048 N=18944 K=3584 (quantize + GEMM)"),
    "c3": dict(index=3, label="q4_k MMQ ffn-down M=2048 N=3584 K=18944 (quantize + GEMM)"),
    "c3q": dict(index=3, label="q8_1 quantize alone M=2048 K=18944", quant_only=True),
}


# ---------------------------------------------------------------------------- helpers

PATH_NAMES = {1: "small-M streams (dp4a; int8 mma.sync)", 2: "tcgen05, codes converted in shared memory",
              3: "tcgen05, codes expanded once per call"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's timed-region length (the job's wall time): an all-reduce MAX
    over the process group (NCCL on GPUs, gloo on the CPU), or ms itself for one rank."""
    if world == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, world: int, ms_max: float, scale: float) -> float:
    """Units processed by all ranks (each rank a replica doing units_per_step per step)
    divided by the slowest rank's time, in units of `scale` per second."""
    return units_per_step * steps * world / (ms_max / 1e3) / scale


# sources each kernel is built from: a kernel's committed DRAM counters stay valid while
# these files are unchanged
_COMMON_SRC = ("ptx.cuh", "common.cuh")
KERNEL_SOURCES = {
    "k_quantize_q8_1": ("quantize.cu", "quant_block.cuh") + _COMMON_SRC,
    "k_mmq_tc": ("gemm_tc.cu", "umma.cuh") + _COMMON_SRC,
    "k_mmq_tcx": ("gemm_expand.cu", "umma.cuh") + _COMMON_SRC,
    "k_expand": ("gemm_expand.cu", "quant_block.cuh", "umma.cuh") + _COMMON_SRC,
    "k_mmq_dp4a_stream": ("gemm_small.cu",) + _COMMON_SRC,
    "k_mmq_i8_stream": ("gemm_small.cu",) + _COMMON_SRC,
    "k_mmq_kq_stream": ("gemm_small.cu",) + _COMMON_SRC,
    "k_mmq_q6_stream": ("gemm_small.cu",) + _COMMON_SRC,
    "k_stream_ksum": ("gemm_small.cu",) + _COMMON_SRC,
    "k_mmq_small_mma": ("gemm_small.cu",) + _COMMON_SRC,
    "k_mmq_small": ("gemm_small.cu",) + _COMMON_SRC,
}


def kernel_source_sha(kernel: str):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_quantized_int8_mmq_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    kernel's current sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(f"{kernel}|{workload}")
    if not e or kernel not in KERNEL_SOURCES or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
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
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle, as it stands, on the host cores, on a bounded sample of the workload."""
    import oracle
    wl = WORKLOADS[args.workload]
    x, w, spec = synth.config_operands(wl["index"])
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    # bounded sample: a band of output rows (all N columns) so that each step is well
    # under a second of CPU work; the quantize of those rows is part of the step
    rows = max(1, min(M, int(args.ref_rows)))
    xs = np.ascontiguousarray(x[:rows])
    cores = oracle.num_threads()
    if wl.get("quant_only"):
        xs = x
    times = []
    ref_steps = args.steps if args.steps > 0 else 10
    for i in range(args.warmup + ref_steps):
        t0 = time.perf_counter()
        xq = oracle.quantize_q8_1(xs)
        if not wl.get("quant_only"):
            oracle.gemm(fmt, xq, w, rows, N, K)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    if wl.get("quant_only"):
        value, unit = (xs.nbytes + xs.size // 32 * 36) / t / 1e9, "GB/s"
        sample = f"full quantize M={M} K={K} per step"
        metric = "q8_1 quantize GB/s"
    else:
        value, unit = 2.0 * rows * N * K / t / 1e12, "TOPS"
        sample = f"rows 0..{rows - 1} of M={M} (all N={N} columns, full K={K}): quantize + contraction per step"
        metric = "MMQ int8 TOPS (2*M*N*K per step: quantize + GEMM)"
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": 0,
        "steps": ref_steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "none", "vs_baseline": None, "dtype": "int64 dots, f64 scales", "data": "synthetic",
        "config": {"workload": wl["label"], "M": M, "N": N, "K": K, "fmt": fmt, "sampled_rows": rows},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(workload: str, budget_s: float):
    """Oracle on the host cores, on a band of rows sized to ~budget_s of CPU time."""
    import oracle
    wl = WORKLOADS[workload]
    x, w, spec = synth.config_operands(wl["index"])
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    if wl.get("quant_only"):
        t0 = time.perf_counter()
        oracle.quantize_q8_1(x)
        dt = time.perf_counter() - t0
        return {"value": (x.nbytes + M * K // 32 * 36) / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
                "kind": "oracle", "sample": f"full quantize M={M} K={K}, {dt:.2f} s"}
    rows = 1
    t0 = time.perf_counter()
    xq = oracle.quantize_q8_1(x[:rows])
    oracle.gemm(fmt, xq, w, rows, N, K)
    dt = time.perf_counter() - t0
    rows = int(max(1, min(M, rows * budget_s / max(dt, 1e-3))))
    # a band of rows; when the whole workload is shorter than the budget, whole passes
    # over it are repeated until the budget is spent
    xs = np.ascontiguousarray(x[:rows])
    passes, t0 = 0, time.perf_counter()
    while True:
        xq = oracle.quantize_q8_1(xs)
        oracle.gemm(fmt, xq, w, rows, N, K)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= 0.8 * budget_s or passes >= 1000:
            break
    band = f"rows 0..{rows - 1} of M={M}" if rows < M else f"all M={M} rows"
    return {"value": 2.0 * rows * N * K * passes / dt / 1e12, "unit": "TOPS", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"{band}, all N={N}, K={K}: quantize + contraction, {passes} pass(es), "
                                        f"{dt:.1f} s"}


# ---------------------------------------------------------------------------- our arm

def oracle_single_core(budget_s: float = 6.0):
    """The oracle on ONE host core (OMP_NUM_THREADS=1, a separate process): c0 in full and a
    band of c1's rows (all N, full K), each quantize + contraction, in TOPS."""
    code = r"""
import json, sys, time
sys.path.insert(0, ROOT)
import numpy as np
import oracle, synth
res = {}
for index, rows in ((0, None), (1, 4)):
    x, w, spec = synth.config_operands(index)
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    xs = np.ascontiguousarray(x if rows is None else x[:rows])
    r = xs.shape[0]
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.gemm(fmt, oracle.quantize_q8_1(xs), w, r, N, K)
        n += 1
        dt = time.perf_counter() - t0
        if dt > BUDGET / 2 or n >= 50:
            break
    res["c%d" % index] = {"value": 2.0 * r * N * K * n / dt / 1e12, "unit": "TOPS", "cores": oracle.num_threads(),
                          "sample": ("all M=%d rows" % M if rows is None else "rows 0..%d of M=%d" % (r - 1, M))
                                    + ", all N=%d, K=%d, %d pass(es), %.2f s" % (N, K, n, dt)}
print(json.dumps(res))
"""
    code = code.replace("ROOT", repr(ROOT)).replace("BUDGET", repr(budget_s))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=120)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"error": f"single-core oracle run failed: {e}"}


def l2_bytes(torch, dev) -> int:
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size) or L2_FALLBACK
    except (AttributeError, RuntimeError):
        return L2_FALLBACK


def timed_replays(step, copies, steps, stream, torch, dev, barrier, clocks, target_s):
    """The K timed steps as CUDA-graph replays (a step is 2 to 4 launches of tens of
    microseconds: launched one by one from Python the host, not the GPU, would set the
    pace).  A graph holds exactly K steps; step i of graph r uses operand copy (r*K + i) %
    copies, and the graphs are replayed in turn, so a copy is reused only after all the
    others (more than 3x L2 between two uses).  The K-step replay is repeated until at
    least `target_s` of device time has passed (and at least MIN_REPLAYS times), each replay
    timed by its own CUDA events on the launching stream; the timed region is bracketed by
    a barrier and a device synchronize on both sides and the clocks are sampled through it.
    A further graph of the same K steps, captured with the library's profiler on and
    replayed once after the timed region, gives each kernel's duration and the launches per
    step without slowing the timed replays.  Returns (median ms per replay, all replay ms,
    per-kernel profile)."""
    import block_quantized_int8_mmq_gb300 as mmq
    ng = copies // math.gcd(steps, copies)
    cap = torch.cuda.Stream(dev)
    prev_prof = mmq.mmq_profile_enable(False)
    graphs = []
    for r in range(ng):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for i in range(steps):
                step((r * steps + i) % copies, cap)
        graphs.append(g)
    mmq.mmq_profile_read(reset=True)
    mmq.mmq_profile_enable(True)
    prof_graph = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.graph(prof_graph, stream=cap):
        for i in range(steps):
            step(i % copies, cap)
    mmq.mmq_profile_enable(prev_prof)
    # upload and first run of every graph, untimed; the first also sizes the replay count
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for g in graphs:
        g.replay()
    b0.record(stream)
    torch.cuda.synchronize(dev)
    per = max(a0.elapsed_time(b0) / len(graphs), 1e-3)
    reps = int(min(MAX_REPLAYS, max(MIN_REPLAYS, math.ceil(target_s * 1e3 / per))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    for k in range(reps):
        ev[k][0].record(stream)
        graphs[k % ng].replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    prof_graph.replay()
    torch.cuda.synchronize(dev)
    prof = mmq.mmq_profile_read(reset=True)
    return statistics.median(ms), ms, prof, clk, reps


def kernel_table(prof, steps):
    kernels = {k: {"launches_per_step": n / steps, "avg_ms": t / n} for k, (n, t) in prof.items()}
    total = sum(t for _, t in prof.values()) / steps
    for k, (n, t) in prof.items():
        kernels[k]["share"] = (t / steps) / total
    return kernels, sum(n for n, _ in prof.values()) / steps


def measure_config(args, workload, rank, world, local, steps, with_e2e=True):
    """One of the named projection workloads: quantize + contraction per step (c1, c2, c3),
    or the quantize alone (c3q).  Returns its bench entry."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", local)
    wl = WORKLOADS[workload]
    x, w, spec = synth.config_operands(wl["index"])
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    quant_only = wl.get("quant_only", False)

    xq_bytes = M * (K // 32) * 36
    set_bytes = x.nbytes + (0 if quant_only else w.nbytes)
    L2 = l2_bytes(torch, dev)
    copies = max(2, -(-3 * L2 // set_bytes))
    xs = [torch.from_numpy(x).to(dev)]
    xs += [xs[0].clone() for _ in range(copies - 1)]
    ws = []
    if not quant_only:
        ws = [torch.from_numpy(w).to(dev)]
        ws += [ws[0].clone() for _ in range(copies - 1)]
    xq = torch.empty(xq_bytes, dtype=torch.uint8, device=dev).view(M, -1)
    out = torch.full((M, N), float("nan"), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(j, s=stream):
        # quantize + contraction: one call (on the expanded tensor-core path the quantize is
        # fused into the activation expansion; xq still receives the q8_1 bytes)
        if quant_only:
            mmq.mmq_quantize_q8_1(xs[j], xq, s)
        else:
            mmq.mmq_linear(xs[j], ws[j], fmt, N, xq=xq, out=out, stream=s)

    for i in range(args.warmup):
        step(i % copies)
    torch.cuda.synchronize(dev)
    assert mmq.mmq_get_device_error(stream) == 0
    path = mmq.mmq_last_path()

    # parity spot check of the warm-up result before timing (proves the kernels ran)
    import oracle
    xr = xq.cpu().numpy()
    assert np.array_equal(xr, oracle.quantize_q8_1(x)), "q8_1 bytes differ from the oracle"
    if not quant_only:
        o = out.cpu().numpy()
        assert not np.isnan(o).any(), "output not written"
        rng = np.random.default_rng(0)
        im, inn = rng.integers(0, M, 256), rng.integers(0, N, 256)
        ref, norm = oracle.gemm_at(fmt, xr, w, M, N, K, im, inn)
        assert np.all(np.abs(o[im, inn] - ref) <= 1e-4 * norm), "GEMM output differs from the oracle"
        out.fill_(float("nan"))

    barrier = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip().isdigit()]
    clocks = ClockSampler(int(visible[local]) if local < len(visible) else local)
    med, all_ms, prof, clk, reps = timed_replays(step, copies, steps, stream, torch, dev, barrier, clocks, args.timed_s)
    if not quant_only:
        assert not torch.isnan(out).any().item(), "timed steps did not write the output"
    assert mmq.mmq_get_device_error(stream) == 0
    kernels, launches_per_step = kernel_table(prof, steps)
    ms_max = max_over_ranks(med, world, dev)

    ops = 2.0 * M * N * K
    peaks = load_peaks()
    if quant_only:
        qbytes = x.nbytes + xq_bytes
        value = whole_job_rate(qbytes, steps, world, ms_max, 1e9)
        unit = "GB/s"
        metric = "q8_1 quantize GB/s (algorithmic bytes: 4 B in + 1.125 B out per value)"
        kname = "k_quantize_q8_1"
        achieved = qbytes / (kernels[kname]["avg_ms"] / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic_for(kname, workload),
                "kernel": kname, "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        value = whole_job_rate(ops, steps, world, ms_max, 1e12)
        unit = "TOPS"
        metric = "MMQ int8 TOPS (2*M*N*K per step: quantize + GEMM)"
        gk = {k: v for k, v in kernels.items() if k.startswith("k_mmq")}
        kname = max(gk, key=lambda k: gk[k]["avg_ms"] * gk[k]["launches_per_step"])
        avg = gk[kname]["avg_ms"]
        if kname in ("k_mmq_tc", "k_mmq_tcx"):
            peak = peaks["bf16_tflops"]
            achieved = ops / (avg / 1e3) / 1e12
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic_for(kname, workload), "kernel": kname,
                    "peak_source": f"{peaks['source']} bf16 burst (f16 tensor rate = bf16 rate)"}
        else:
            wbytes = w.nbytes + xq_bytes + M * N * 4
            gbs = wbytes / (avg / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "traffic": traffic_for(kname, workload), "kernel": kname,
                    "peak_source": peaks["source"] + " hbm_gbs"}

    e2e = None
    if with_e2e:
        e2e = measure_e2e(mmq, torch, dev, stream, x, ws, fmt, M, N, K, quant_only, xq, ops,
                          ms_step=ms_max / steps, target_s=args.timed_s)
    entry = {
        "metric": metric, "value": value, "unit": unit, "ms_per_step": ms_max / steps,
        "tok_per_s": M * steps * world / (ms_max / 1e3), "steps": steps,
        "config": {"workload": wl["label"], "M": M, "N": N, "K": K, "fmt": fmt,
                   "l2": f"rotating {copies} operand copies ({copies * set_bytes / 2**20:.0f} MiB > 3x the "
                         f"{L2 / 2**20:.0f} MiB L2)",
                   "timing": f"CUDA graphs of exactly {steps} steps, replayed {reps} times ({sum(all_ms):.0f} ms of "
                             f"device time); value from the median replay ({min(all_ms):.3f} .. {max(all_ms):.3f} "
                             "ms); kernel durations from one profiled replay after the timed region"},
        "roofline": roof, "kernels": kernels, "path": PATH_NAMES.get(path, "quantize"), "clocks": clk,
        "gpu_launches": int(round(launches_per_step * steps * reps)),
        "gpu_launches_per_step": launches_per_step,
    }
    if e2e:
        entry["e2e"] = e2e
    return entry


def measure_e2e(mmq, torch, dev, stream, x, ws, fmt, M, N, K, quant_only, xq, ops, ms_step, target_s):
    """End to end through the public API: every step copies its input from pinned host
    memory to the device, runs the fused quantize + contraction (or the quantize) and copies
    the result back to pinned host memory.  The three run on their own streams with two
    device buffers each way, ordered by events, so the copies of neighbouring steps overlap
    a step's compute (the way a serving loop feeds the GPU); throughput over as many steps
    as fill MIN_TIMED_S (the same length as the device-side timing)."""
    xh = torch.from_numpy(x).pin_memory()
    res_shape, res_dtype = ((M, K // 32 * 36), torch.uint8) if quant_only else ((M, N), torch.float32)
    oh = torch.empty(res_shape, dtype=res_dtype).pin_memory()
    nbuf = 2
    xd = [torch.empty(x.shape, dtype=torch.float32, device=dev) for _ in range(nbuf)]
    od = [torch.empty(res_shape, dtype=res_dtype, device=dev) for _ in range(nbuf)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    comp_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]
    copies = len(ws) if ws else 1

    def run(n):
        for i in range(n):
            bi = i % nbuf
            if i >= nbuf:
                s_in.wait_event(comp_done[bi])   # the input buffer's last reader is done
            with torch.cuda.stream(s_in):
                xd[bi].copy_(xh, non_blocking=True)
            in_done[bi].record(s_in)
            s_comp.wait_event(in_done[bi])
            if i >= nbuf:
                s_comp.wait_event(out_done[bi])  # the output buffer's last copy is done
            if quant_only:
                mmq.mmq_quantize_q8_1(xd[bi], od[bi], s_comp)
            else:
                mmq.mmq_linear(xd[bi], ws[i % copies], fmt, N, xq=xq, out=od[bi], stream=s_comp)
            comp_done[bi].record(s_comp)
            s_out.wait_event(comp_done[bi])
            with torch.cuda.stream(s_out):
                oh.copy_(od[bi], non_blocking=True)
            out_done[bi].record(s_out)

    for st in (s_in, s_comp, s_out):
        st.wait_stream(stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(3)
    b.record(s_out)
    torch.cuda.synchronize(dev)
    assert np.array_equal(oh.numpy(), od[2 % nbuf].cpu().numpy()), "e2e output not copied back"
    per = max(a.elapsed_time(b) / 3, ms_step)
    n = int(min(E2E_MAX_STEPS, max(20, math.ceil(target_s * 1e3 / per))))
    a.record(s_in)
    s_comp.wait_event(a)
    s_out.wait_event(a)
    run(n)
    b.record(s_out)
    torch.cuda.synchronize(dev)
    e_ms = a.elapsed_time(b)
    h2d, d2h = x.nbytes, oh.numel() * oh.element_size()
    if quant_only:
        val, unit = (x.nbytes + oh.numel()) * n / (e_ms / 1e3) / 1e9, "GB/s"
    else:
        val, unit = ops * n / (e_ms / 1e3) / 1e12, "TOPS"
    return {"value": val, "unit": unit, "steps": n, "ms": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "copy-in, compute and copy-out on three streams, two buffers each way"}


def run_ours(args, rank, world, local):
    """The default line: c1 (the configuration the metric is quoted on) as `value`, and, on
    one GPU, every other config of the metric in `per_config` (c2, c3, c3q, and the 7B
    layer at 2K-token prefill x28)."""
    import torch
    torch.cuda.set_device(local)
    steps = args.steps if args.steps > 0 else 20
    main = measure_config(args, args.workload, rank, world, local, steps)
    line = {
        "metric": main["metric"], "value": main["value"], "unit": main["unit"], "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 codes (exact on f16 tensor cores), f32 scales and output",
        "data": "synthetic (seeded; 7B GQA projection shapes)",
        "config": dict(main["config"], parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "tok_per_s": main["tok_per_s"],
        "roofline": main["roofline"], "kernels": main["kernels"], "path": main["path"], "clocks": main["clocks"],
        "gpu_launches": main["gpu_launches"],
    }
    if "e2e" in main:
        line["e2e"] = main["e2e"]
    if rank == 0 and world == 1 and not args.no_per_config:
        per = {}
        for wlname in ("c2", "c3", "c3q"):
            if wlname != args.workload:
                e = measure_config(args, wlname, rank, world, local, steps)
                e.pop("gpu_launches_per_step", None)
                per[wlname] = e
                torch.cuda.empty_cache()
        per["layer"] = run_layer(args)
        per["small_m"] = run_small_m(args)
        line["per_config"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_budget)
        line["cpu_baseline"]["single_core"] = oracle_single_core()
    return line


SMALL_M_CASES = [("q4_k", 1), ("q4_k", 2), ("q4_k", 8), ("q5_k", 1), ("q5_k", 8), ("q6_k", 1), ("q8_0", 1),
                 ("q8_0", 8)]


def run_small_m(args):
    """The metric's small-M half: the GEMM alone (quantize excluded) at M = 1..8 on the 7B
    ffn-up projection (N = 18944, K = 3584) in each weight format, on the automatic path;
    per line the dominant kernel's HBM roofline (weight + activation + output bytes)."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    N, K = 18944, 3584
    lines = []
    for fmt in ("q4_k", "q5_k", "q6_k", "q8_0"):
        w = (synth.layer_weights(0, "gate", N, K) if fmt == "q4_k"
             else synth.weights(fmt, synth.substream(synth.BASE_SEED + 5, N + K), N, K))
        for (f, M) in SMALL_M_CASES:
            if f != fmt:
                continue
            ln = _sweep_line(mmq, torch, dev, peaks, fmt, M, N, K, w, args, "auto")
            kname = ln["kernels"][0] if ln["kernels"] else None
            ln["roofline"] = {"bound": "hbm", "achieved": ln["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": ln["frac_hbm"], "kernel": kname,
                              "traffic": traffic_for(kname, f"sweep {fmt} M={M} N={N} K={K}") if kname else None}
            lines.append(ln)
        torch.cuda.empty_cache()
    return {"metric": "MMQ GEMM alone at M <= 8, 18944 x 3584", "unit": "GB/s", "lines": lines,
            "config": {"workload": "7B ffn-up projection N=18944 K=3584, M in 1..8, each weight format",
                       "l2": "rotating weight copies >= 3x L2", "cuda_graph": True}}


def _rotating(torch, dev, arr, copies):
    t = torch.from_numpy(arr).to(dev)
    return [t] + [t.clone() for _ in range(copies - 1)]


def run_layer(args):
    """28 layers x (4 activation quantizes + q, k, v, o, gate, up, down GEMMs) at M=2048, Q4_K:
    the metric's "7B-layer prefill ms @2K".  Each layer uses its own device copy of the
    projection weights (the seven matrices are generated once from their seeds and cloned
    per layer), so L2 holds none of them.  The 28 layers are one CUDA graph, replayed until
    at least MIN_TIMED_S of device time has passed; the value is the median replay."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    M, H, F = 2048, 3584, 18944
    L = synth.LAYERS_7B
    w_host = {name: synth.layer_weights(0, name, N, K) for (name, N, K) in synth.LAYER_7B}
    w_dev = [{name: torch.from_numpy(w_host[name]).to(dev) for name in w_host} for _ in range(1)]
    for _ in range(L - 1):
        w_dev.append({name: t.clone() for name, t in w_dev[0].items()})
    acts = [torch.from_numpy(synth.layer_activations(0, M, K, i)).to(dev) for i, K in enumerate((H, H, H, F))]
    xq_h = torch.empty(M * (H // 32) * 36, dtype=torch.uint8, device=dev).view(M, -1)
    xq_f = torch.empty(M * (F // 32) * 36, dtype=torch.uint8, device=dev).view(M, -1)
    outs = {name: torch.empty((M, N), device=dev) for (name, N, K) in synth.LAYER_7B}
    stream = torch.cuda.current_stream(dev)

    def layer(l, stream=stream):
        # each activation is quantized once, by the fused call of its first projection
        # (q, o, gate, down), whose q8_1 output the other projections reuse (k, v, up)
        w = w_dev[l]
        for i, names in enumerate((("q", "k", "v"), ("o",), ("gate", "up"), ("down",))):
            K = F if i == 3 else H
            xq = xq_f if i == 3 else xq_h
            first = names[0]
            mmq.mmq_linear(acts[i], w[first], "q4_k", outs[first].shape[1], xq=xq, out=outs[first], stream=stream)
            for name in names[1:]:
                N = outs[name].shape[1]
                mmq.mmq_gemm_q4_k(xq, w[name], M, N, K, outs[name], stream)

    for l in range(min(L, args.warmup)):
        layer(l)
    torch.cuda.synchronize(dev)
    assert mmq.mmq_get_device_error(stream) == 0
    # the 28 layers as one CUDA graph (a layer is ~20 launches: launched one by one the
    # host would add gaps between them); a second copy captured with the profiler on
    cap = torch.cuda.Stream(dev)
    prev = mmq.mmq_profile_enable(False)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for l in range(L):
            layer(l, stream=cap)
    mmq.mmq_profile_read(reset=True)
    mmq.mmq_profile_enable(True)
    cap.wait_stream(stream)
    prof_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(prof_graph, stream=cap):
        for l in range(L):
            layer(l, stream=cap)
    mmq.mmq_profile_enable(prev)
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    graph.replay()
    b0.record(stream)
    torch.cuda.synchronize(dev)
    assert mmq.mmq_get_device_error(stream) == 0
    reps = int(min(MAX_REPLAYS, max(MIN_REPLAYS, math.ceil(args.timed_s * 1e3 / max(a0.elapsed_time(b0), 1e-3)))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    clocks = ClockSampler(0)
    torch.cuda.synchronize(dev)
    clocks.start()
    for a, b in ev:
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    assert mmq.mmq_get_device_error(stream) == 0
    all_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.median(all_ms)
    prof_graph.replay()
    torch.cuda.synchronize(dev)
    prof = mmq.mmq_profile_read(reset=True)
    kernels, per_pass = kernel_table(prof, 1)
    gemm_ops = 2.0 * M * sum(N * K for (_, N, K) in synth.LAYER_7B) * L
    tcx = kernels.get("k_mmq_tcx")
    roof = None
    if tcx:
        t_tcx = tcx["avg_ms"] * tcx["launches_per_step"]
        achieved = gemm_ops / (t_tcx / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops_sustained"], "traffic": None, "kernel": "k_mmq_tcx",
                "peak_source": f"{peaks['source']} bf16 sustained (a kernel timed inside a long step)",
                "note": "all projections' 2MNK over the summed k_mmq_tcx time of one 28-layer pass"}
    return {"metric": "7B-layer prefill ms @2K (28 layers: quantizes + Q4_K projections)", "value": ms,
            "unit": "ms", "higher_is_better": False, "tok_per_s": M / (ms / 1e3), "tops": gemm_ops / (ms / 1e3) / 1e12,
            "n_gpus": 1, "steps": reps, "warmup": args.warmup, "data": "synthetic (seeded, weights cloned per layer)",
            "config": {"workload": "7B GQA layer x28 at M=2048, Q4_K (attention, norms, SiLU excluded)",
                       "timing": f"the 28 layers captured in one CUDA graph, replayed {reps} times "
                                 f"({sum(all_ms):.0f} ms); value = the median replay ({min(all_ms):.2f} .. "
                                 f"{max(all_ms):.2f} ms); each activation quantized once, fused into its first "
                                 "projection"},
            "roofline": roof, "kernels": kernels, "gpu_launches": int(round(reps * per_pass)), "clocks": clk}


def run_decode(args):
    """One-token decode through 28 7B layers (q, k, v, o, gate, up, down per layer), for each
    weight format: each projection input quantized once by the fused call of its first
    projection, the 28 layers captured in one CUDA graph.  Weights are per-layer device
    copies (3.7 to 6.9 GB per format), so nothing is served from L2; the roofline is the
    weight bytes per token over the measured HBM bandwidth."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    M, H, F = 1, 3584, 18944
    L = synth.LAYERS_7B
    stream = torch.cuda.current_stream(dev)
    acts = [torch.from_numpy(synth.layer_activations(0, M, K, i)).to(dev) for i, K in enumerate((H, H, H, F))]
    xq_h = torch.empty((M, H // 32 * 36), dtype=torch.uint8, device=dev)
    xq_f = torch.empty((M, F // 32 * 36), dtype=torch.uint8, device=dev)
    outs = {name: torch.empty((M, N), device=dev) for (name, N, K) in synth.LAYER_7B}
    lines = []
    for fmt in ("q4_k", "q5_k", "q6_k", "q8_0"):
        w0 = {name: torch.from_numpy(synth.layer_weights(0, name, N, K) if fmt == "q4_k" else
                                     synth.weights(fmt, synth.substream(synth.BASE_SEED + 7, N + K), N, K)).to(dev)
              for (name, N, K) in synth.LAYER_7B}
        w_dev = [w0] + [{name: t.clone() for name, t in w0.items()} for _ in range(L - 1)]
        wbytes = sum(t.numel() for t in w0.values()) * L

        def layer(l, s):
            w = w_dev[l]
            for i, names in enumerate((("q", "k", "v"), ("o",), ("gate", "up"), ("down",))):
                K = F if i == 3 else H
                xq = xq_f if i == 3 else xq_h
                mmq.mmq_linear(acts[i], w[names[0]], fmt, outs[names[0]].shape[1], xq=xq, out=outs[names[0]], stream=s)
                for name in names[1:]:
                    mmq.gemm(fmt, xq, w[name], M, outs[name].shape[1], K, outs[name], s)

        for l in range(min(L, args.warmup)):
            layer(l, stream)
        torch.cuda.synchronize(dev)
        assert mmq.mmq_get_device_error(stream) == 0
        mmq.mmq_profile_read(reset=True)
        prev = mmq.mmq_profile_enable(True)
        layer(0, stream)
        mmq.mmq_profile_enable(prev)
        per_layer = sum(n for n, _ in mmq.mmq_profile_read(reset=True).values())
        prev = mmq.mmq_profile_enable(False)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for l in range(L):
                layer(l, cap)
        mmq.mmq_profile_enable(prev)
        graph.replay()
        torch.cuda.synchronize(dev)
        reps = max(3, args.steps if args.steps > 0 else 50)
        clocks = ClockSampler(0)
        clocks.start()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        assert mmq.mmq_get_device_error(stream) == 0
        ms = a.elapsed_time(b) / reps
        gbs = wbytes / (ms / 1e3) / 1e9
        lines.append({"fmt": fmt, "ms_per_token": ms, "tok_per_s": 1e3 / ms, "weight_bytes_per_token": wbytes,
                      "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "launches_per_token": L * per_layer,
                      "clocks": clk})
        del w_dev, w0, graph
        torch.cuda.empty_cache()
    return {"metric": "7B one-token decode (28 layers of q, k, v, o, gate, up, down projections)", "unit": "mixed",
            "lines": lines, "data": "synthetic (seeded, weights cloned per layer)", "peaks": peaks,
            "config": {"workload": "7B GQA layer x28 at M=1 per weight format (attention, norms, SiLU excluded)",
                       "timing": "28 layers in one CUDA graph, replayed back to back; each projection input "
                                 "quantized once, fused into its first projection"}}


def run_moe(args):
    """Expert-grouped contraction at a mixture-of-experts prefill shape: 2048 tokens, top-8
    of 128 experts (seeded, uniform: each token picks 8 distinct experts), expert matrices
    N=768 x K=2048, i.e. 16384 routed rows.  The grouping (count, scan, scatter) and the
    contraction are timed together, in CUDA-graph replays over rotating weight copies (> 3x
    L2).  The main line is Q4_K on the default (expanded) path; "lines" adds Q4_K on the
    converter kernel and Q6_K experts, and a small batch (16 tokens: 128 routed rows, about
    one per expert) where the automatic choice is the grouped weight stream, beside the
    expanded path forced on the same call; each line with its per-kernel device times."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    lines = [_moe_line(mmq, torch, dev, peaks, fmt, path, args, T)
             for (fmt, path, T) in (("q4_k", "auto", 2048), ("q4_k", "tc", 2048), ("q6_k", "auto", 2048),
                                    ("q4_k", "auto", 16), ("q4_k", "expand", 16), ("q6_k", "auto", 16))]
    main = dict(lines[0])
    main["lines"] = lines
    return main


def _moe_line(mmq, torch, dev, peaks, fmt, path, args, T=2048):
    TOPK, E, N, K = 8, 128, 768, 2048
    R = T * TOPK
    rng = np.random.default_rng(synth.substream(synth.BASE_SEED + 6, 1))
    ids = np.stack([rng.permutation(E)[:TOPK] for _ in range(T)]).reshape(-1).astype(np.int32)
    x = synth.activations(synth.substream(synth.BASE_SEED + 6, 2), T, K, True)
    w = synth.weights(fmt, synth.substream(synth.BASE_SEED + 6, 3), E * N, K)
    copies = max(2, -(-3 * l2_bytes(torch, dev) // w.nbytes))
    ws = _rotating(torch, dev, w, copies)
    xq_tok = mmq.mmq_quantize_q8_1(torch.from_numpy(x).to(dev))
    xq = xq_tok.repeat_interleave(TOPK, dim=0).contiguous()  # row t*8 + s: token t (slot s)
    idd = torch.from_numpy(ids).to(dev)
    out = torch.empty((R, N), device=dev)
    stream = torch.cuda.current_stream(dev)
    prev_path = mmq.mmq_set_path({"tc": mmq.PATH_TC, "expand": mmq.PATH_EXPAND, "small": mmq.PATH_SMALL,
                                  "auto": mmq.PATH_AUTO}[path])
    try:
        for i in range(args.warmup):
            mmq.mmq_gemm_grouped(fmt, xq, idd, ws[i % copies], E, N, K, out=out, stream=stream)
        torch.cuda.synchronize(dev)
        used = PATH_NAMES.get(mmq.mmq_last_path(), "?")
        assert mmq.mmq_get_device_error(stream) == 0
        # spot parity on a few rows against the oracle (the rows' own experts)
        import oracle
        xr = xq.cpu().numpy()
        o = out.cpu().numpy()
        for r in (0, 1, R // 2, R - 1):
            e = int(ids[r])
            ref, norm = oracle.gemm(fmt, np.ascontiguousarray(xr[r:r + 1]),
                                    np.ascontiguousarray(w[e * N:(e + 1) * N]), 1, N, K)
            assert np.all(np.abs(o[r] - ref[0]) <= 1e-4 * norm[0]), f"grouped row {r} differs from the oracle"
        # per-kernel device times of one call (serialised by the profile's events)
        prev_prof = mmq.mmq_profile_enable(True)
        mmq.mmq_profile_read(reset=True)
        mmq.mmq_gemm_grouped(fmt, xq, idd, ws[0], E, N, K, out=out, stream=stream)
        torch.cuda.synchronize(dev)
        kernels = {k: round(v[1] * 1e3, 2) for k, v in sorted(mmq.mmq_profile_read(reset=True).items())}
        mmq.mmq_profile_enable(prev_prof)
        iters = max(20, args.steps)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(iters):
                mmq.mmq_gemm_grouped(fmt, xq, idd, ws[i % copies], E, N, K, out=out, stream=cap)
    finally:
        mmq.mmq_set_path(prev_path)
    graph.replay()
    torch.cuda.synchronize(dev)
    # replays of the graph for at least args.timed_s of device time (the clock samples need
    # a timed region longer than their period); the median replay gives the value
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    replays = max(MIN_REPLAYS, math.ceil(args.timed_s * 1e3 / max(a.elapsed_time(b), 1e-3)))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    clocks = ClockSampler(0)
    clocks.start()
    for (x0, x1) in ev:
        x0.record(stream)
        graph.replay()
        x1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    assert mmq.mmq_get_device_error(stream) == 0
    ms = statistics.median(x0.elapsed_time(x1) for (x0, x1) in ev) / iters
    ops = 2.0 * R * N * K
    # the weights of the experts that received rows (each read at least once per call)
    wbytes = w.nbytes // E * len(np.unique(ids))
    del ws
    return {"metric": "expert-grouped MMQ TOPS (2*R*N*K, R = routed rows)", "value": ops / (ms / 1e3) / 1e12,
            "unit": "TOPS", "ms_per_call": ms, "higher_is_better": True, "fmt": fmt, "path": used,
            "replays": replays,
            "kernels_us": kernels,
            "weight_gbs": wbytes / (ms / 1e3) / 1e9, "frac_hbm_weights": wbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "n_gpus": 1, "steps": iters, "warmup": args.warmup, "data": "synthetic (seeded routing and weights)",
            "config": {"workload": f"MoE {'prefill' if T >= 256 else 'small batch'}: {T} tokens x top-8 of 128 experts, "
                                   f"{fmt.upper()} experts 768x2048" + (", forced path " + path if path != "auto" else ""),
                       "R": R, "E": E, "N": N, "K": K, "l2": f"rotating {copies} weight copies",
                       "cuda_graph": True},
            "clocks": clk}


def run_sweep(args):
    """M sweep on the 3584x3584 Q4_K projection, plus the small-M cases (M = 1, 2, 4, 8)
    on the 18944x3584 and 3584x18944 projections in each weight format: one line per
    case (quantize excluded: the GEMM is timed alone, through CUDA events on the
    launching stream)."""
    import torch
    import block_quantized_int8_mmq_gb300 as mmq
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    lines = []
    cases = [("q4_k", M, 3584, 3584, "q") for M in synth.M_SWEEP]
    # small M on the larger projections too: a 7 MB weight is below the size at which any
    # kernel on this GPU streams at full HBM bandwidth
    for fmt in ("q4_k", "q8_0", "q5_k", "q6_k"):
        cases += [(fmt, M, 18944, 3584, "gate") for M in (1, 2, 4, 8)]
        cases += [(fmt, M, 3584, 18944, "down") for M in (1, 2, 4, 8)]
    for fmt in ("q5_k", "q6_k"):  # on the expanded path
        cases += [(fmt, M, 3584, 3584, "q") for M in (512, 2048)]
    for fmt in ("q4_k", "q8_0"):  # a few tens of rows
        cases += [(fmt, M, 18944, 3584, "gate") for M in (16, 32, 64)]
    # tens to hundreds of rows on the long-K projection: few output tiles, K split (the
    # small-M streams' grids reshaped into one wave up to 40 rows, the expanded path beyond)
    cases += [("q4_k", M, 3584, 18944, "down") for M in (16, 24, 32, 64, 128, 256)]
    cases += [("q8_0", 16, 3584, 18944, "down")]
    # three or four rows around 4864 weight rows (two 16-row tiles per SM), where the
    # automatic small-M choice changes kernel for the K-quants
    for fmt in ("q4_k", "q5_k"):
        cases += [(fmt, M, N, 3584, "wide") for N in (4096, 4864, 5632) for M in (3, 4)]
    if args.only:  # one case, "fmt:M:N:K" (for profiling a single kernel)
        f, m, n, k = args.only.split(":")
        cases = [c for c in cases if c[:4] == (f, int(m), int(n), int(k))]
        if not cases:
            raise SystemExit(f"--only {args.only}: not a sweep case")
    wcache = {}
    for (fmt, M, N, K, proj) in cases:
        if (fmt, proj, N) not in wcache:
            wcache.clear()
            wcache[(fmt, proj, N)] = (synth.layer_weights(0, proj, N, K) if fmt == "q4_k" and proj != "wide"
                                      else synth.weights(fmt, synth.substream(synth.BASE_SEED + 5, N + K), N, K))
        w = wcache[(fmt, proj, N)]
        # up to eight rows of a K % 256 == 0 weight: each small-M kernel that can take the
        # shape, besides the automatic choice (Q6_K: the dp4a stream at any M, in passes of
        # up to four rows)
        routes = [("auto", mmq.SMALL_ROUTE_AUTO)]
        if M <= 8 and K % 256 == 0:
            routes += ([("dp4a", mmq.SMALL_ROUTE_DP4A)] if M <= 4 or fmt == "q6_k" else []) + \
                [("mma", mmq.SMALL_ROUTE_MMA)]
        for (route_name, route) in routes:
            mmq.mmq_debug_small_route(route)
            try:
                lines.append(_sweep_line(mmq, torch, dev, peaks, fmt, M, N, K, w, args, route_name))
            finally:
                mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_AUTO)
    return {"metric": "MMQ M sweep (GEMM only)", "unit": "mixed", "lines": lines,
            "data": "synthetic (seeded)", "peaks": peaks,
            "config": {"workload": "3584x3584 Q4_K projection, M in " + str(synth.M_SWEEP)
                                   + "; M in [1, 2, 4, 8] on 18944x3584 and 3584x18944, Q4_K, Q8_0, Q5_K"
                                   + " and Q6_K; Q5_K and Q6_K 3584x3584 at M = 512, 2048; Q4_K and Q5_K"
                                   + " M = 3, 4 on N = 4096, 4864, 5632 (K = 3584); Q4_K M = 16 ... 256 and"
                                   + " Q8_0 M = 16 on 3584x18944; up to 8 rows: every"
                                   + " small-M kernel that takes the shape (route) besides the automatic one",
                       "l2": "rotating weight copies >= 3x L2", "cuda_graph": True}}


def _sweep_line(mmq, torch, dev, peaks, fmt, M, N, K, w, args, route_name):
    """One sweep case: the GEMM alone, replayed from a CUDA graph, timed by CUDA events."""
    x = synth.activations(synth.substream(synth.BASE_SEED + 4, 7000 + M), M, K, True)
    wbytes = w.nbytes
    copies = max(2, -(-3 * l2_bytes(torch, dev) // (wbytes + x.nbytes)))
    ws = _rotating(torch, dev, w, copies)
    xd = torch.from_numpy(x).to(dev)
    xq = mmq.mmq_quantize_q8_1(xd)
    out = torch.empty((M, N), device=dev)
    stream = torch.cuda.current_stream(dev)
    iters = max(20, args.steps)
    prev_prof = mmq.mmq_profile_enable(True)
    mmq.mmq_profile_read(reset=True)
    mmq.gemm(fmt, xq, ws[0], M, N, K, out, stream)
    torch.cuda.synchronize(dev)
    kernels = sorted(mmq.mmq_profile_read(reset=True))
    mmq.mmq_profile_enable(prev_prof)
    for i in range(args.warmup):
        mmq.gemm(fmt, xq, ws[i % copies], M, N, K, out, stream)
    torch.cuda.synchronize(dev)
    path = mmq.mmq_last_path()
    # the timed launches are captured in one CUDA graph, so the gaps between
    # back-to-back launches (comparable to a small-M kernel) are not counted
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(iters):
            mmq.gemm(fmt, xq, ws[i % copies], M, N, K, out)
    graph.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    assert mmq.mmq_get_device_error(stream) == 0
    ms = a.elapsed_time(b) / iters
    ops = 2.0 * M * N * K
    abytes = wbytes + xq.numel() + M * N * 4
    gbs = abytes / (ms / 1e3) / 1e9
    tops = ops / (ms / 1e3) / 1e12
    del ws
    return {"fmt": fmt, "M": M, "N": N, "K": K, "ms": ms, "tops": tops, "gbs": gbs,
            "tok_per_s": M / (ms / 1e3), "path": PATH_NAMES.get(path, "?"), "route": route_name,
            "kernels": kernels, "frac_hbm": gbs / peaks["hbm_gbs"], "frac_tensor": tops / peaks["bf16_tflops"],
            "algorithmic_bytes": abytes}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="steps per timed replay (0: 20)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["layer", "sweep", "moe", "decode"], default="c1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="only the main workload (no per_config entries)")
    ap.add_argument("--timed-s", type=float, default=MIN_TIMED_S,
                    help="device time each timed region lasts at least (replays of the K-step graph); 0: %d replays"
                         % MIN_REPLAYS)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-rows", type=int, default=32, help="rows per reference-arm step")
    ap.add_argument("--only", default="", help="sweep: run the one case fmt:M:N:K")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()

    if args.impl == "reference":
        if args.workload in ("layer", "sweep", "moe", "decode"):
            args.workload = "c3" if args.workload == "layer" else "c1"
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0

    if args.workload in ("layer", "sweep", "moe", "decode"):
        if rank == 0:
            fn = {"layer": run_layer, "sweep": run_sweep, "moe": run_moe, "decode": run_decode}[args.workload]
            print(json.dumps(fn(args)), flush=True)
        return 0
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
