#!/usr/bin/env python
"""Benchmark of the fused SwiGLU + MoE top-k weight + FP8 cast on GB300.

One step = one launch of the fused kernel over one batch of the workload
(default: the largest configuration, T=100003 expanded rows with a ragged
tail, H=3072, 1x128 fp32 scales, E4M3 codes, top-k weights; synthetic inputs
from workloads.py). Prints ONE JSON line on rank 0.

  value     tokens/s over all ranks, device-timed with CUDA events around K
            back-to-back launches (replayed from a CUDA graph) on the
            launching stream, inputs resident in HBM. L2 (129 MB) is defeated
            by rotating several input/output sets whose total is > 2x L2, so
            every launch reads cold inputs and also evicts the previous
            launch's dirty outputs (steady state).
  roofline  algorithmic bytes per launch / average launch time vs the
            measured HBM copy bandwidth; `steady` repeats the launches for at
            least 0.3 s of device time, as a check on the K-step figure.
  per_config  the other large fused workloads (the clamp / UE8M0 one, the
            FP4 one and the 8192-row one), each timed over at least 0.3 s of
            device time with its own clock record (default workload only).
  e2e       the same metric through the host-buffer C-ABI call with pinned
            host buffers: every step copies its inputs host->device and its
            codes and scales back, chunked so the copies overlap the kernel.
  cpu_baseline  the CPU oracle on a bounded sample of rows (rank 0, N=1).

--impl reference times the CPU oracle itself (the only reference this method
has: the pages ship no runnable code), on the same workload and metric.
Multi-GPU (torchrun): every rank runs its own replica of the workload (rows are
independent, so the work shards with no collective); value sums the ranks'
rows over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/s and achieved HBM GB/s (fraction of GB300 peak) for fused SwiGLU+FP8 cast"
DEFAULT_WORKLOAD = "ragged_T100003_H3072_g128"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle sample for cpu_baseline")
    p.add_argument("--scale-layout", choices=["row", "col", "col_packed"], default="row",
                   help="scale layout of the fused op (the host-buffer e2e leg needs row)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--e2e-chunk-rows", type=int, default=2048)
    p.add_argument("--transposed", action="store_true",
                   help="fused workloads: write the codes transposed (tk_swiglu_quant_run_transposed)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-context", action="store_true", help="skip the unfused PyTorch context timing")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-steady", action="store_true",
                   help="skip the >= 0.3 s steady-state timing reported beside the K-step figure")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the other large fused workloads reported under per_config")
    p.add_argument("--jsonl", default=None, help="also append the JSON line to this file")
    return p.parse_args(argv)


# ------------------------------------------------------------ distributed

class Dist:
    def __init__(self, backend: str):
        import torch.distributed as dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = dist if self.world > 1 else None
        if self.dist is not None and not dist.is_initialized():
            dist.init_process_group(backend=backend)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float, device=None) -> float:
        if self.dist is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float, device=None) -> float:
        if self.dist is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


class RankOnly:
    """Rank identity without a process group (the CPU reference arm)."""

    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))


# ----------------------------------------------------------------- clocks

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 50 ms while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(", ") for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ peaks

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ------------------------------------------------------------- CPU oracle

def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it ("model name" on x86; the
    implementer and part numbers on Arm), with the logical core count."""
    import platform
    name = ""
    parts = set()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key == "model name" and not name:
                    name = val
                elif key in ("cpu implementer", "cpu part"):
                    parts.add("%s %s" % (key.replace("cpu ", ""), val))
    except OSError:
        pass
    if not name:
        name = "%s (%s)" % (platform.machine(), ", ".join(sorted(parts))) if parts else platform.machine()
    return "%s, %d logical cores" % (name, os.cpu_count() or 1)


def time_oracle(wl, seconds: float, seed_rows: int = 8) -> dict:
    """Time the CPU oracle on a bounded row sample of the workload: a short
    calibration, then a sample sized to about `seconds` of single-core work."""
    import numpy as np
    import oracle
    from activation_fp8_quantization_gb300 import workloads as wls

    lib = oracle.load()
    small = wl.with_rows(max(8, seed_rows))
    t = time.perf_counter()
    oracle_step(wl, *cpu_inputs(small), lib)()
    per_row = (time.perf_counter() - t) / small.T
    rows = int(max(8, min(wl.T, seconds / max(per_row, 1e-9))))
    rows = max(8, (rows // 8) * 8)
    step = oracle_step(wl, *cpu_inputs(wl.with_rows(rows)), lib)
    t = time.perf_counter()
    step()
    dt = time.perf_counter() - t
    return {"rows": rows, "seconds": dt, "tokens_per_s": rows / dt,
            "gbs": wl.algo_bytes(rows) / dt / 1e9}


def cpu_inputs(wl):
    """(x, w) for the fused op and the cast; (inputs dict, None) for the combine."""
    from activation_fp8_quantization_gb300 import workloads as wls
    if wl.op == "reduce":
        return wls.make_reduce_inputs(wl, "cpu"), None
    if wl.op == "backward":
        x, w, dy = wls.make_backward_inputs(wl, "cpu")
        return x, (w, dy)
    return wls.make_inputs(wl, "cpu")


def _oracle_worker(job):
    """One spawned worker: time the oracle on `rows` rows of the workload."""
    name, rows = job
    import oracle
    from activation_fp8_quantization_gb300 import workloads as wls
    wl = wls.ALL_WORKLOADS[name]
    lib = oracle.load()
    step = oracle_step(wl, *cpu_inputs(wl.with_rows(rows)), lib)
    t = time.perf_counter()
    step()
    return rows, time.perf_counter() - t


def time_oracle_all_cores(wl, seconds: float) -> dict:
    """The oracle over every host core: one spawned process per core (a pool
    started with spawn, so no process is forked from a CUDA context), each
    timing its own share of about `seconds` of work; throughput is all rows
    over the slowest worker's time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    one = time_oracle(wl, 0.5)
    per_row = one["seconds"] / one["rows"]
    rows = int(max(8, min(wl.T, seconds / max(per_row, 1e-9))))
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_worker, [(wl.name, 8)] * cores)          # start-up and library load
        res = pool.map(_oracle_worker, [(wl.name, rows)] * cores)
    slowest = max(dt for _, dt in res)
    total = sum(r for r, _ in res)
    return {"rows": total, "seconds": slowest, "tokens_per_s": total / slowest, "cores": cores}


def oracle_step(wl, x, w, lib):
    """A closure running the CPU oracle once on these rows (inputs prepared)."""
    import oracle
    from activation_fp8_quantization_gb300 import workloads as wls

    if wl.op == "backward":
        xb, db = wls.bf16_bits(x), wls.bf16_bits(w[1])
        wv = w[0].numpy()

        def step():
            oracle.swiglu_backward(xb, db, wv, clamp=wl.clamp, lib=lib)
            oracle.swiglu_quant(xb, wv, wl.group, wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, lib=lib)
        return step
    if wl.op == "reduce":
        d = x
        pos, wt = d["pos"].numpy(), d["w"].numpy()
        if d["y_scale"] is None:
            yb = wls.bf16_bits(d["y"])
            return lambda: oracle.moe_reduce(yb, pos, wt, d["gs"], lib=lib)
        yc, ys = d["y"].numpy(), d["y_scale"].numpy()
        return lambda: oracle.moe_reduce(yc, pos, wt, d["gs"], y_scale=ys, lib=lib)
    if wl.op == "cast":
        y = x.float().numpy()
        if wl.channel:
            return lambda: oracle.quant_cols_f32(y, wl.scale_fmt, wl.out_fmt, lib=lib)
        return lambda: oracle.quant_rows_f32(y, wl.group, wl.scale_fmt, wl.out_fmt, lib=lib)
    xb = wls.bf16_bits(x)
    wn = None if w is None else w.numpy()
    return lambda: oracle.swiglu_quant(xb, wn, wl.group, wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, lib=lib)


def run_reference(args, dist):
    """--impl reference: the CPU oracle as it stands, on the host cores."""
    from activation_fp8_quantization_gb300 import workloads as wls
    import numpy as np
    import oracle

    if dist.rank != 0:
        return 0
    wl = wls.ALL_WORKLOADS[args.workload]
    lib = oracle.load()
    # one step = a bounded sample of the workload; size it so K + W steps fit in ~2 minutes
    calib = time_oracle(wl, 0.5)
    per_row = calib["seconds"] / calib["rows"]
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(8, min(wl.T, budget / per_row)))
    step = oracle_step(wl, *cpu_inputs(wl.with_rows(rows)), lib)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": metric_of(wl), "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64/f32", "data": "synthetic",
        "config": config_of(wl, args.gpus),
        "hbm_gbs": wl.algo_bytes(rows) * args.steps / dt / 1e9,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                         "sample": "%d of %d rows per step, single-threaded C oracle" % (rows, wl.T)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    emit(line, args)
    return 0


def config_of(wl, n: int) -> dict:
    c = {"workload": wl.name, "T": wl.T, "H": wl.H, "group": wl.group, "scale_fmt": wl.scale_fmt,
         "out_fmt": wl.out_fmt, "topk_weights": wl.w_dist is not None, "clamp": wl.clamp,
         "parallelism": "replicas x%d" % n}
    if wl.op != "swiglu":
        c.update({"op": wl.op, "in_dtype": wl.in_dtype})
    if wl.op == "cast":
        c["granularity"] = "per channel (scales [H]; x read twice)" if wl.channel else (
            "per token" if wl.group == 0 else "per 1x%d block" % wl.group)
    return c


def metric_of(wl) -> str:
    if wl.op == "backward":
        return "tokens/s and achieved HBM GB/s (fraction of GB300 peak) for the SwiGLU backward with FP8 recompute"
    if wl.op == "reduce":
        return "tokens/s and achieved HBM GB/s (fraction of GB300 peak) for the weighted top-k combine"
    if wl.op == "cast":
        return "tokens/s and achieved HBM GB/s (fraction of GB300 peak) for the standalone FP8 cast"
    return METRIC


def emit(line: dict, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.jsonl:
        with open(args.jsonl, "a") as f:
            f.write(s + "\n")


# ------------------------------------------------------------- GPU timing

# The large fused workloads reported beside the headline on the same line
# (each timed over at least PER_CONFIG_MIN_MS of device time).
PER_CONFIG = ["moe_T32768_H2048_g128_ue8m0_clamp7", "fp4_T65536_H2048_g32_ue8m0_clamp7", "moe_T8192_H2048_g128"]
PER_CONFIG_MIN_MS = 300.0


def n_sets_for(per_set: int) -> int:
    """Input/output sets to rotate so that the sets not in use hold > 3x L2."""
    return max(2, -(-3 * L2_BYTES // per_set) + 1)


class FusedBench:
    """The fused op or the standalone cast of one workload on one device:
    the plan, `n_sets` rotating input/output sets and a launch(i) that
    enqueues one launch on set i % n_sets through the C ABI."""

    def __init__(self, wl, dev: int, scale_layout: str = "row", transposed: bool = False):
        import torch
        import activation_fp8_quantization_gb300 as tk
        from activation_fp8_quantization_gb300 import _abi
        from activation_fp8_quantization_gb300 import workloads as wls

        self.wl, self.dev = wl, dev
        T = wl.T
        if wl.op == "cast":
            op = tk.QuantCast(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, wl.in_dtype, dev, scale_layout,
                              granularity=wl.gran)
            op.count_clamped = False
        else:
            op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, wl.w_dist is not None, wl.clamp,
                                wl.clamp is not None, dev, scale_layout)
        self.op = op
        self.transposed = transposed and wl.op == "swiglu"
        self.algo = wl.algo_bytes()
        self.n_sets = n_sets_for(self.algo)
        x0, w0 = wls.make_inputs(wl, "cuda")
        self.x0, self.w0 = x0, w0
        q_shape, s_shape, s_dtype = op.output_shapes(T)
        if self.transposed:
            q_shape = (wl.H, tk.tk_swiglu_quant_transposed_size(op.plan, T)[1])
        self.xs, self.ws, qs, ss = [], [], [], []
        for i in range(self.n_sets):
            self.xs.append(x0 if i == 0 else x0.clone())
            self.ws.append(None if w0 is None else (w0 if i == 0 else w0.clone()))
            qs.append(torch.empty(q_shape, dtype=torch.uint8, device=dev))
            ss.append(torch.empty(s_shape, dtype=s_dtype, device=dev))
        self.qs, self.ss = qs, ss
        self.counts = torch.zeros(2, dtype=torch.int64, device=dev) if op.count_clamped else None
        self.workspace, self.ws_bytes = None, 0
        if wl.op == "cast" and op.workspace_bytes(T):
            self.ws_bytes = op.workspace_bytes(T)
            self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.lib = _abi.lib()
        self.stream = torch.cuda.Stream(device=dev)
        self.sh = self.stream.cuda_stream
        self.ptrs = [(self.xs[i].data_ptr(), None if self.ws[i] is None else self.ws[i].data_ptr(),
                      qs[i].data_ptr(), ss[i].data_ptr()) for i in range(self.n_sets)]
        self.cp = None if self.counts is None else self.counts.data_ptr()
        self._tk, self._abi = tk, _abi

    def launch(self, i: int):
        wl, lib, T = self.wl, self.lib, self.wl.T
        xp, wp, qp, spp = self.ptrs[i % self.n_sets]
        if wl.op == "cast":
            st = lib.tk_quant_cast_run_ws(self.op.plan, T, xp, qp, spp,
                                          None if self.workspace is None else self.workspace.data_ptr(),
                                          self.ws_bytes, self.sh)
        elif self.transposed:
            st = lib.tk_swiglu_quant_run_transposed(self.op.plan, T, xp, wp, qp, spp, self.cp, self.sh)
        else:
            st = lib.tk_swiglu_quant_run(self.op.plan, T, xp, wp, qp, spp, self.cp, self.sh)
        if st != 0:
            raise self._tk.TkError(st, self._abi.tk_last_error_message())

    def kernel_name(self) -> str | None:
        if self.transposed:
            return "transpose_quant_kernel"
        if self.wl.op == "swiglu":
            return self.op.launch_info(self.wl.T)["kernel"]
        return self.op.launch_info(self.wl.T)["kernels"]

    def launches_per_step(self) -> int:
        return self.op.launch_info(self.wl.T)["launches"] if self.wl.op == "cast" else 1


def time_steady(fb: FusedBench, min_ms: float, sample_clocks: bool) -> dict:
    """Per-launch device time over back-to-back graph replays totalling at
    least min_ms of device time (after a warm-up), with clocks sampled
    meanwhile. For context beside the K-step headline, and for the per-config
    rows."""
    import torch
    stream, n = fb.stream, fb.n_sets
    with torch.cuda.stream(stream):
        for i in range(3):
            fb.launch(i)
    stream.synchronize()
    chunk = n * max(1, 120 // n)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(chunk):
            fb.launch(i)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
    stream.synchronize()
    per = ev0.elapsed_time(ev1) / chunk
    reps = max(1, int(min_ms / max(per * chunk, 1e-3)) + 1)
    clocks = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if clocks:
        clocks.start()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            graph.replay()
        ev1.record(stream)
    stream.synchronize()
    ms = ev0.elapsed_time(ev1)
    launches = reps * chunk
    us = 1e3 * ms / launches
    gbs = fb.algo / (us / 1e6) / 1e9
    return {"us_per_launch": us, "gbs": gbs, "launches": launches, "device_ms": ms,
            "clocks": clocks.stop() if clocks else None}


def run_ours(args, dist: Dist):
    import torch
    from activation_fp8_quantization_gb300 import workloads as wls

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = dist.local_rank
    torch.cuda.set_device(dev)
    wl = wls.ALL_WORKLOADS[args.workload]
    T = wl.T
    algo = wl.algo_bytes()
    if wl.op == "reduce":
        return run_reduce(args, dist, wl, dev, n_sets_for(algo))
    if wl.op == "backward":
        return run_backward(args, dist, wl, dev, n_sets_for(algo))

    fb = FusedBench(wl, dev, args.scale_layout, args.transposed)
    transposed = fb.transposed
    n_sets = fb.n_sets
    ms, clk = time_graph(args, dist, fb.stream, fb.launch, n_sets, dev)
    ms_max = dist.max(ms, device=dev)
    ms_per_step = ms_max / args.steps
    rows_total = dist.sum(float(T * args.steps), device=dev)
    value = rows_total / (ms_max / 1e3)
    achieved = algo / (ms_per_step / 1e3) / 1e9
    peaks = measured_peaks()
    steady = None
    if not args.no_steady:
        steady = time_steady(fb, PER_CONFIG_MIN_MS, False)
        steady["frac"] = steady["gbs"] / peaks["hbm_gbs"]

    e2e = None
    if not args.no_e2e and wl.op == "swiglu" and args.scale_layout == "row" and not transposed:
        e2e = measure_e2e(fb.op, wl, fb.x0, fb.w0, dev, args, dist)
    context = None
    if dist.rank == 0 and not transposed and not args.no_context:
        context = torch_unfused_context(wl, fb.xs, fb.ws, fb.stream)
    kernel = fb.kernel_name()
    launches = args.steps * fb.launches_per_step()
    del fb
    torch.cuda.empty_cache()

    per_config = None
    if dist.rank == 0 and not args.no_per_config and args.workload == DEFAULT_WORKLOAD and not transposed:
        per_config = {}
        for name in PER_CONFIG:
            pw = wls.ALL_WORKLOADS[name]
            pfb = FusedBench(pw, dev, args.scale_layout)
            r = time_steady(pfb, PER_CONFIG_MIN_MS, True)
            per_config[name] = {"us_per_launch": r["us_per_launch"], "gbs": r["gbs"],
                                "frac": r["gbs"] / peaks["hbm_gbs"], "kernel": pfb.kernel_name(),
                                "tokens_per_s": pw.T / (r["us_per_launch"] / 1e6),
                                "algo_bytes_per_launch": pfb.algo, "launches": r["launches"],
                                "device_ms": r["device_ms"], "clocks": r["clocks"],
                                "traffic": load_traffic(name, family_of(pw)),
                                "l2_write_bytes": load_profile_field(name, family_of(pw), "l2_write_bytes_per_launch")}
            del pfb
            torch.cuda.empty_cache()

    cpu = None
    if dist.rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        r = time_oracle(wl, args.cpu_seconds)
        cpu = {"value": r["tokens_per_s"], "unit": "tokens/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
               "sample": "%d of %d rows of the same workload, single-threaded C oracle, %.1f s"
                         % (r["rows"], wl.T, r["seconds"])}
        ra = time_oracle_all_cores(wl, args.cpu_seconds)
        cpu["all_cores"] = {"value": ra["tokens_per_s"], "unit": "tokens/s", "cores": ra["cores"],
                            "sample": "%d rows per core, one spawned process per core, slowest %.1f s"
                                      % (ra["rows"] // ra["cores"], ra["seconds"])}
    if dist.rank != 0:
        return 0
    fam = family_of(wl, transposed)
    traffic = load_traffic(wl.name, fam)
    line = {
        "metric": metric_of(wl), "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {**config_of(wl, args.gpus), "scale_layout": args.scale_layout,
                   "codes": "transposed [H, ld]" if transposed else "row-major [T, H]",
                   "l2": "inputs larger than L2: %d rotating input/output sets, %.0f MB" % (
                       n_sets, n_sets * algo / 1e6)},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": kernel,
                     "peak_source": peaks["source"], "algo_bytes_per_launch": algo,
                     "l2_write_bytes": load_profile_field(wl.name, fam, "l2_write_bytes_per_launch"),
                     "steady": steady},
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "context_torch_unfused": context,
        "gpu_launches": launches,
        "clocks": clk,
    }
    emit(line, args)
    return 0


def torch_unfused_context(wl, xs, ws, stream, steps: int = 100):
    """The same op as PyTorch eager ops on the device, unfused, for context
    only: silu(g') * u' * w, the group absmax, the scale and a cast to
    torch.float8_e4m3fn (fp32 or power-of-two scales). Not the library's
    path; its codes are not checked here."""
    import torch
    import torch.nn.functional as F
    if wl.op != "swiglu" or wl.out_fmt != "e4m3":
        return None
    T, H = wl.T, wl.H
    g_sz = wl.group or H
    n = len(xs)

    def step(i):
        x = xs[i % n]
        g, u = x[:, :H].float(), x[:, H:].float()
        if wl.clamp is not None:
            g = g.clamp(max=wl.clamp)
            u = u.clamp(-wl.clamp, wl.clamp)
        y = F.silu(g) * u
        if ws[i % n] is not None:
            y = y * ws[i % n][:, None]
        y = y.view(T, H // g_sz, g_sz)
        amax = y.abs().amax(-1, keepdim=True)
        if wl.scale_fmt == "fp32":
            s = amax / 448.0
            s = torch.where(s == 0, torch.ones_like(s), s)
        else:
            s = torch.exp2(torch.ceil(torch.log2(torch.clamp(amax, min=1e-38) / 448.0)))
        return (y / s).to(torch.float8_e4m3fn), s

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"ms_per_step": ms, "value": T / (ms / 1e3), "unit": "tokens/s", "steps": steps,
            "path": "PyTorch eager, unfused (silu, multiply, amax, divide, float8 cast), same inputs"}


def time_graph(args, dist, stream, launch, n_sets, dev):
    """Warm up, capture `chunk` launches in a CUDA graph, replay to exactly
    K launches, timed with events on `stream`; returns (ms, clocks)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(i)
    stream.synchronize()
    chunk = min(args.steps, n_sets * max(1, 600 // n_sets))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(chunk):
            launch(i)
    reps, rem = divmod(args.steps, chunk)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    clocks = ClockSampler(torch.cuda.current_device()) if dist.local_rank == 0 else None
    if clocks:
        clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            graph.replay()
        for i in range(rem):
            launch(i)
        ev1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    return ev0.elapsed_time(ev1), (clocks.stop() if clocks else None)


def run_reduce(args, dist, wl, dev, n_sets):
    """The combine on its workload: tokens/s over rotating input sets."""
    import torch
    import activation_fp8_quantization_gb300 as tk
    from activation_fp8_quantization_gb300 import _abi
    from activation_fp8_quantization_gb300 import workloads as wls

    op = tk.MoeReduce(wl.H, wl.topk, wl.in_dtype, dev)
    d0 = wls.make_reduce_inputs(wl, "cuda")
    sets = []
    for i in range(n_sets):
        d = d0 if i == 0 else {k: (v.clone() if torch.is_tensor(v) else v) for k, v in d0.items()}
        d["out"] = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
        sets.append(d)
    lib = _abi.lib()
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    R = d0["y"].shape[0]
    ptrs = [(d["y"].data_ptr(), None if d["y_scale"] is None else d["y_scale"].data_ptr(),
             d["pos"].data_ptr(), d["w"].data_ptr(), d["out"].data_ptr()) for d in sets]

    def launch(i):
        yp, ysp, pp, wp, op_ = ptrs[i % n_sets]
        st = lib.tk_moe_reduce_run(op.plan, wl.T, yp, ysp, R, pp, wp, d0["gs"], op_, sh)
        if st != 0:
            raise tk.TkError(st, _abi.tk_last_error_message())

    info = op.launch_info(wl.T, d0["y"], d0["y_scale"])
    ms, clk = time_graph(args, dist, stream, launch, n_sets, dev)
    ms_max = dist.max(ms, device=dev)
    ms_per_step = ms_max / args.steps
    value = dist.sum(float(wl.T * args.steps), device=dev) / (ms_max / 1e3)
    algo = wl.algo_bytes()
    achieved = algo / (ms_per_step / 1e3) / 1e9
    peaks = measured_peaks()
    cpu = None
    if dist.rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        r = time_oracle(wl, args.cpu_seconds)
        cpu = {"value": r["tokens_per_s"], "unit": "tokens/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
               "sample": "%d of %d tokens of the same workload, single-threaded C oracle, %.1f s"
                         % (r["rows"], wl.T, r["seconds"])}
    if dist.rank != 0:
        return 0
    line = {
        "metric": metric_of(wl), "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "K": wl.topk, "H": wl.H, "in_fmt": wl.in_dtype,
                   "empty_slots": wl.empty_frac, "parallelism": "replicas x%d" % args.gpus,
                   "l2": "inputs larger than L2: %d rotating input/output sets, %.0f MB" % (
                       n_sets, n_sets * algo / 1e6)},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic(wl.name, PROFILE_FAMILY["reduce"]),
                     "kernel": "moe_reduce_%s" % ("bulk_kernel" if info["kernel"] == "bulk" else "kernel"),
                     "peak_source": peaks["source"], "algo_bytes_per_launch": algo},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clk,
    }
    emit(line, args)
    return 0


def run_backward(args, dist, wl, dev, n_sets):
    """The SwiGLU backward (dx, dw and the recomputed codes and scales) over
    rotating input/output sets."""
    import torch
    import activation_fp8_quantization_gb300 as tk
    from activation_fp8_quantization_gb300 import _abi
    from activation_fp8_quantization_gb300 import workloads as wls

    op = tk.SwigluBackward(wl.H, True, wl.clamp, recompute=dict(group_size=wl.group, scale_fmt=wl.scale_fmt,
                                                                out_fmt=wl.out_fmt, scale_layout=args.scale_layout))
    T = wl.T
    x0, w0, dy0 = wls.make_backward_inputs(wl, "cuda")
    q_shape, s_shape, s_dtype = tk._out_shapes(T, wl.H, wl.group, wl.scale_fmt, wl.out_fmt, args.scale_layout)
    sets = []
    for i in range(n_sets):
        sets.append(dict(
            x=x0 if i == 0 else x0.clone(), w=w0 if i == 0 else w0.clone(), dy=dy0 if i == 0 else dy0.clone(),
            dx=torch.empty((T, 2 * wl.H), dtype=torch.bfloat16, device=dev),
            dw=torch.empty((T,), dtype=torch.float32, device=dev),
            q=torch.empty(q_shape, dtype=torch.uint8, device=dev),
            s=torch.empty(s_shape, dtype=s_dtype, device=dev)))
    ptrs = [tuple(d[k].data_ptr() for k in ("x", "w", "dy", "dx", "dw", "q", "s")) for d in sets]
    lib = _abi.lib()
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream

    def launch(i):
        xp, wp, dyp, dxp, dwp, qp, sp = ptrs[i % n_sets]
        st = lib.tk_swiglu_backward_run(op.plan, T, xp, wp, dyp, dxp, dwp, qp, sp, sh)
        if st != 0:
            raise tk.TkError(st, _abi.tk_last_error_message())

    ms, clk = time_graph(args, dist, stream, launch, n_sets, dev)
    ms_max = dist.max(ms, device=dev)
    ms_per_step = ms_max / args.steps
    value = dist.sum(float(T * args.steps), device=dev) / (ms_max / 1e3)
    algo = wl.algo_bytes()
    achieved = algo / (ms_per_step / 1e3) / 1e9
    peaks = measured_peaks()
    cpu = None
    if dist.rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        r = time_oracle(wl, args.cpu_seconds)
        cpu = {"value": r["tokens_per_s"], "unit": "tokens/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
               "sample": "%d of %d rows of the same workload (backward and recomputed forward), "
                         "single-threaded C oracle, %.1f s" % (r["rows"], T, r["seconds"])}
    if dist.rank != 0:
        return 0
    line = {
        "metric": metric_of(wl), "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {**config_of(wl, args.gpus), "scale_layout": args.scale_layout,
                   "l2": "inputs larger than L2: %d rotating input/output sets, %.0f MB" % (
                       n_sets, n_sets * algo / 1e6)},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic(wl.name, PROFILE_FAMILY["backward"]),
                     "kernel": "swiglu_backward_kernel", "peak_source": peaks["source"],
                     "algo_bytes_per_launch": algo},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clk,
    }
    emit(line, args)
    return 0


def _code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed to one
    space (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The device-code files each profile family's kernels are built from.
FAMILY_SOURCES = {
    "swiglu_quant": ["tk_kernels.cuh", "tk_internal.h", "tk_swiglu_kernels.cu"],
    "quant_cast": ["tk_kernels.cuh", "tk_internal.h", "tk_cast_kernels.cu"],
    "channel_cast": ["tk_kernels.cuh", "tk_internal.h", "tk_channel.h", "tk_channel_kernels.cu"],
    "transposed_quant": ["tk_kernels.cuh", "tk_internal.h", "tk_transpose.h", "tk_transpose_kernels.cu"],
    "moe_reduce": ["tk_kernels.cuh", "tk_internal.h", "tk_reduce.h", "tk_reduce_kernels.cu"],
    "swiglu_backward": ["tk_kernels.cuh", "tk_internal.h", "tk_backward.h", "tk_backward_kernels.cu"],
}


def kernel_source_hash(family: str | None = None) -> str:
    """sha256 over the device code a profile family's kernels are built from
    (every kernel file and header but the host-side tk_api.cu when family is
    None), comments and layout left out, to tell whether a committed ncu
    summary still describes the kernel that runs."""
    import hashlib
    csrc = os.path.join(ROOT, "activation_fp8_quantization_gb300", "csrc")
    if family is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")) and n != "tk_api.cu"]
    else:
        names = FAMILY_SOURCES[family]
    h = hashlib.sha256()
    for name in sorted(names):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()


PROFILE_FAMILY = {"swiglu": "swiglu_quant", "cast": "quant_cast", "channel": "channel_cast", "reduce": "moe_reduce",
                  "backward": "swiglu_backward", "transposed": "transposed_quant"}


def family_of(wl, transposed: bool = False) -> str:
    if transposed:
        return PROFILE_FAMILY["transposed"]
    if wl.op == "cast" and wl.channel:
        return PROFILE_FAMILY["channel"]
    return PROFILE_FAMILY[wl.op]


def load_traffic(workload: str, family: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu summary profiles/<family>_<workload>.md, or None
    if there is none or it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (family, workload))
    fields = {}
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("- ") and ": " in line:
                    k, v = line[2:].strip().split(": ", 1)
                    fields[k.strip("`")] = v.strip().strip("`")
    except OSError:
        return None
    if fields.get("source_sha256") != kernel_source_hash(family):
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def load_profile_field(workload: str, family: str, key: str):
    """Another integer field of the same summary (None if absent or stale)."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (family, workload))
    fields = {}
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("- ") and ": " in line:
                    k, v = line[2:].strip().split(": ", 1)
                    fields[k.strip("`")] = v.strip().strip("`")
    except OSError:
        return None
    if fields.get("source_sha256") != kernel_source_hash(family):
        return None
    try:
        return int(fields[key])
    except (KeyError, ValueError):
        return None


def measure_e2e(op, wl, x0, w0, dev, args, dist: Dist):
    """The same metric through the host-buffer C-ABI calls: inputs start and
    outputs end in page-locked host memory, rotated over sets larger than the
    host's last-level cache. Reported: tk_swiglu_quant_run_mapped, whose
    kernel reads x and w and writes the codes and scales across the host link
    in place. Also timed, as context: tk_swiglu_quant_run_host, which stages
    chunks through device memory with overlapped copies on three streams."""
    import torch
    import activation_fp8_quantization_gb300 as tk
    from activation_fp8_quantization_gb300 import _abi

    T = wl.T
    # sets rotated so that the host's last-level cache never holds a step's
    # inputs (two suffice once a set is several hundred MB)
    n_sets = 4 if wl.algo_bytes() < (512 << 20) else 2
    q_shape, s_shape, s_dtype = op.output_shapes(T)
    xs = [x0.cpu().pin_memory() for _ in range(n_sets)]
    ws = [None if w0 is None else w0.cpu().pin_memory() for _ in range(n_sets)]
    qs = [torch.empty(q_shape, dtype=torch.uint8).pin_memory() for _ in range(n_sets)]
    ss = [torch.empty(s_shape, dtype=s_dtype).pin_memory() for _ in range(n_sets)]
    c_h = torch.zeros(2, dtype=torch.int64).pin_memory() if op.count_clamped else None
    stream = torch.cuda.Stream(device=dev)
    lib = _abi.lib()
    pipe = tk.HostPipe(op, args.e2e_chunk_rows)
    cp = None if c_h is None else c_h.data_ptr()

    def mapped(i):
        k = i % n_sets
        st = lib.tk_swiglu_quant_run_mapped(op.plan, T, xs[k].data_ptr(),
                                            None if ws[k] is None else ws[k].data_ptr(), qs[k].data_ptr(),
                                            ss[k].data_ptr(), cp, stream.cuda_stream)
        if st != 0:
            raise tk.TkError(st, _abi.tk_last_error_message())

    def piped(i):
        k = i % n_sets
        pipe(xs[k], ws[k], q=qs[k], scales=ss[k], clamped_count=c_h, stream=stream)

    def timed(step):
        n = max(1, args.e2e_steps)
        for i in range(3):
            step(i)
        stream.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(n):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        return dist.max(ev0.elapsed_time(ev1), device=dev), n

    ms_p, n = timed(piped)
    ms, n = timed(mapped)
    rows_total = dist.sum(float(T * n), device=dev)
    h2d = xs[0].numel() * xs[0].element_size() + (0 if ws[0] is None else ws[0].numel() * 4) + (
        0 if c_h is None else 16)
    d2h = qs[0].numel() + ss[0].numel() * ss[0].element_size() + (0 if c_h is None else 16)
    return {"value": rows_total / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n,
            "path": "tk_swiglu_quant_run_mapped: the kernel reads x, w and writes codes, scales in page-locked "
                    "host memory across the host link (%d rotating sets)" % n_sets,
            "host_pipe": {"value": rows_total / (ms_p / 1e3), "ms_per_step": ms_p / n,
                          "path": "tk_swiglu_quant_run_host, %d-row chunks through device memory"
                                  % args.e2e_chunk_rows}}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        # rank 0 alone times the CPU oracle; other ranks exit without work
        return run_reference(args, RankOnly())
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        raise SystemExit("--gpus %d does not match the %d process(es) launched: for N > 1 run "
                         "python -m torch.distributed.run --nproc-per-node N bench.py --gpus N" % (args.gpus, world))
    dist = Dist("nccl")
    try:
        return run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
