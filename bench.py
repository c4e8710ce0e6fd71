"""Benchmark of the GB300 TN GEMM (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference|vendor]

A step is one GEMM over one synthetic problem of the named workload (default:
the FP16 M=N=K=4096 GEMM with fp32 accumulation and C).  Inputs live in HBM before
timing starts; successive steps rotate through enough input/output sets that
each step's operands were evicted from L2 by the others.  Under torchrun each
rank runs its own independent problem on its own GPU (weak scaling, no
collective on the data path); the reported value is all ranks' FLOPs over the
slowest rank's time.

--impl reference times the CPU oracle (the deliberately slow fp64 reference) on
a bounded row sample of the same workload per step, on the host cores.

--impl vendor times the vendor library (cuBLAS through torch) on the same workload,
for context (one GPU, a short JSON line with "impl": "vendor").
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense tensor rates relative to bf16 (2.25 PF): fp8 4.5 PF, fp4 13.5 PF
NOMINAL_RATIO = {"f16": 1.0, "bf16": 1.0, "mxfp8": 2.0, "fp8e4m3": 2.0, "fp8e5m2": 2.0, "nvfp4": 6.0}
DTYPE_NAME = {"nvfp4": "nvfp4 (e2m1+e4m3/16)", "mxfp8": "mxfp8 (e4m3+e8m0/32)", "bf16": "bf16",
              "fp8e4m3": "fp8 e4m3", "fp8e5m2": "fp8 e5m2"}
METRIC = "GEMM TFLOPS (FP16 TN, NVFP4/MXFP8 block-scaled) and % of dense tensor peak"
KERNEL_SOURCES = ["cute_layouts_mma_gb300/csrc/gemm_kernel.cuh", "cute_layouts_mma_gb300/csrc/ptx.cuh",
                  "cute_layouts_mma_gb300/csrc/layout.cuh", "cute_layouts_mma_gb300/csrc/gemm_f16.cu",
                  "cute_layouts_mma_gb300/csrc/gemm_bs.cu", "cute_layouts_mma_gb300/csrc/gemm_dense.cu"]


# ----------------------------------------------------------------------------- helpers

def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: whole-line comments and blank lines are left
    out, so that recorded counters stay attached to unchanged code."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                t = line.strip()
                if t and not t.startswith("//"):
                    h.update(t.encode())
                    h.update(b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def workload_bytes(w) -> int:
    """Algorithmic HBM bytes of one launch: read A, B, scales, C once; write D once."""
    if w.kind in ("f16", "bf16"):
        ab = 2 * (w.M + w.N) * w.K
        sf = 0
    elif w.kind in ("fp8e4m3", "fp8e5m2"):
        ab = (w.M + w.N) * w.K
        sf = 0
    elif w.kind == "nvfp4":
        ab = (w.M + w.N) * w.K // 2
        sf = (w.M + w.N) * w.K // 16
    else:
        ab = (w.M + w.N) * w.K
        sf = (w.M + w.N) * w.K // 32
    c = 2 * w.M * w.N if w.with_c else 0
    return ab + sf + c + 2 * w.M * w.N


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU is busy (every
    `period_ms`, each sample time-stamped so that it can be matched to a timed window)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def rows(self):
        import datetime
        out = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 11:
                continue
            try:
                t = datetime.datetime.strptime(f[10], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                out.append({"sm": float(f[1]), "max": float(f[2]), "util": float(f[4]),
                            "hw": f[6], "hwt": f[7], "swt": f[8], "pcap": f[9], "t": t})
            except ValueError:
                continue
        return out

    def median_mhz(self, t0: float, t1: float):
        """Median SM clock of the samples taken between host times t0 and t1 (the sample
        nearest to the window's middle if none falls inside)."""
        rows = self.rows()
        if not rows:
            return None
        inside = [r["sm"] for r in rows if t0 <= r["t"] <= t1]
        if inside:
            return statistics.median(inside)
        mid = 0.5 * (t0 + t1)
        return min(rows, key=lambda r: abs(r["t"] - mid))["sm"]

    def summary(self):
        rows = self.rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        busy = [r for r in rows if r["util"] > 50] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["max"] for r in busy),
                "reasons": sorted(reasons), "samples": len(busy)}


# ----------------------------------------------------------------------------- GPU arm

class GemmRunner:
    """Device-resident rotating problem sets for one workload, plus the launch call."""

    def __init__(self, w, dev, sets: int):
        import torch
        import cute_layouts_mma_gb300 as tg
        from cute_layouts_mma_gb300 import inputs
        self.w, self.dev, self.tg = w, dev, tg
        base = inputs.make_problem(w.kind, w.M, w.N, w.K, w.seed, w.dist, w.with_c)
        self.host = base
        out_dtype = torch.float16 if w.kind == "f16" else torch.bfloat16  # bf16 C / D otherwise
        first = {k: (base[k].to(dev) if base.get(k) is not None else None) for k in ("A", "B", "C", "SFA", "SFB")}
        self.sets = []
        for i in range(sets):
            s = {k: (v if i == 0 or v is None else v.clone()) for k, v in first.items()}
            s["D"] = torch.empty(w.M, w.N, dtype=out_dtype, device=dev)
            self.sets.append(s)
        self.fmt = {"nvfp4": tg.GEMM_FMT_NVFP4, "mxfp8": tg.GEMM_FMT_MXFP8, "fp8e4m3": tg.GEMM_FP8_E4M3,
                    "fp8e5m2": tg.GEMM_FP8_E5M2}.get(w.kind)

    def launch(self, i: int, stream=None):
        s = self.sets[i % len(self.sets)]
        if self.w.kind == "f16":
            self.tg.gemm_f16(s["A"], s["B"], s["C"], s["D"], self.w.accum, stream)
        elif self.w.kind == "bf16":
            self.tg.gemm_bf16(s["A"], s["B"], s["C"], s["D"], stream)
        elif self.w.kind in ("fp8e4m3", "fp8e5m2"):
            self.tg.gemm_fp8(s["A"], s["B"], s["C"], s["D"], self.fmt, stream)
        else:
            self.tg.gemm_block_scaled(s["A"], s["SFA"], s["B"], s["SFB"], s["C"], s["D"], self.fmt, stream)


def vendor_blocked_scales(sf):
    """Row-major scales [rows][cols] (u8) in the vendor library's blocked order: 128-row x
    4-column blocks, row-block major, each block 512 bytes with scale (r, c) at byte
    16 * (r % 32) + 4 * (r // 32) + c -- the 32-lane base tile of the TMEM scale placement
    (local_lane = r % 32, TCol = r // 32, byte = c).  Rows and columns are zero-padded."""
    import torch
    rows, cols = sf.shape
    rb, cb = (rows + 127) // 128, (cols + 3) // 4
    padded = torch.zeros(rb * 128, cb * 4, dtype=sf.dtype, device=sf.device)
    padded[:rows, :cols] = sf
    return padded.view(rb, 4, 32, cb, 4).permute(0, 3, 2, 1, 4).contiguous().flatten()


class VendorRunner:
    """The same workload through the vendor library (cuBLAS via torch), for context only.
    Block-scaled calls take their scales in the vendor's blocked order (converted once,
    outside timing); its block-scaled and FP8 calls add no C."""

    def __init__(self, w, dev, sets: int):
        import torch
        from cute_layouts_mma_gb300 import inputs
        self.w = w
        base = inputs.make_problem(w.kind, w.M, w.N, w.K, w.seed, w.dist, w.with_c)
        out_dtype = torch.float16 if w.kind == "f16" else torch.bfloat16
        self.sets = []
        one = torch.ones((), dtype=torch.float32, device=dev)
        for i in range(sets):
            s = {"D": torch.empty(w.M, w.N, dtype=out_dtype, device=dev), "one": one}
            if w.kind in ("f16", "bf16"):
                s["A"], s["B"] = base["A"].to(dev), base["B"].to(dev)
                s["C"] = base["C"].to(dev) if base.get("C") is not None else None
            elif w.kind in ("fp8e4m3", "fp8e5m2"):
                dt = torch.float8_e4m3fn if w.kind == "fp8e4m3" else torch.float8_e5m2
                s["A"], s["B"] = base["A"].to(dev).view(dt), base["B"].to(dev).view(dt)
            else:
                dt = torch.float4_e2m1fn_x2 if w.kind == "nvfp4" else torch.float8_e4m3fn
                sdt = torch.float8_e4m3fn if w.kind == "nvfp4" else torch.float8_e8m0fnu
                s["A"], s["B"] = base["A"].to(dev).view(dt), base["B"].to(dev).view(dt)
                s["SFA"] = vendor_blocked_scales(base["SFA"].to(dev)).view(sdt)
                s["SFB"] = vendor_blocked_scales(base["SFB"].to(dev)).view(sdt)
            self.sets.append(s)

    def launch(self, i: int, stream=None):
        import torch
        s = self.sets[i % len(self.sets)]
        if self.w.kind in ("f16", "bf16"):
            if s["C"] is not None:
                torch.addmm(s["C"], s["A"], s["B"].t(), out=s["D"])
            else:
                torch.mm(s["A"], s["B"].t(), out=s["D"])
        elif self.w.kind in ("fp8e4m3", "fp8e5m2"):
            torch._scaled_mm(s["A"], s["B"].t(), s["one"], s["one"], out_dtype=torch.bfloat16, out=s["D"])
        else:
            torch._scaled_mm(s["A"], s["B"].t(), s["SFA"], s["SFB"], out_dtype=torch.bfloat16, out=s["D"])


def vendor_arm(args):
    """Times the vendor library on the workload (context for the tables, not a bench line)."""
    import torch
    w = __import__("cute_layouts_mma_gb300.inputs", fromlist=["WORKLOADS"]).WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if w.kind == "f16" and w.accum == 1:
        print(json.dumps({"impl": "vendor", "workload": w.name, "unavailable": "no fp16-accumulate GEMM in torch"}))
        return
    runner = VendorRunner(w, dev, rotating_sets(w))
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            runner.launch(i)
    torch.cuda.synchronize()
    if args.quick:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                runner.launch(i)
        torch.cuda.synchronize()
        print(json.dumps({"impl": "vendor", "quick": True, "workload": w.name}), flush=True)
        return
    peaks, peak_src = load_peaks()
    with ClockSampler(0) as clocks:
        reps = time_repeats(runner, args.steps, stream, args.repeats, graph=not args.no_graph)
    ms = statistics.median(r[0] for r in reps) / args.steps
    rl = roofline(w, ms, peaks, peak_src)
    rl["traffic"] = None  # the recorded DRAM traffic belongs to this library's kernel
    print(json.dumps({"impl": "vendor", "workload": w.name, "ms_per_step": round(ms, 5),
                      "tflops": round(w.flops / (ms * 1e-3) / 1e12, 2), "roofline": rl,
                      "clocks": clocks.summary(),
                      "note": "cuBLAS through torch; block-scaled and FP8 calls add no C"}), flush=True)


def rotating_sets(w) -> int:
    ws = workload_bytes(w)
    return min(1024, max(2, math.ceil(3 * L2_BYTES / ws) + 1)) if ws < 3 * L2_BYTES else 2


def time_steps(runner, steps: int, stream, graph: bool = True) -> float:
    """Milliseconds for `steps` back-to-back launches, CUDA events on `stream`.

    With graph=True the `steps` launches are captured once into a CUDA graph and the
    graph is replayed (once untimed, once timed), so host launch overhead does not
    leak into the measurement; every step is still one launch of the GEMM kernel.
    """
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                runner.launch(i)
        with torch.cuda.stream(stream):
            g.replay()
            start.record(stream)
            g.replay()
            end.record(stream)
        end.synchronize()
        return start.elapsed_time(end)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            runner.launch(i, stream)
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def time_repeats(runner, steps: int, stream, repeats: int, graph: bool = True):
    """The timed region -- `steps` back-to-back launches, captured once into a CUDA graph
    (graph=True) -- run `repeats` times, each bracketed by CUDA events on `stream` and a
    synchronize.  Returns [(ms, host_t0, host_t1)] per repeat; the host times let the
    clock samples be matched to each repeat."""
    import torch
    out = []
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                runner.launch(i)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
    for _ in range(repeats):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.time()
        with torch.cuda.stream(stream):
            start.record(stream)
            if g is not None:
                g.replay()
            else:
                for i in range(steps):
                    runner.launch(i, stream)
            end.record(stream)
        end.synchronize()
        out.append((start.elapsed_time(end), t0, time.time()))
    return out


def peak_for(w, peaks):
    """(bound, peak, unit) of the workload's kernel."""
    if w.kind == "mxfp8" and w.M <= 128:
        return "hbm", peaks["hbm_gbs"], "GB/s"
    return "tensor", peaks["bf16_tflops"] * NOMINAL_RATIO[w.kind], "TFLOP/s"


def roofline(w, ms_per_launch, peaks, peak_src):
    bound, peak, unit = peak_for(w, peaks)
    if bound == "hbm":
        achieved = workload_bytes(w) / (ms_per_launch * 1e-3) / 1e9
    else:
        achieved = w.flops / (ms_per_launch * 1e-3) / 1e12
    extra = {}
    if bound == "tensor":
        # the timed region follows a second of untimed launches, so the part runs at its
        # power-capped steady state: also state the fraction of the sustained peak
        sustained = peaks["bf16_tflops_sustained"] * NOMINAL_RATIO[w.kind]
        extra = {"peak_sustained": sustained, "frac_sustained": round(achieved / sustained, 4)}
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), **extra, "traffic": recorded_traffic(w.name),
            "peak_source": peak_src + (" (bf16 x nominal dtype ratio)"
                                       if bound == "tensor" and NOMINAL_RATIO[w.kind] != 1.0 else ""),
            "algorithmic_bytes": workload_bytes(w), "algorithmic_flops": w.flops}


def e2e_measure(runner, steps: int, stream, h2d_streams: int = 1):
    """Same metric through the public call with host buffers.  Every step copies its
    inputs from pinned host memory to the device, runs the GEMM and reads D back to
    pinned host memory.  Steps are pipelined over the runner's device buffer sets:
    the host -> device copies of step i+1 (spread over `h2d_streams` streams, one
    operand per stream), the GEMM of step i and the device -> host read of step i-1
    run on separate streams, ordered by events; a set is refilled only after the
    read of the step that last used it."""
    import torch
    sets = runner.sets
    nsets = len(sets)
    names = [k for k in ("A", "B", "SFA", "SFB", "C") if sets[0].get(k) is not None]
    host_in = {k: runner.host[k].pin_memory() for k in names}
    host_out = [torch.empty(sets[0]["D"].shape, dtype=sets[0]["D"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    dev = sets[0]["D"].device
    in_streams = [torch.cuda.Stream(dev) for _ in range(h2d_streams)]
    out_stream = torch.cuda.Stream(dev)
    done_reading = [None] * nsets  # event: last D read of the set finished
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    total = steps + 2  # two untimed steps fill the pipeline
    for it in range(total):
        j = it % nsets
        s = sets[j]
        if it == 2:
            start.record(in_streams[0])
            for st in in_streams[1:] + [stream, out_stream]:
                st.wait_stream(in_streams[0])
        copied = []
        for n, k in enumerate(names):
            st = in_streams[n % h2d_streams]
            if done_reading[j] is not None:
                st.wait_event(done_reading[j])
            with torch.cuda.stream(st):
                s[k].copy_(host_in[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st)
            copied.append(ev)
        for ev in copied:
            stream.wait_event(ev)
        runner.launch(j, stream)
        gemm_done = torch.cuda.Event()
        gemm_done.record(stream)
        out_stream.wait_event(gemm_done)
        with torch.cuda.stream(out_stream):
            host_out[it % 2].copy_(s["D"], non_blocking=True)
        done = torch.cuda.Event()
        done.record(out_stream)
        done_reading[j] = done
    end.record(out_stream)
    end.synchronize()
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    return ms, h2d, d2h


def oracle_rows(w, p, rows, exact: bool = False):
    """The oracle's result for the given rows of workload w's problem p (output bits,
    plus the unrounded fp64 sums when exact)."""
    import oracle
    if w.kind == "f16":
        return oracle.gemm_f16(p["A"], p["B"], p.get("C"), rows=rows, exact=exact)
    dense = {"bf16": oracle.BF16, "fp8e4m3": oracle.E4M3, "fp8e5m2": oracle.E5M2}
    if w.kind in dense:
        f = dense[w.kind]
        return oracle.gemm_dense(p["A"], p["B"], p.get("C"), f, f, oracle.BF16, rows=rows, exact=exact)
    fmt = oracle.NVFP4 if w.kind == "nvfp4" else oracle.MXFP8
    return oracle.gemm_block_scaled(fmt, p["A"], p["SFA"], p["B"], p["SFB"], p.get("C"), rows=rows, exact=exact)


def operand_bounds(w, p):
    """max |a| and max |b| of the decoded (scaled) operands."""
    import torch
    if w.kind in ("f16", "bf16"):
        return float(p["A"].float().abs().max()), float(p["B"].float().abs().max())
    if w.kind in ("fp8e4m3", "fp8e5m2", "mxfp8"):
        dt = torch.float8_e5m2 if w.kind == "fp8e5m2" else torch.float8_e4m3fn
        mx = lambda x: float(x.view(dt).float().abs().max())
        if w.kind != "mxfp8":
            return mx(p["A"]), mx(p["B"])
        sf = lambda x: float(2.0 ** (x.max().item() - 127))
        return mx(p["A"]) * sf(p["SFA"]), mx(p["B"]) * sf(p["SFB"])
    sf = lambda x: float(x.view(torch.float8_e4m3fn).float().max())
    return 6.0 * sf(p["SFA"]), 6.0 * sf(p["SFB"])  # E2M1 magnitudes reach 6


def parity_of(w, p, rows, d64, D):
    """GPU output rows against the oracle's exact sums: |D - exact| <= 1e-3*sqrt(K)*max|a|*max|b|
    plus half an output ulp (the tolerance the parity tests use)."""
    import numpy as np
    import torch
    got = D[rows].float().cpu().double().numpy()
    err = np.abs(got - d64)
    a, b = operand_bounds(w, p)
    tol = 1e-3 * math.sqrt(w.K) * a * b
    mbits, emin = (10, -14) if w.kind == "f16" else (7, -126)
    half_ulp = 0.5 * 2.0 ** (np.floor(np.log2(np.maximum(np.abs(d64), 2.0 ** emin))) - mbits)
    return {"rows": len(rows), "max_abs_err": float(err.max()), "tolerance": tol,
            "ok": bool((err <= tol + half_ulp).all() and np.isfinite(got).all()),
            "rule": "|D - exact| <= 1e-3*sqrt(K)*max|a|*max|b| + half an output ulp, on the cpu_baseline rows"}


def cpu_baseline(w, budget_s: float):
    """The oracle, as it stands, on a row sample of the workload; TFLOP/s."""
    import numpy as np
    import oracle
    from cute_layouts_mma_gb300 import inputs
    p = inputs.make_problem(w.kind, w.M, w.N, w.K, w.seed, w.dist, w.with_c)

    out = {}

    def run(rows):
        t0 = time.perf_counter()
        out["d16"], out["d64"] = oracle_rows(w, p, rows, exact=True)
        return time.perf_counter() - t0

    threads = oracle.num_threads()
    probe_rows = list(range(min(w.M, threads)))
    t_probe = run(probe_rows)
    per_row = t_probe / len(probe_rows)
    nrows = int(min(w.M, max(len(probe_rows), budget_s / per_row)))
    rng = np.random.default_rng(0)
    rows = sorted(rng.choice(w.M, size=nrows, replace=False).tolist())
    t = run(rows)
    tflops = 2.0 * nrows * w.N * w.K / t / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{nrows} of {w.M} output rows (all N columns), fp64 oracle, {t:.1f} s"}, t, \
        (p, rows, out["d64"])


def reduce_max(value: float, world: int, device) -> float:
    """Max of a per-rank value over all ranks (the slowest rank's step time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job TFLOP/s: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def gpu_arm(args):
    import torch
    import torch.distributed as dist
    from cute_layouts_mma_gb300 import inputs
    rank, local_rank, world = env_rank()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = inputs.WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    runner = GemmRunner(w, dev, rotating_sets(w))
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    with ClockSampler(local_rank) as clocks:
        for i in range(args.warmup):
            with torch.cuda.stream(stream):
                runner.launch(i, stream)
        torch.cuda.synchronize()
        # extra untimed warm-up so the clocks settle and the sampler sees load
        t0 = time.perf_counter()
        while not args.quick and time.perf_counter() - t0 < 1.0:
            time_steps(runner, 20, stream, graph=False)
        barrier()
        torch.cuda.synchronize()
        reps = time_repeats(runner, args.steps, stream, 1 if args.quick else args.repeats, graph=not args.no_graph)
        torch.cuda.synchronize()
        barrier()
    rep_ms = [r[0] / args.steps for r in reps]
    ms = reduce_max(statistics.median(rep_ms), world, dev)
    repeats = []
    for (total, t0, t1), m in zip(reps, rep_ms):
        mhz = clocks.median_mhz(t0, t1)
        repeats.append({"ms_per_step": round(m, 5), "sm_mhz": mhz,
                        "us_x_ghz": round(m * 1e3 * mhz / 1e3, 2) if mhz else None})
    assert runner.tg.gemm_last_device_error() == runner.tg.GEMM_OK

    if args.quick:  # profiling runs: only the W + K launches above
        if rank == 0:
            print(json.dumps({"quick": True, "workload": w.name, "ms_per_step": ms,
                              "tflops": world * w.flops / (ms * 1e-3) / 1e12}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    e2e_ms, h2d, d2h = e2e_measure(runner, max(3, min(args.steps, 20)), stream)
    value = job_value(world, w.flops, ms)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("f16" if w.accum == 0 else "f16 (f16 accumulate)") if w.kind == "f16" else DTYPE_NAME[w.kind],
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "with_c": w.with_c,
                   "accum": "f32" if w.accum == 0 else "f16",
                   "l2": f"{len(runner.sets)} rotating input/output sets ({workload_bytes(w) * len(runner.sets) >> 20} MiB) so every step's operands are cold in L2",
                   "parallelism": f"independent problem per GPU x{world}"},
        "roofline": roofline(w, ms, peaks, peak_src),
        "clocks": clocks.summary(),
        "e2e": {"value": round(world * w.flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "method": "per step: pinned host -> device copy of A, B (and C / scales), the GEMM, device -> "
                          "pinned host read of D; steps pipelined over the device buffer sets (copies of "
                          "step i+1, GEMM of step i and read of step i-1 overlap on three streams)"},
        "gpu_launches": args.steps * len(reps),
        "timing": (f"{args.repeats} repeats of the K launches ("
                   + ("CUDA-graph replay" if not args.no_graph else "back-to-back launches")
                   + "); value and ms_per_step from the median repeat"),
        "repeats": repeats,
        "repeat_spread": {"min_ms": round(min(rep_ms), 5), "median_ms": round(statistics.median(rep_ms), 5),
                          "max_ms": round(max(rep_ms), 5)},
    }
    if rank == 0 and world == 1 and not args.no_extras:
        extras = {}
        for name, ww in inputs.WORKLOADS.items():
            if name == w.name:
                continue
            r = GemmRunner(ww, dev, rotating_sets(ww))
            for i in range(3):
                r.launch(i, stream)
            torch.cuda.synchronize()
            n = 30 if ww.flops > 1e10 else 200
            mse = time_steps(r, n, stream, graph=not args.no_graph) / n
            extras[name] = {"ms": round(mse, 5), "tflops": round(ww.flops / (mse * 1e-3) / 1e12, 2),
                            "roofline": roofline(ww, mse, peaks, peak_src)}
            del r
            torch.cuda.empty_cache()
        assert runner.tg.gemm_last_device_error() == runner.tg.GEMM_OK
        line["per_workload"] = extras
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, (p, rows, d64) = cpu_baseline(w, args.cpu_seconds)
        line["cpu_baseline"] = cb
        # the timed launches' own output (set 0), checked on the oracle's rows
        line["parity"] = parity_of(w, p, rows, d64, runner.sets[0]["D"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def reference_arm(args):
    """The CPU oracle as the reference implementation, timed per step on a row sample."""
    rank, _, world = env_rank()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from cute_layouts_mma_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    p = inputs.make_problem(w.kind, w.M, w.N, w.K, w.seed, w.dist, w.with_c)
    threads = oracle.num_threads()

    def run(rows):
        oracle_rows(w, p, rows)

    probe = list(range(min(w.M, threads)))
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    total_steps = args.steps + args.warmup
    rows_per_step = int(max(1, min(w.M, args.reference_seconds / total_steps / per_row)))
    rng = np.random.default_rng(0)
    samples = [sorted(rng.choice(w.M, size=rows_per_step, replace=False).tolist()) for _ in range(total_steps)]
    for i in range(args.warmup):
        run(samples[i])
    t0 = time.perf_counter()
    for i in range(args.steps):
        run(samples[args.warmup + i])
    t = time.perf_counter() - t0
    ms = t * 1e3 / args.steps
    value = 2.0 * rows_per_step * w.N * w.K / (ms * 1e-3) / 1e12
    sample = f"{rows_per_step} of {w.M} output rows per step (all N columns), fp64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of K steps each (value: the median one); clocks sampled per repeat")
    ap.add_argument("--workload", default="fp16_4096")
    ap.add_argument("--impl", choices=["ours", "reference", "vendor"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain back-to-back launches instead of a CUDA-graph replay")
    ap.add_argument("--quick", action="store_true",
                    help="profiling mode: only W warm-up and K timed launches, short JSON line")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of cpu_baseline")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="oracle time budget of the whole --impl reference run")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    elif args.impl == "vendor":
        vendor_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
