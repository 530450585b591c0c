#!/usr/bin/env python
"""Throughput of the fused quantize + block-scaled GEMM linear layer on GB300.

Workload: the Llama-3-8B decoder layer's linears (QKV 4096->6144, O 4096->4096,
gate/up 4096->2x14336, down 14336->4096) at 8192 tokens, forward + data
gradient + weight gradient, run under both the MXFP8 and the NVFP4 scheme.
One step = that whole set once per scheme: every operand is quantized by the
library's producer kernels (weights too, every step) and multiplied by its
tcgen05 block-scaled GEMM, all through the C ABI.

Metric: GEMM TFLOP/s of the whole job = sum(2*M*N*K over the step's GEMMs) /
step time (quantize time included).  Inputs are larger than L2 (129 MB) and
the step streams ~10 GB, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); the step time is the max over ranks.
--impl reference times the CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused quant+block-scaled GEMM TFLOP/s (MXFP8/NVFP4), % of tensor & HBM peak"
UNIT = "TFLOP/s"
SCHEMES = ("mxfp8", "nvfp4")
BLOCK = {"mxfp8": 32, "nvfp4": 16, "mxfp4": 32, "moss": 32, "nvfp4_local": 16}
CODE_BYTES = {"mxfp8": 1.0, "moss": 1.0, "mxfp4": 0.5, "nvfp4": 0.5, "nvfp4_local": 0.5}
NOMINAL_RATIO = {"mxfp8": 2.0, "moss": 2.0, "mxfp4": 6.0, "nvfp4": 6.0, "nvfp4_local": 6.0}  # dense fp8 / fp4 vs bf16


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (the slowest rank defines the job's time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms.  Started before the warm-up
    (nvidia-smi takes a moment to start); only the samples whose timestamps fall
    inside the window marked by start_window()/end_window() are summarised."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.window = [None, None]

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def start_window(self):
        self.window[0] = datetime.datetime.now()

    def end_window(self):
        self.window[1] = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)  # let the sample that straddles the window's end land
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = self.window
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    mhz, mx_mhz = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                if lo is not None and ts < lo - datetime.timedelta(milliseconds=25):
                    continue
                if hi is not None and ts > hi + datetime.timedelta(milliseconds=25):
                    continue
                sm.append(mhz)
                smax = mx_mhz
                try:
                    power.append(float(parts[4]))
                except ValueError:
                    pass
                for n, v in zip(names, parts[6:10]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons) if sm else ["unsampled"], "samples": len(sm),
                "power_w_median": float(np.median(power)) if power else None}


GEMM_KERNEL_NAME = {"cta_n128": "bs_gemm_kernel<{fmt}, 128x128 tiles>",
                    "cta_n256": "bs_gemm_kernel<{fmt}, 128x256 tiles>",
                    "pair": "bs_gemm_pair_kernel<{fmt}, 256x256 tiles, CTA pair>",
                    "pair_ws": "bs_gemm_ws_kernel<{fmt}, 256x256 tiles, CTA pair, warp-specialised>"}


def quant_bytes(fmt: str, elems: int, amax_pass: bool) -> float:
    """Algorithmic HBM bytes of one quantize call: bf16 read (+ the amax pass's
    read) + codes + one scale byte per block."""
    return elems * (2.0 + (2.0 if amax_pass else 0.0) + CODE_BYTES[fmt] + 1.0 / BLOCK[fmt])


def dual_bytes(fmt: str, elems: int, amax_pass: bool) -> float:
    """Algorithmic HBM bytes of one dual-direction producer call: one bf16 read
    (+ the amax pass's read) and two sets of codes and scale bytes."""
    return elems * (2.0 + (2.0 if amax_pass else 0.0) + 2.0 * (CODE_BYTES[fmt] + 1.0 / BLOCK[fmt]))


KERNEL_SOURCES = {"gemm": ("gemm.cu", "mx_ptx.cuh", "mx_codec.cuh"), "quant": ("quantize.cu", "mx_ptx.cuh", "mx_codec.cuh")}


def source_hash(kind: str) -> str:
    """Hash of the sources one kernel class is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_precision_gemms_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


COUNTERS = os.path.join("profiles", "counters.json")


def ncu_counters(kind: str, fmt: str, workload: int = 5):
    """The committed ncu counters of one kernel class (per launch: DRAM bytes;
    tensor-pipe, ALU/FMA-pipe and issue activity in percent), if they were taken
    on the current sources of that kernel; else None.  Classes of the headline
    workload are keyed '<kind>_<fmt>', those of another workload
    '<kind>_<fmt>@<workload>'."""
    try:
        with open(os.path.join(ROOT, COUNTERS)) as f:
            t = json.load(f)
    except Exception:
        return None
    key = f"{kind}_{fmt}" if workload == 5 else f"{kind}_{fmt}@{workload}"
    e = t.get("kernels", {}).get(key)
    if e is None or e.get("source_hash") != source_hash(kind):
        return None
    return e


def ncu_traffic(kind: str, fmt: str, workload: int = 5):
    """DRAM bytes (read + write) per launch of one kernel class, or None."""
    e = ncu_counters(kind, fmt, workload)
    return None if e is None else e.get("dram_bytes_per_launch")


def tensor_peak(pk: dict, fmt: str) -> float:
    """Dense tensor peak of a format (TFLOP/s): the measured bf16 burst figure
    (cuBLAS) times the nominal FP8 / FP4 to bf16 ratio.  The timed region is
    well under a second, so the burst (not the sustained) bf16 figure applies."""
    return pk["bf16_tflops"] * NOMINAL_RATIO[fmt]


def class_rates(per: dict, pk: dict, workload: int = 5) -> dict:
    """Per (format, kind) class: ms per step, calls, rate, fraction of its roof,
    and the committed ncu counters of the class when they match the sources."""
    kernels = {}
    for (f, k), a in sorted(per.items()):
        ctr = ncu_counters(k, f, workload)
        if k == "gemm":
            tf = a["work"] / (a["ms"] * 1e-3) / 1e12
            e = {"ms_per_step": round(a["ms"], 3), "calls": a["calls"], "TFLOP/s": round(tf, 1),
                 "frac_of_tensor_peak": round(tf / tensor_peak(pk, f), 4)}
            if ctr and "tensor_active_pct" in ctr:
                e["tensor_active_pct"] = ctr["tensor_active_pct"]
            kernels[f"{f}_gemm"] = e
        else:
            gb = a["work"] / (a["ms"] * 1e-3) / 1e9
            e = {"ms_per_step": round(a["ms"], 3), "calls": a["calls"], "GB/s": round(gb, 1),
                 "frac_of_hbm_peak": round(gb / pk["hbm_gbs"], 4)}
            if ctr:
                for n in ("alu_pipe_pct", "fma_pipe_pct", "issue_active_pct", "dram_throughput_pct"):
                    if n in ctr:
                        e[n] = ctr[n]
            kernels[f"{f}_quantize"] = e
    return kernels


def fused_fraction(per: dict, pk: dict, ms: float) -> dict:
    """The step's roofline fraction: the time every class would take at its own
    roof (quantize bytes at the HBM peak, GEMM flops at the format's tensor
    peak), summed since the kernels run one after another, over the measured
    step time."""
    ideal = 0.0
    for (f, k), a in per.items():
        ideal += a["work"] / (tensor_peak(pk, f) * 1e12) if k == "gemm" else a["work"] / (pk["hbm_gbs"] * 1e9)
    ideal_ms = ideal * 1e3
    return {"ideal_ms": round(ideal_ms, 3), "measured_ms": round(ms, 3), "frac": round(ideal_ms / ms, 4)}


# ------------------------------------------------------------ our library
class Plan:
    """Preallocated device buffers for one step of a workload under one format.

    Each GEMM of the workload runs its passes: fwd Y = X W^T, dgrad dX = dY W,
    wgrad dW = dY^T X.  fwd reads X and W rowwise; dgrad reads dY rowwise and
    W colwise; wgrad reads dY and X colwise.  A tensor needed in both
    directions is read once by the dual-direction producer.  `wgrad` holds the
    weight-gradient options: Hadamard on both operands, rounding and seed of
    dY^T."""

    def __init__(self, mx, wl, fmt, device, wgrad=None):
        self.mx, self.fmt = mx, fmt
        self.wgrad = dict(hadamard=False, rounding="rne", seed=0)
        self.wgrad.update(wgrad or {})
        self.gemms = []
        for g in wl.gemms:
            T, Kin, Nout = g.tokens, g.k_in, g.n_out
            e = dict(g=g, T=T, Kin=Kin, Nout=Nout)
            p = g.passes
            if "fwd" in p:
                e["xq"] = mx.MXTensor(fmt, T, Kin, device)       # X rowwise
                e["wq"] = mx.MXTensor(fmt, Nout, Kin, device)    # W rowwise
                e["Y"] = torch.empty(T, Nout, dtype=torch.bfloat16, device=device)
            if "dgrad" in p:
                e["dyq"] = mx.MXTensor(fmt, T, Nout, device)     # dY rowwise
                e["wtq"] = mx.MXTensor(fmt, Kin, Nout, device)   # W^T (colwise)
                e["dX"] = torch.empty(T, Kin, dtype=torch.bfloat16, device=device)
            if "wgrad" in p:
                e["dytq"] = mx.MXTensor(fmt, Nout, T, device)    # dY^T (colwise)
                e["xtq"] = mx.MXTensor(fmt, Kin, T, device)      # X^T (colwise)
                e["dW"] = torch.empty(Nout, Kin, dtype=torch.float32, device=device)
            self.gemms.append(e)
        self.has_ts = fmt in ("nvfp4", "moss")

    def _quant(self, x, row_key, col_key, e, col_opts):
        """(fn, algorithmic bytes) of the producer call(s) for one input tensor."""
        mx, fmt, ts = self.mx, self.fmt, self.has_ts
        if row_key in e and col_key in e:
            fn = lambda: mx.quantize_dual(x, fmt, row_out=e[row_key], col_out=e[col_key], **col_opts)  # noqa: E731
            return fn, dual_bytes(fmt, e[row_key].rows * e[row_key].k, ts)
        if row_key in e:
            return (lambda: mx.quantize(x, fmt, "row", out=e[row_key]),
                    quant_bytes(fmt, e[row_key].rows * e[row_key].k, ts))
        opts = {{"col_hadamard": "hadamard", "col_rounding": "rounding"}.get(k, k): v for k, v in col_opts.items()}
        return (lambda: mx.quantize(x, fmt, "col", out=e[col_key], **opts),
                quant_bytes(fmt, e[col_key].rows * e[col_key].k, ts))

    def calls(self, inputs):
        """The step as a list of (kind, fn, flops_or_bytes) in issue order."""
        return [c[:3] for c in self.roles(inputs)]

    def roles(self, inputs):
        """The step's calls with their place in the layer: (kind, fn, work,
        layer index, role), role one of qx, qw, fwd, qdy, dgrad, wgrad."""
        mx, out = self.mx, []
        wg = self.wgrad
        had = dict(col_hadamard=True) if wg["hadamard"] else {}
        dy_col = dict(col_rounding=wg["rounding"], seed=wg["seed"], **had) if (wg["rounding"] != "rne" or had) else {}
        for li, e in enumerate(self.gemms):
            g = e["g"]
            T, Kin, Nout = e["T"], e["Kin"], e["Nout"]
            flops = 2.0 * T * Kin * Nout
            if g.x is not None and ("xq" in e or "xtq" in e):
                fn, b = self._quant(inputs[g.x.name], "xq", "xtq", e, had)
                out.append(("quant", fn, b, li, "qx"))
            if g.w is not None and ("wq" in e or "wtq" in e):
                fn, b = self._quant(inputs[g.w.name], "wq", "wtq", e, {})
                out.append(("quant", fn, b, li, "qw"))
            if "Y" in e:
                out.append(("gemm", lambda e=e: mx.gemm(e["xq"], e["wq"], out=e["Y"]), flops, li, "fwd"))
            if g.dy is not None and ("dyq" in e or "dytq" in e):
                fn, b = self._quant(inputs[g.dy.name], "dyq", "dytq", e, dy_col)
                out.append(("quant", fn, b, li, "qdy"))
            if "dX" in e:
                out.append(("gemm", lambda e=e: mx.gemm(e["dyq"], e["wtq"], out=e["dX"]), flops, li, "dgrad"))
            if "dW" in e:
                out.append(("gemm", lambda e=e: mx.gemm(e["dytq"], e["xtq"], out=e["dW"]), flops, li, "wgrad"))
        return out


# The workloads timed next to the headline one, with their weight-gradient
# options (workload 4: Hadamard-32 on both wgrad operands, stochastic rounding
# of dY^T with Philox seed 42).
SIDE_WORKLOADS = {2: {}, 3: {}, 4: dict(hadamard=True, rounding="sr", seed=42)}


def time_calls(calls, steps, warmup, stream, clk=None, count=None):
    """Runs warm-up steps, then `steps` timed steps of `calls` with CUDA events on
    `stream` (one pair per call).  Returns (ms per step, per-class dict, the
    increase of count() over the timed steps, or None)."""
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in calls]
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step(events=None):
        for i, c in enumerate(calls):
            if events is not None:
                events[i][0].record(stream)
            c[2]()
            if events is not None:
                events[i][1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    c0 = count() if count else None
    if clk is not None:
        clk.start_window()
    t0.record(stream)
    for s in range(steps):
        step(ev[s])
    t1.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.end_window()
    counted = count() - c0 if count else None
    per = {}
    for i, (fmt, kind, fn, work) in enumerate(calls):
        d = sum(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)) / steps
        a = per.setdefault((fmt, kind), {"ms": 0.0, "work": 0.0, "calls": 0})
        a["ms"] += d
        a["work"] += work
        a["calls"] += 1
    return t0.elapsed_time(t1) / steps, per, counted


def issue_three_streams(role_calls, s1, s2):
    """Issues one step on three streams, for capture: the current stream runs
    each layer's X and W producers and its fwd GEMM, `s1` its dY producer and
    dgrad GEMM (after W's producer), `s2` its wgrad GEMM (after X's and dY's
    producers)."""
    main = torch.cuda.current_stream()
    s1.wait_stream(main)
    s2.wait_stream(main)
    place = {"qx": main, "qw": main, "fwd": main, "qdy": s1, "dgrad": s1, "wgrad": s2}
    needs = {"dgrad": ("qw",), "wgrad": ("qx", "qdy")}
    ev = {}
    for fmt, kind, fn, work, li, role in role_calls:
        unit = (fmt, li)
        st = place[role]
        for dep in needs.get(role, ()):
            if (unit, dep) in ev:
                st.wait_event(ev[(unit, dep)])
        with torch.cuda.stream(st):
            fn()
        if role in ("qx", "qw", "qdy"):
            e = torch.cuda.Event()
            e.record(st)
            ev[(unit, role)] = e
    main.wait_stream(s1)
    main.wait_stream(s2)


def issue_two_streams(role_calls, side):
    """Issues one step on two streams, for capture: the current stream runs each
    layer's X and W producers and its fwd and dgrad GEMMs, `side` runs its dY
    producer and wgrad GEMM; events carry the two cross-stream dependencies
    (dgrad reads dY's rowwise operand, wgrad reads X's colwise one).  Layers are
    independent of one another, so the graph may run either stream's kernels
    in the other's idle SMs (the tail of a GEMM's last wave)."""
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    ev = {}
    for fmt, kind, fn, work, li, role in role_calls:
        unit = (fmt, li)
        on_side = role in ("qdy", "wgrad")
        st = side if on_side else main
        if role == "dgrad" and (unit, "qdy") in ev:
            main.wait_event(ev[(unit, "qdy")])
        if role == "wgrad" and (unit, "qx") in ev:
            side.wait_event(ev[(unit, "qx")])
        with torch.cuda.stream(st):
            fn()
        if role in ("qx", "qdy"):
            e = torch.cuda.Event()
            e.record(st)
            ev[(unit, role)] = e
    main.wait_stream(side)


def graph_time(calls, steps, warmup, stream, clk=None, count=None, issue=None):
    """One step captured as a CUDA graph (every call launches on the capture
    stream, or as `issue` places it; operands and outputs are preallocated, so
    the graph replays the same work), then `warmup` untimed and `steps` timed
    replays with CUDA events on `stream`.  Returns (ms per step, library
    launches per step)."""
    g = torch.cuda.CUDAGraph()
    c0 = count() if count else None
    with torch.cuda.graph(g):
        if issue is not None:
            issue()
        else:
            for c in calls:
                c[2]()
    per_step = count() - c0 if count else None
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start_window()
    t0.record(stream)
    for _ in range(steps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.end_window()
    del g
    return t0.elapsed_time(t1) / steps, per_step


def run_ours(args, world, rank, local):
    import fp4_precision_gemms_gb300 as mx
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    mx.build()
    wl = workloads.workloads()[args.workload]
    inputs = workloads.materialize(wl, device=device)
    plans = [Plan(mx, wl, fmt, device) for fmt in wl.formats]
    calls = []
    for p in plans:
        calls += [(p.fmt,) + c for c in p.calls(inputs)]
    gemm_flops = sum(c[3] for c in calls if c[1] == "gemm")
    stream = torch.cuda.current_stream()

    # which GEMM kernel each scheme's launches use (named in the roofline)
    variants = {}
    for fmt, kind, fn, _ in calls:
        fn()
        if kind == "gemm":
            variants.setdefault(fmt, set()).add(mx.last_gemm_variant())
    gemm_kernels = {f: " + ".join(GEMM_KERNEL_NAME[v].format(fmt=f) for v in sorted(vs)) for f, vs in variants.items()}
    with ClockSampler(device.index) as clk:
        torch.cuda.synchronize()
        assert mx.last_device_status() == mx.MX_OK
        barrier(world)
        # per-class CUDA-event times of the step launched call by call (the roofline
        # and the class fractions), then the step itself as one CUDA graph
        ms_eager, per, launches = time_calls(calls, args.steps, args.warmup, stream,
                                             None if args.graph else clk, count=mx.launch_count)
        ms = ms_eager
        if args.graph:
            torch.cuda.synchronize()
            barrier(world)
            issue = None
            role_calls = [(p.fmt,) + c for p in plans for c in p.roles(inputs)]
            if args.streams == 2:
                side = torch.cuda.Stream(device=device)
                issue = lambda: issue_two_streams(role_calls, side)  # noqa: E731
            elif args.streams == 3:
                s1, s2 = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
                issue = lambda: issue_three_streams(role_calls, s1, s2)  # noqa: E731
            ms, per_step = graph_time(calls, args.steps, args.warmup, stream, clk, count=mx.launch_count, issue=issue)
            launches = per_step * args.steps
    barrier(world)
    status = mx.last_device_status()
    ms = reduce_max(ms, world)
    ms_eager = reduce_max(ms_eager, world)
    result = dict(ms=ms, ms_eager=ms_eager, gemm_flops=gemm_flops, per=per, launches=launches, clocks=clk.summary(),
                  gemm_kernels=gemm_kernels, status=status, calls_per_step=len(calls))
    if not args.no_side:
        result["side"] = run_side_workloads(mx, device, stream, args)
    if not args.no_e2e:
        result["e2e"] = run_e2e(mx, wl, inputs, device, args, world)
    result["wl"] = wl
    result["inputs"] = inputs
    return result


def run_side_workloads(mx, device, stream, args):
    """The other single-GPU workloads (MOSS linear, NVFP4 MLP forward, MXFP4
    wgrad with Hadamard-32 and SR), each timed on its own: ms per step and the
    per-class (format, kind) durations."""
    out = {}
    for idx, wg in SIDE_WORKLOADS.items():
        wl = workloads.workloads()[idx]
        inputs = workloads.materialize(wl, device=device)
        plans = [Plan(mx, wl, fmt, device, wgrad=wg) for fmt in wl.formats]
        calls = [(p.fmt,) + c for p in plans for c in p.calls(inputs)]
        flops = sum(c[3] for c in calls if c[1] == "gemm")
        ms, per, _ = time_calls(calls, args.side_steps, args.warmup, stream)
        ms_eager = ms
        if args.graph:
            issue = None
            role_calls = [(p.fmt,) + c for p in plans for c in p.roles(inputs)]
            if args.streams == 2:
                side = torch.cuda.Stream(device=device)
                issue = lambda: issue_two_streams(role_calls, side)  # noqa: E731
            elif args.streams == 3:
                s1, s2 = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
                issue = lambda: issue_three_streams(role_calls, s1, s2)  # noqa: E731
            ms, _ = graph_time(calls, args.side_steps, args.warmup, stream, issue=issue)
        out[wl.name] = dict(ms=ms, ms_eager=ms_eager, gemm_flops=flops, per=per, wgrad=wg, index=idx)
        del inputs
    torch.cuda.synchronize()
    return out


def run_e2e(mx, wl, dev_inputs, device, args, world):
    """The same step through the public linear-layer API with host buffers:
    pinned-host -> device copies of every input, mx.linear_fwd_save (which keeps
    X^T and W^T for the backward) and mx.linear_bwd_saved, so X, W and dY are
    each read once on the device, as in the kernel-level step; device ->
    pinned-host copies of every output; all inside the timed region.  Copies
    run on their own streams and overlap the compute of neighbouring layers;
    the device buffers alternate between two sets by step parity, so a step's
    copies overlap the previous step's as well."""
    host_in = {k: v.cpu().pin_memory() for k, v in dev_inputs.items()}
    units = [(fmt, g) for fmt in wl.formats for g in wl.gemms]
    host_out = []
    for fmt, g in units:  # one pinned host copy of each result (each step overwrites it)
        T, Kin, Nout = g.tokens, g.k_in, g.n_out
        host_out.append(dict(hY=torch.empty(T, Nout, dtype=torch.bfloat16).pin_memory(),
                             hdX=torch.empty(T, Kin, dtype=torch.bfloat16).pin_memory(),
                             hdW=torch.empty(Nout, Kin, dtype=torch.float32).pin_memory()))
    compute = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    sets = []
    for _ in range(2):
        bufs = []
        for u, (fmt, g) in enumerate(units):
            T, Kin, Nout = g.tokens, g.k_in, g.n_out
            b = dict(g=g, fmt=fmt, host=host_out[u])
            b["X"], b["W"], b["dY"] = (torch.empty_like(dev_inputs[g.x.name]), torch.empty_like(dev_inputs[g.w.name]),
                                       torch.empty_like(dev_inputs[g.dy.name]))
            b["Y"] = torch.empty(T, Nout, dtype=torch.bfloat16, device=device)
            b["dX"] = torch.empty(T, Kin, dtype=torch.bfloat16, device=device)
            b["dW"] = torch.empty(Nout, Kin, dtype=torch.float32, device=device)
            b["wsf"] = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "fwd"), dtype=torch.uint8, device=device)
            b["wsb"] = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "bwd_saved"), dtype=torch.uint8,
                                   device=device)
            b["saved"] = torch.empty(mx.saved_bytes(T, Kin, Nout, fmt), dtype=torch.uint8, device=device)
            b["in_ready"], b["computed"], b["out_done"] = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            b["computed"].record(compute)
            b["out_done"].record(compute)
            bufs.append(b)
        sets.append(bufs)
    h2d = sum(host_in[g.x.name].nbytes + host_in[g.w.name].nbytes + host_in[g.dy.name].nbytes for _, g in units)
    d2h = sum(b["Y"].nbytes + b["dX"].nbytes + b["dW"].nbytes for b in sets[0])
    flops = sum(6.0 * g.tokens * g.k_in * g.n_out for _, g in units)

    def step(k):
        bufs = sets[k % 2]
        for b in bufs:
            g = b["g"]
            h2d_s.wait_event(b["computed"])  # this set's previous step no longer reads these inputs
            with torch.cuda.stream(h2d_s):
                b["X"].copy_(host_in[g.x.name], non_blocking=True)
                b["W"].copy_(host_in[g.w.name], non_blocking=True)
                b["dY"].copy_(host_in[g.dy.name], non_blocking=True)
            b["in_ready"].record(h2d_s)
        for b in bufs:
            compute.wait_event(b["in_ready"])
            compute.wait_event(b["out_done"])  # this set's previous outputs have left
            mx.linear_fwd_save(b["X"], b["W"], b["fmt"], workspace=b["wsf"], saved=b["saved"], out=b["Y"])
            mx.linear_bwd_saved(b["dY"], b["saved"], b["g"].k_in, b["fmt"], workspace=b["wsb"], dX=b["dX"],
                                dW=b["dW"])
            b["computed"].record(compute)
            d2h_s.wait_event(b["computed"])
            h = b["host"]
            with torch.cuda.stream(d2h_s):
                h["hY"].copy_(b["Y"], non_blocking=True)
                h["hdX"].copy_(b["dX"], non_blocking=True)
                h["hdW"].copy_(b["dW"], non_blocking=True)
            b["out_done"].record(d2h_s)

    def drain():  # every result of every step issued so far is on the host
        for bufs in sets:
            for b in bufs:
                compute.wait_event(b["out_done"])

    for k in range(max(2, min(args.warmup, 4))):
        step(k)
    drain()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(args.steps):
        step(k)
    drain()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(t0.elapsed_time(t1) / args.steps, world)
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3)}


# ------------------------------------------------------------ CPU oracle
def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_sample(wl, host_inputs, S: int):
    """One bounded sample of the workload on the CPU oracle: for every scheme,
    GEMM and pass, an S x S block of the output with the full reduction depth,
    including the oracle's quantization of the S operand rows it needs.
    Returns (gemm flops, seconds)."""
    import oracle as orc
    flops = 0.0
    t = time.perf_counter()
    for fmt in wl.formats:
        for g in wl.gemms:
            X, W, dY = host_inputs[g.x.name], host_inputs[g.w.name], host_inputs[g.dy.name]
            s_t, s_k, s_n = min(S, g.tokens), min(S, g.k_in), min(S, g.n_out)
            # fwd: Y[:s_t, :s_n] over K = k_in
            a = orc.quantize(bits_of(X[:s_t]), fmt)
            b = orc.quantize(bits_of(W[:s_n]), fmt)
            orc.gemm(a, b)
            flops += 2.0 * s_t * s_n * g.k_in
            # dgrad: dX[:s_t, :s_k] over K = n_out
            a = orc.quantize(bits_of(dY[:s_t]), fmt)
            b = orc.quantize(bits_of(W[:, :s_k]), fmt, "col")
            orc.gemm(a, b)
            flops += 2.0 * s_t * s_k * g.n_out
            # wgrad: dW[:s_n, :s_k] over K = tokens
            a = orc.quantize(bits_of(dY[:, :s_n]), fmt, "col")
            b = orc.quantize(bits_of(X[:, :s_k]), fmt, "col")
            orc.gemm(a, b)
            flops += 2.0 * s_n * s_k * g.tokens
    return flops, time.perf_counter() - t


def host_inputs_for(wl, dev_inputs=None):
    if dev_inputs is not None:
        return {k: v.cpu() for k, v in dev_inputs.items()}
    return workloads.materialize(wl)


def cpu_baseline(wl, host_inputs, S: int):
    import oracle as orc
    flops, sec = oracle_sample(wl, host_inputs, S)
    return {"value": round(flops / sec / 1e12, 6), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": (f"{S}x{S} output block of every GEMM (fwd, dgrad, wgrad; full reduction depth) of both "
                       f"schemes, with the oracle quantizing the operand rows it needs; {flops / 1e9:.1f} GFLOP "
                       f"in {sec:.1f} s")}


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    wl = workloads.workloads()[args.workload]
    host = host_inputs_for(wl)
    S = args.ref_sample
    for _ in range(args.warmup):
        oracle_sample(wl, host, S)
    flops, sec = 0.0, 0.0
    for _ in range(args.steps):
        f, s = oracle_sample(wl, host, S)
        flops += f
        sec += s
    value = flops / sec / 1e12
    ms = sec / args.steps * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": config_of(wl, args),
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": f"per step: {S}x{S} output block of every GEMM pass of both schemes "
                                       f"({flops / args.steps / 1e9:.1f} GFLOP), oracle quantize included"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_case(args):
    """One kernel on its own, for tuning and small ncu captures:
    step:<fmt>:<gemm|quant>[:<workload>] (that class's calls of one step of a
    workload, default the headline one, after one untimed pass of the whole
    step), gemm:<fmt>:MxNxK, gemmq:<fmt>:<out fmt>:MxNxK (quantized epilogue) or
    quant:<fmt>:<row|col|dual>[+had][+sr]:RxC (bf16 Student-t inputs; +had
    applies Hadamard-32, +sr stochastic rounding with seed 42, to the colwise
    operand of a dual call) or amax:RxC (the tensor-amax pass)."""
    import fp4_precision_gemms_gb300 as mx
    mx.build()
    mx.set_gemm_variant(args.gemm_variant)
    mx.set_quant_impl(args.quant_impl)
    parts = args.case.split(":")
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if parts[0] == "step":  # one kernel class of a workload's step: step:<fmt>:<gemm|quant>[:<workload>]
        fmt, kind = parts[1], parts[2]
        idx = int(parts[3]) if len(parts) > 3 else 5
        wl = workloads.workloads()[idx]
        inputs = workloads.materialize(wl, device=dev)
        calls = Plan(mx, wl, fmt, dev, wgrad=SIDE_WORKLOADS.get(idx)).calls(inputs)
        for c in calls:  # every operand the class reads exists before the timed calls
            c[1]()
        sel = [c for c in calls if c[0] == kind]
        fn = lambda: [c[1]() for c in sel]  # noqa: E731
        work = sum(c[2] for c in sel)
        unit = "TFLOP/s" if kind == "gemm" else "GB/s"
    elif parts[0] == "gemm":
        fmt = parts[1]
        M, N, K = (int(v) for v in parts[2].split("x"))
        a = mx.quantize(workloads.draw("student_t3", (M, K), 1, device=dev), fmt)
        b = mx.quantize(workloads.draw("normal", (N, K), 2, 0.02, device=dev), fmt)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        fn = lambda: mx.gemm(a, b, out=out)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif parts[0] == "gemmq":  # GEMM whose epilogue writes the next layer's MX operand
        fmt, ofmt = parts[1], parts[2]
        M, N, K = (int(v) for v in parts[3].split("x"))
        a = mx.quantize(workloads.draw("student_t3", (M, K), 1, device=dev), fmt)
        b = mx.quantize(workloads.draw("normal", (N, K), 2, 0.02, device=dev), fmt)
        q = mx.MXTensor(ofmt, M, N, dev)
        fn = lambda: mx.gemm_quantized(a, b, ofmt, out=q)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif parts[0] == "amax":  # the tensor-amax pass alone: amax:RxC
        R, Cc = (int(v) for v in parts[1].split("x"))
        x = workloads.draw("student_t3", (R, Cc), 1, device=dev)
        am = torch.empty(1, dtype=torch.float32, device=dev)
        fn = lambda: mx.amax(x, out=am)  # noqa: E731
        work, unit = 2.0 * R * Cc, "GB/s"
    else:  # direction row, col or dual, optionally +had (Hadamard-32) and +sr (stochastic rounding)
        fmt, dopts = parts[1], parts[2].split("+")
        direction = dopts[0]
        qo = {}
        if "had" in dopts:
            qo["hadamard"] = True
        if "sr" in dopts:
            qo.update(rounding="sr", seed=42)
        R, Cc = (int(v) for v in parts[3].split("x"))
        x = workloads.draw("student_t3", (R, Cc), 1, device=dev)
        rows, k = (R, Cc) if direction == "row" else (Cc, R)
        q = mx.MXTensor(fmt, rows, k, dev)
        # global formats: time the producer pass alone (amax precomputed); nvfp4_local
        # computes its region maxima inside the timed call (a second read of x)
        amax_in = mx.amax(x) if fmt in ("nvfp4", "moss") else None
        if direction == "dual":
            qc = mx.MXTensor(fmt, Cc, R, dev)
            q = mx.MXTensor(fmt, R, Cc, dev)
            do = {("col_" + k if k in ("hadamard", "rounding") else k): v for k, v in qo.items()}
            fn = lambda: mx.quantize_dual(x, fmt, row_out=q, col_out=qc, amax_in=amax_in, **do)  # noqa: E731
            work = dual_bytes(fmt, R * Cc, False)
        else:
            fn = lambda: mx.quantize(x, fmt, direction, out=q, amax_in=amax_in, **qo)  # noqa: E731
            work = quant_bytes(fmt, R * Cc, False)
        unit = "GB/s"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"case": args.case, "ms": round(ms, 4), unit: round(rate, 2),
                      "status": mx.last_device_status()}), flush=True)


def config_of(wl, args):
    return {"workload": wl.name, "tokens": wl.gemms[0].tokens, "schemes": list(wl.formats),
            "gemms": {g.name: [g.k_in, g.n_out] for g in wl.gemms},
            "passes": ["fwd", "dgrad", "wgrad"], "outputs": "Y bf16, dX bf16, dW fp32",
            "weights_requantized_every_step": True,
            "l2": "no flush: inputs larger than L2 (step streams ~10 GB)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the step launched call by call instead of as one CUDA graph")
    ap.add_argument("--streams", type=int, default=3, choices=[1, 2, 3],
                    help="streams the step's graph is captured on (2: each layer's dY producer and wgrad "
                         "GEMM on a second stream; 3: dY producer and dgrad on the second, wgrad on a third)")
    ap.add_argument("--no-side", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--side-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=1024)
    ap.add_argument("--ref-sample", type=int, default=256)
    ap.add_argument("--case", default=None, help="time one kernel: gemm:fmt:MxNxK or quant:fmt:dir:RxC")
    ap.add_argument("--gemm-variant", default="auto", help="force a GEMM kernel variant (tuning aid)")
    ap.add_argument("--quant-impl", default="auto", help="force a producer implementation (tuning aid)")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    r = run_ours(args, world, rank, local)
    wl = r["wl"]
    pk, src = peaks()
    value = world * r["gemm_flops"] / (r["ms"] * 1e-3) / 1e12
    # dominant kernel = the (scheme, kind) class with the most time
    dom_key = max(r["per"], key=lambda k: r["per"][k]["ms"])
    d = r["per"][dom_key]
    fmt, kind = dom_key
    ctr = ncu_counters(kind, fmt) or {}
    if kind == "gemm":
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e12
        peak = tensor_peak(pk, fmt)
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "kernel": r["gemm_kernels"][fmt],
                "peak_source": (f"derived from {src}: bf16_tflops (cuBLAS bf16 burst) x {NOMINAL_RATIO[fmt]:g}, "
                                f"the nominal dense {fmt} / bf16 ratio"),
                "traffic": ctr.get("dram_bytes_per_launch"),
                "tensor_active_pct": ctr.get("tensor_active_pct")}
    else:
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "kernel": f"quantize<{fmt}>", "peak_source": f"{src}: hbm_gbs",
                "traffic": ctr.get("dram_bytes_per_launch")}
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["ms"], 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3/e2m1 block-scaled MMA, f32 accumulate", "data": "synthetic",
            "config": config_of(wl, args), "roofline": roof,
            "fused_roofline": dict(fused_fraction(r["per"], pk, r["ms"]),
                                   definition="(sum of quantize bytes / HBM peak + sum of GEMM flops / tensor peak) "
                                              "/ measured step time"),
            "kernels": class_rates(r["per"], pk),
            "gpu_launches": int(r["launches"]), "clocks": r["clocks"], "device_status": int(r["status"]),
            "launch": {"mode": "cuda_graph" if args.graph else "eager", "streams": args.streams if args.graph else 1,
                       "eager_ms_per_step": round(r["ms_eager"], 3),
                       "note": ("the step replayed as one CUDA graph (three streams: each layer's X and W producers "
                                "and fwd GEMM on the first, its dY producer and dgrad GEMM on the second, its wgrad "
                                "GEMM on the third, events for the cross-stream reads); "
                                "per-class times (kernels, roofline) come from the same step launched call by call "
                                "on one stream with CUDA events around each call")}}
    if "side" in r:
        side = {}
        for name, w in r["side"].items():
            side[name] = {"TFLOP/s": round(w["gemm_flops"] / (w["ms"] * 1e-3) / 1e12, 1),
                          "ms_per_step": round(w["ms"], 3), "eager_ms_per_step": round(w["ms_eager"], 3),
                          "gemm_tflop_per_step": round(w["gemm_flops"] / 1e12, 4),
                          "wgrad_options": w["wgrad"],
                          "fused_roofline": fused_fraction(w["per"], pk, w["ms"]),
                          "kernels": class_rates(w["per"], pk, w["index"])}
        line["workloads"] = side
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, host_inputs_for(wl, r["inputs"]), args.cpu_sample)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
