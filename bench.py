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


def ncu_traffic(kind: str, fmt: str):
    """Mean DRAM bytes (read + write) per launch of one kernel class over one
    step, from the committed ncu summary, if it was taken on the current
    sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get("kernels", {}).get(f"{kind}_{fmt}")
    if e is None or e.get("source_hash") != source_hash(kind):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------ our library
class Plan:
    """Preallocated device buffers for one step of the layer-linears workload."""

    def __init__(self, mx, wl, fmt, device):
        self.mx, self.fmt = mx, fmt
        self.gemms = []
        for i, g in enumerate(wl.gemms):
            T, Kin, Nout = g.tokens, g.k_in, g.n_out
            e = dict(g=g, T=T, Kin=Kin, Nout=Nout)
            e["xq"] = mx.MXTensor(fmt, T, Kin, device)       # X rowwise
            e["wq"] = mx.MXTensor(fmt, Nout, Kin, device)    # W rowwise
            e["dyq"] = mx.MXTensor(fmt, T, Nout, device)     # dY rowwise
            e["wtq"] = mx.MXTensor(fmt, Kin, Nout, device)   # W^T (colwise)
            e["dytq"] = mx.MXTensor(fmt, Nout, T, device)    # dY^T (colwise)
            e["xtq"] = mx.MXTensor(fmt, Kin, T, device)      # X^T (colwise)
            e["Y"] = torch.empty(T, Nout, dtype=torch.bfloat16, device=device)
            e["dX"] = torch.empty(T, Kin, dtype=torch.bfloat16, device=device)
            e["dW"] = torch.empty(Nout, Kin, dtype=torch.float32, device=device)
            self.gemms.append(e)
        self.has_ts = fmt in ("nvfp4", "moss")

    def calls(self, inputs):
        """The step as a list of (kind, fn, flops_or_bytes) in issue order.  Each of
        X, W and dY is read once by the dual-direction producer, which emits the
        rowwise operand and the transposed operand the other pass needs."""
        mx, fmt, out = self.mx, self.fmt, []
        for e in self.gemms:
            g = e["g"]
            X, W, dY = inputs[g.x.name], inputs[g.w.name], inputs[g.dy.name]
            T, Kin, Nout = e["T"], e["Kin"], e["Nout"]
            ts = self.has_ts
            out.append(("quant", lambda X=X, e=e: mx.quantize_dual(X, fmt, row_out=e["xq"], col_out=e["xtq"]),
                        dual_bytes(fmt, T * Kin, ts)))
            out.append(("quant", lambda W=W, e=e: mx.quantize_dual(W, fmt, row_out=e["wq"], col_out=e["wtq"]),
                        dual_bytes(fmt, Nout * Kin, ts)))
            out.append(("gemm", lambda e=e: mx.gemm(e["xq"], e["wq"], out=e["Y"]), 2.0 * T * Kin * Nout))
            out.append(("quant", lambda dY=dY, e=e: mx.quantize_dual(dY, fmt, row_out=e["dyq"], col_out=e["dytq"]),
                        dual_bytes(fmt, T * Nout, ts)))
            out.append(("gemm", lambda e=e: mx.gemm(e["dyq"], e["wtq"], out=e["dX"]), 2.0 * T * Kin * Nout))
            out.append(("gemm", lambda e=e: mx.gemm(e["dytq"], e["xtq"], out=e["dW"]), 2.0 * T * Kin * Nout))
        return out


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

    def step(events=None):
        for i, (fmt, kind, fn, _) in enumerate(calls):
            if events is not None:
                events[i][0].record(stream)
            fn()
            if events is not None:
                events[i][1].record(stream)

    # which GEMM kernel each scheme's launches use (named in the roofline)
    variants = {}
    for fmt, kind, fn, _ in calls:
        fn()
        if kind == "gemm":
            variants.setdefault(fmt, set()).add(mx.last_gemm_variant())
    gemm_kernels = {f: " + ".join(GEMM_KERNEL_NAME[v].format(fmt=f) for v in sorted(vs)) for f, vs in variants.items()}
    # per-call events for every timed step
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in calls]
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index) as clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        assert mx.last_device_status() == mx.MX_OK
        launches0 = mx.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        clk.start_window()
        t0.record(stream)
        for s in range(args.steps):
            step(ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
        clk.end_window()
    barrier(world)
    launches = mx.launch_count() - launches0
    status = mx.last_device_status()
    ms = t0.elapsed_time(t1) / args.steps
    ms = reduce_max(ms, world)
    # per-kernel-class durations (ms per step)
    per = {}
    for i, (fmt, kind, fn, work) in enumerate(calls):
        d = sum(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)) / args.steps
        k = (fmt, kind)
        a = per.setdefault(k, {"ms": 0.0, "work": 0.0, "calls": 0})
        a["ms"] += d
        a["work"] += work
        a["calls"] += 1
    result = dict(ms=ms, gemm_flops=gemm_flops, per=per, launches=launches, clocks=clk.summary(),
                  gemm_kernels=gemm_kernels,
                  status=status, calls_per_step=len(calls))
    if not args.no_e2e:
        result["e2e"] = run_e2e(mx, wl, inputs, device, args, world)
    result["wl"] = wl
    result["inputs"] = inputs
    return result


def run_e2e(mx, wl, dev_inputs, device, args, world):
    """The same step through the public linear-layer API with host buffers:
    pinned-host -> device copies of every input, mx.linear_fwd / linear_bwd,
    device -> pinned-host copies of every output, all inside the timed region
    (copies overlap the compute of neighbouring layers on their own streams)."""
    host_in = {k: v.cpu().pin_memory() for k, v in dev_inputs.items()}
    bufs = []
    for fmt in wl.formats:
        for g in wl.gemms:
            T, Kin, Nout = g.tokens, g.k_in, g.n_out
            b = dict(g=g, fmt=fmt)
            b["X"], b["W"], b["dY"] = (torch.empty_like(dev_inputs[g.x.name]), torch.empty_like(dev_inputs[g.w.name]),
                                       torch.empty_like(dev_inputs[g.dy.name]))
            b["Y"] = torch.empty(T, Nout, dtype=torch.bfloat16, device=device)
            b["dX"] = torch.empty(T, Kin, dtype=torch.bfloat16, device=device)
            b["dW"] = torch.empty(Nout, Kin, dtype=torch.float32, device=device)
            b["wsf"] = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "fwd"), dtype=torch.uint8, device=device)
            b["wsb"] = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "bwd"), dtype=torch.uint8, device=device)
            b["hY"] = torch.empty(b["Y"].shape, dtype=b["Y"].dtype).pin_memory()
            b["hdX"] = torch.empty(b["dX"].shape, dtype=b["dX"].dtype).pin_memory()
            b["hdW"] = torch.empty(b["dW"].shape, dtype=b["dW"].dtype).pin_memory()
            bufs.append(b)
    h2d = sum(host_in[b["g"].x.name].nbytes + host_in[b["g"].w.name].nbytes + host_in[b["g"].dy.name].nbytes
              for b in bufs)
    d2h = sum(b["Y"].nbytes + b["dX"].nbytes + b["dW"].nbytes for b in bufs)
    flops = sum(6.0 * b["g"].tokens * b["g"].k_in * b["g"].n_out for b in bufs)

    # Three streams: host->device copies, compute, device->host copies.  Unit
    # u's inputs land while unit u-1 computes and its outputs leave while unit
    # u+1 computes; events keep a buffer from being overwritten before the
    # previous step is done with it.
    compute = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    for b in bufs:
        b["in_ready"], b["computed"], b["out_done"] = ev(), ev(), ev()
        b["computed"].record(compute)
        b["out_done"].record(compute)

    def step():
        for b in bufs:
            g = b["g"]
            h2d_s.wait_event(b["computed"])  # the previous step no longer reads these inputs
            with torch.cuda.stream(h2d_s):
                b["X"].copy_(host_in[g.x.name], non_blocking=True)
                b["W"].copy_(host_in[g.w.name], non_blocking=True)
                b["dY"].copy_(host_in[g.dy.name], non_blocking=True)
            b["in_ready"].record(h2d_s)
        for b in bufs:
            compute.wait_event(b["in_ready"])
            compute.wait_event(b["out_done"])  # the previous step's outputs have left
            mx.linear_fwd(b["X"], b["W"], b["fmt"], workspace=b["wsf"], out=b["Y"])
            mx.linear_bwd(b["dY"], b["X"], b["W"], b["fmt"], workspace=b["wsb"], dX=b["dX"], dW=b["dW"])
            b["computed"].record(compute)
            d2h_s.wait_event(b["computed"])
            with torch.cuda.stream(d2h_s):
                b["hY"].copy_(b["Y"], non_blocking=True)
                b["hdX"].copy_(b["dX"], non_blocking=True)
                b["hdW"].copy_(b["dW"], non_blocking=True)
            b["out_done"].record(d2h_s)
        for b in bufs:  # the step ends when its last result is on the host
            compute.wait_event(b["out_done"])

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step()
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
    gemm:<fmt>:MxNxK, gemmq:<fmt>:<out fmt>:MxNxK (quantized epilogue) or
    quant:<fmt>:<row|col|dual>:RxC  (bf16 Student-t inputs)."""
    import fp4_precision_gemms_gb300 as mx
    mx.build()
    mx.set_gemm_variant(args.gemm_variant)
    mx.set_quant_impl(args.quant_impl)
    parts = args.case.split(":")
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if parts[0] == "gemm":
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
    else:
        fmt, direction = parts[1], parts[2]
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
            fn = lambda: mx.quantize_dual(x, fmt, row_out=q, col_out=qc, amax_in=amax_in)  # noqa: E731
            work = dual_bytes(fmt, R * Cc, False)
        else:
            fn = lambda: mx.quantize(x, fmt, direction, out=q, amax_in=amax_in)  # noqa: E731
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
    if kind == "gemm":
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e12
        peak = pk["bf16_tflops_sustained"] * NOMINAL_RATIO[fmt]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "kernel": r["gemm_kernels"][fmt],
                "peak_source": f"{src}: bf16_tflops_sustained x {NOMINAL_RATIO[fmt]:g} (nominal {fmt} / bf16 ratio)",
                "traffic": ncu_traffic("gemm", fmt)}
    else:
        achieved = d["work"] / (d["ms"] * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "kernel": f"quantize<{fmt}>", "peak_source": f"{src}: hbm_gbs",
                "traffic": ncu_traffic("quant", fmt)}
    kernels = {}
    for (f, k), a in sorted(r["per"].items()):
        if k == "gemm":
            tf = a["work"] / (a["ms"] * 1e-3) / 1e12
            pkk = pk["bf16_tflops_sustained"] * NOMINAL_RATIO[f]
            kernels[f"{f}_gemm"] = {"ms_per_step": round(a["ms"], 3), "calls": a["calls"], "TFLOP/s": round(tf, 1),
                                    "frac_of_tensor_peak": round(tf / pkk, 4)}
        else:
            gb = a["work"] / (a["ms"] * 1e-3) / 1e9
            kernels[f"{f}_quantize"] = {"ms_per_step": round(a["ms"], 3), "calls": a["calls"],
                                        "GB/s": round(gb, 1), "frac_of_hbm_peak": round(gb / pk["hbm_gbs"], 4)}
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["ms"], 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3/e2m1 block-scaled MMA, f32 accumulate", "data": "synthetic",
            "config": config_of(wl, args), "roofline": roof, "kernels": kernels,
            "gpu_launches": int(r["launches"]), "clocks": r["clocks"], "device_status": int(r["status"])}
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
