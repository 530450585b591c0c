"""The benchmark's accounting, checked on the CPU: the step's flop count against
the workload's shapes, the algorithmic bytes of a producer call, and the rule
that DRAM traffic is reported only for the sources it was measured on."""
import json

import pytest
import torch

import bench
import workloads


class _StubMX:
    """Stands in for the library: the plan only needs operand objects."""

    class MXTensor:
        def __init__(self, fmt, rows, k, device=None):
            self.fmt, self.rows, self.k = fmt, rows, k


def test_step_flops_are_three_gemms_per_linear_per_scheme():
    wl = workloads.workloads()[5]
    want = 0
    for g in wl.gemms:  # fwd, dgrad and wgrad all contract T x Kin x Nout
        want += 3 * 2 * g.tokens * g.k_in * g.n_out
    want *= len(wl.formats)
    assert want == wl.flops()
    got = 0.0
    calls = 0
    inputs = {t: None for g in wl.gemms for t in (g.x.name, g.w.name, g.dy.name)}
    for fmt in wl.formats:
        plan = bench.Plan(_StubMX, wl, fmt, torch.device("cpu"))
        for kind, _fn, units in plan.calls(inputs):
            calls += 1
            if kind == "gemm":
                got += units
    assert got == want
    # per scheme and linear: three dual-direction producer calls and three GEMMs
    assert calls == len(wl.formats) * len(wl.gemms) * 6


def test_producer_bytes_per_element():
    # one bf16 read, then codes + one scale byte per block in each direction
    assert bench.dual_bytes("mxfp8", 1, False) == pytest.approx(2 + 2 * (1 + 1 / 32))
    assert bench.dual_bytes("nvfp4", 1, True) == pytest.approx(2 + 2 + 2 * (0.5 + 1 / 16))
    assert bench.quant_bytes("mxfp4", 1, False) == pytest.approx(2 + 0.5 + 1 / 32)


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "fp4_precision_gemms_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["gemm"]:
        (csrc / f).write_text(f"// {f}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"dram_bytes_per_launch": 123456, "tensor_active_pct": 71.5, "source_hash": bench.source_hash("gemm")}
    (tmp_path / "profiles" / "counters.json").write_text(json.dumps({"kernels": {"gemm_mxfp8": entry}}))
    assert bench.ncu_traffic("gemm", "mxfp8") == 123456
    assert bench.ncu_counters("gemm", "mxfp8")["tensor_active_pct"] == 71.5
    assert bench.ncu_traffic("gemm", "nvfp4") is None  # no counters for that class
    (csrc / "gemm.cu").write_text("// gemm.cu, edited\n")
    assert bench.ncu_traffic("gemm", "mxfp8") is None  # the kernel changed since the capture


@pytest.mark.parametrize("idx,kinds", [
    (2, ["quant", "quant", "gemm", "quant", "gemm", "gemm"]),         # MOSS: X, W, dY dual; three passes
    (3, ["quant", "quant", "gemm", "quant", "quant", "gemm"]),         # NVFP4 MLP fwd: rowwise only
    (4, ["quant", "quant", "gemm"]),                                    # MXFP4 wgrad: X^T, dY^T, dW
])
def test_side_workload_plans(idx, kinds):
    """The other workloads' steps: which producer calls and GEMMs run, their
    flops and the bytes of each producer call (one direction or both)."""
    wl = workloads.workloads()[idx]
    inputs = {t.name: None for g in wl.gemms for t in (g.x, g.w, g.dy) if t is not None}
    calls = bench.Plan(_StubMX, wl, wl.formats[0], torch.device("cpu"), wgrad=bench.SIDE_WORKLOADS[idx]).calls(inputs)
    assert [c[0] for c in calls] == kinds
    assert sum(c[2] for c in calls if c[0] == "gemm") == wl.flops()
    fmt = wl.formats[0]
    ts = fmt in ("nvfp4", "moss")
    qbytes = [c[2] for c in calls if c[0] == "quant"]
    if idx == 4:  # X^T and dY^T, one direction each, no tensor scale
        assert qbytes == [bench.quant_bytes(fmt, 8192 * 4096, False), bench.quant_bytes(fmt, 8192 * 14336, False)]
    if idx == 3:
        assert qbytes[0] == bench.quant_bytes(fmt, 8192 * 4096, ts)
    if idx == 2:
        assert qbytes[0] == bench.dual_bytes(fmt, 4096 * 4096, ts)


def test_fused_fraction_adds_each_class_at_its_roof():
    pk = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    per = {("mxfp8", "gemm"): {"work": 4e12, "ms": 2.0}, ("nvfp4", "gemm"): {"work": 6e12, "ms": 1.0},
           ("mxfp8", "quant"): {"work": 8e9, "ms": 2.0}}
    f = bench.fused_fraction(per, pk, 8.0)
    # 4e12 / 4000e12 s + 6e12 / 12000e12 s + 8e9 / 8000e9 s = 1 + 0.5 + 1 ms
    assert f["ideal_ms"] == pytest.approx(2.5)
    assert f["frac"] == pytest.approx(2.5 / 8.0)
