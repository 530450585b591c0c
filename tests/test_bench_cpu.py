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
    entry = {"dram_bytes_per_launch": 123456, "source_hash": bench.source_hash("gemm")}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kernels": {"gemm_mxfp8": entry}}))
    assert bench.ncu_traffic("gemm", "mxfp8") == 123456
    assert bench.ncu_traffic("gemm", "nvfp4") is None  # no counters for that class
    (csrc / "gemm.cu").write_text("// gemm.cu, edited\n")
    assert bench.ncu_traffic("gemm", "mxfp8") is None  # the kernel changed since the capture
