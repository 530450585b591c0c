"""Seeded synthetic inputs and workload shapes for the block-scaled linear layer.

Shared by the tests, the smoke check and the benchmark.  This module holds no
arithmetic of the method (no scaling, rounding or encoding): it only draws
seeded random bf16 tensors with the distributions of the workloads below and
names their shapes.

Distributions (drawn in fp32, rounded to bf16 by torch's round-to-nearest-even
cast):
  normal(s)        : s * N(0, 1)
  student_t3(s)    : s * Z / sqrt(chi2_3 / 3), chi2_3 = sum of three squared N(0,1)
  lognormal_cols   : N(0, 1) * exp(N(0, 1)) per column (a per-channel scale)
  outliers(p, f)   : N(0, 1), with each entry multiplied by f with probability p

Seeds: tensor t of workload w uses seed 1000 * w + t.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def draw(kind: str, shape, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """One seeded bf16 tensor of the given distribution kind."""
    g = _gen(seed, device)
    if kind == "normal":
        x = _normal(shape, g, device)
    elif kind == "student_t3":
        z = _normal(shape, g, device)
        chi2 = sum(_normal(shape, g, device) ** 2 for _ in range(3))
        x = z / torch.sqrt(chi2 / 3.0)
    elif kind == "lognormal_cols":
        z = _normal(shape, g, device)
        col = torch.exp(_normal((1, shape[1]), g, device))
        x = z * col
    elif kind == "outliers":
        z = _normal(shape, g, device)
        mask = torch.rand(*shape, generator=g, device=device) < 0.01
        x = torch.where(mask, z * 50.0, z)
    else:
        raise ValueError(kind)
    return (x * scale).to(torch.bfloat16)


def all_bf16_patterns() -> torch.Tensor:
    """Every finite bf16 bit pattern (65536 minus the Inf/NaN ones), as bf16."""
    bits = torch.arange(0, 65536, dtype=torch.int32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    return bits[finite].to(torch.int16).view(torch.bfloat16)


@dataclass
class Tensor:
    name: str
    shape: tuple
    kind: str
    scale: float = 1.0


@dataclass
class Gemm:
    """One linear layer Y = X W^T with X [tokens, k_in], W [n_out, k_in]."""
    name: str
    tokens: int
    k_in: int
    n_out: int
    x: Tensor = None
    w: Tensor = None
    dy: Tensor = None
    passes: tuple = ("fwd",)  # subset of fwd, dgrad, wgrad

    def flops(self) -> int:
        return 2 * self.tokens * self.k_in * self.n_out * len(self.passes)


@dataclass
class Workload:
    index: int
    name: str
    formats: tuple
    gemms: list = field(default_factory=list)
    note: str = ""

    def flops(self) -> int:
        return sum(g.flops() for g in self.gemms) * len(self.formats)


def _t(name, shape, kind, scale=1.0):
    return Tensor(name, tuple(shape), kind, scale)


def workloads() -> dict:
    """The five workloads of the block-scaled linear layer (index 1..5)."""
    w = {}
    w[1] = Workload(1, "mxfp8_tiny_256", ("mxfp8",), [
        Gemm("tiny", 256, 256, 256, x=_t("A", (256, 256), "outliers"),
             w=_t("B", (256, 256), "outliers"))],
        note="A,B bf16 256x256, N(0,1) with 1% of entries x50; C = A B^T fp32")
    w[2] = Workload(2, "moss_fp8_linear_4096x11008", ("moss",), [
        Gemm("linear", 4096, 4096, 11008, x=_t("X", (4096, 4096), "lognormal_cols"),
             w=_t("W", (11008, 4096), "normal", 0.02),
             dy=_t("dY", (4096, 11008), "student_t3", 1e-3),
             passes=("fwd", "dgrad", "wgrad"))],
        note="MOSS two-level FP8 linear fwd + dgrad + wgrad")
    w[3] = Workload(3, "nvfp4_llama3_8b_mlp_fwd_8192tok", ("nvfp4",), [
        Gemm("gate_up", 8192, 4096, 28672, x=_t("X", (8192, 4096), "student_t3"),
             w=_t("W_gu", (28672, 4096), "normal", 0.02)),
        Gemm("down", 8192, 14336, 4096, x=_t("H", (8192, 14336), "student_t3"),
             w=_t("W_d", (4096, 14336), "normal", 0.02))],
        note="NVFP4 Llama-3-8B MLP forward; gate and up fused into one N=28672 GEMM")
    w[4] = Workload(4, "mxfp4_wgrad_h32_sr_8192tok", ("mxfp4",), [
        Gemm("down_wgrad", 8192, 4096, 14336, x=_t("X", (8192, 4096), "normal"),
             dy=_t("dY", (8192, 14336), "student_t3", 1e-3), passes=("wgrad",))],
        note="MXFP4 wgrad dW = dY^T X with Hadamard-32 on both operands, SR (seed 42) on dY")
    gl = []
    for name, kin, nout, xk in (("qkv", 4096, 6144, "student_t3"), ("o", 4096, 4096, "student_t3"),
                                ("gate_up", 4096, 28672, "student_t3"),
                                ("down", 14336, 4096, "student_t3")):
        gl.append(Gemm(name, 8192, kin, nout, x=_t("X_" + name, (8192, kin), xk),
                       w=_t("W_" + name, (nout, kin), "normal", 0.02),
                       dy=_t("dY_" + name, (8192, nout), "student_t3", 1e-3),
                       passes=("fwd", "dgrad", "wgrad")))
    w[5] = Workload(5, "llama3_8b_layer_linears_fwd_bwd_8192tok", ("mxfp8", "nvfp4"), gl,
                    note="Llama-3-8B decoder-layer linears (QKV, O, gate/up, down) fwd + bwd")
    return w


def materialize(wl: Workload, device="cpu") -> dict:
    """Draw every input tensor of a workload: {tensor name: bf16 tensor}."""
    out = {}
    idx = 0
    for g in wl.gemms:
        for t in (g.x, g.w, g.dy):
            if t is None:
                continue
            idx += 1
            out[t.name] = draw(t.kind, t.shape, 1000 * wl.index + idx, t.scale, device)
    return out
