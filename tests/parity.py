"""Comparison helpers shared by the GPU parity tests (CUDA path vs oracle)."""
import numpy as np
import torch

import oracle as orc

# GEMM tolerance: |C - C_ref| <= TOL * alpha * sum_k |a_k b_k| (fp32 accumulation
# order of K products; the fp32 worst case K * 2^-24 stays below it for K <= 16K).
GEMM_TOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def sf_valid_mask(rows: int, kblocks: int) -> np.ndarray:
    return orc.sf_swizzle(np.ones((rows, kblocks), dtype=np.uint8), fill=0).astype(bool)


def assert_quant_equal(q, ref, what=""):
    """Codes, scale bytes (at every real position of the swizzled layout), amax and
    tensor scale of the CUDA result equal the oracle's bit for bit."""
    codes = q.codes.cpu().numpy()
    assert codes.shape == ref.codes.shape, (codes.shape, ref.codes.shape)
    bad = np.flatnonzero(codes.ravel() != ref.codes.ravel())
    if bad.size:
        i = np.unravel_index(bad[0], codes.shape)
        raise AssertionError(f"{what}: {bad.size} code bytes differ; first at {i}: "
                             f"gpu {codes[i]:#04x} oracle {ref.codes[i]:#04x}")
    rows, kb = ref.sf_logical.shape
    exp = orc.sf_swizzle(ref.sf_logical, fill=0)
    mask = sf_valid_mask(rows, kb)
    got = q.sf.cpu().numpy()[:exp.size]
    bad = np.flatnonzero((got != exp) & mask)
    if bad.size:
        raise AssertionError(f"{what}: {bad.size} scale bytes differ; first at swizzled offset "
                             f"{bad[0]}: gpu {got[bad[0]]} oracle {exp[bad[0]]}")
    if ref.tensor_scale is not None:
        am = q.amax.cpu().numpy().astype(np.float32)
        ts = q.tensor_scale.cpu().numpy().astype(np.float32)
        assert np.array_equal(am, np.atleast_1d(np.asarray(ref.amax, dtype=np.float32))), (what, am, ref.amax)
        assert np.array_equal(ts, np.atleast_1d(np.asarray(ref.tensor_scale, dtype=np.float32))), \
            (what, ts, ref.tensor_scale)


def assert_gemm_close(c_gpu: torch.Tensor, c_ref: np.ndarray, c_abs: np.ndarray, what="",
                      tol: float = GEMM_TOL):
    c = c_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert c.shape == c_ref.shape, (c.shape, c_ref.shape)
    assert np.isfinite(c).all(), f"{what}: non-finite output"
    bound = tol * c_abs + 1e-30
    if c_gpu.dtype == torch.bfloat16:
        bound = bound + np.abs(c_ref) * 2.0 ** -8
    err = np.abs(c - c_ref)
    bad = np.flatnonzero(err > bound)
    if bad.size:
        i = np.unravel_index(bad[0], c.shape)
        raise AssertionError(f"{what}: {bad.size} of {c.size} outputs out of tolerance; first at {i}: "
                             f"gpu {c[i]!r} oracle {c_ref[i]!r} bound {bound[i]!r}")
    return float((err / np.maximum(c_abs, 1e-300)).max())


def sample_rows_cols(m: int, n: int, count: int = 128, seed: int = 7):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(m, size=min(count, m), replace=False))
    cols = np.sort(rng.choice(n, size=min(count, n), replace=False))
    return rows, cols
