"""The linear layer's forward, data-gradient and weight-gradient passes through the
C ABI (mx_linear_fwd / mx_linear_bwd) against the oracle's composition of the
same quantizations and GEMMs."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads
from parity import assert_gemm_close, assert_quant_equal, bits

pytestmark = pytest.mark.gpu

FMTS = ["mxfp8", "mxfp4", "nvfp4", "moss", "nvfp4_local"]


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("tkn", [(256, 512, 384), (384, 1024, 256)])
def test_forward(mx, fmt, tkn):
    T, Kin, Nout = tkn
    X = workloads.draw("student_t3", (T, Kin), 61)
    W = workloads.draw("normal", (Nout, Kin), 62, 0.02)
    for out_dtype in (torch.bfloat16, torch.float32):
        Y = mx.linear_fwd(X.cuda(), W.cuda(), fmt, out_dtype=out_dtype)
        ref, cabs = orc.gemm(orc.quantize(bits(X), fmt), orc.quantize(bits(W), fmt))
        assert_gemm_close(Y, ref, cabs, f"fwd {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_backward(mx, fmt):
    T, Kin, Nout = 512, 256, 768
    X = workloads.draw("student_t3", (T, Kin), 71)
    W = workloads.draw("normal", (Nout, Kin), 72, 0.02)
    dY = workloads.draw("student_t3", (T, Nout), 73, 1e-3)
    dX, dW = mx.linear_bwd(dY.cuda(), X.cuda(), W.cuda(), fmt, dx_dtype=torch.float32)
    ref, cabs = orc.gemm(orc.quantize(bits(dY), fmt), orc.quantize(bits(W), fmt, "col"))
    assert_gemm_close(dX, ref, cabs, f"dgrad {fmt}")
    ref, cabs = orc.gemm(orc.quantize(bits(dY), fmt, "col"), orc.quantize(bits(X), fmt, "col"))
    assert_gemm_close(dW, ref, cabs, f"wgrad {fmt}")


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
@pytest.mark.parametrize("seed,sid", [(42, 0), (1234, 5)])
def test_fp4_wgrad_hadamard_sr(mx, fmt, seed, sid):
    """The weight gradient with H32 on both operands along tokens and SR on dY
    (the mxfp route of the pages, and the same options on NVFP4)."""
    T, Kin, Nout = 512, 256, 384
    X = workloads.draw("normal", (T, Kin), 81)
    W = workloads.draw("normal", (Nout, Kin), 82, 0.02)
    dY = workloads.draw("student_t3", (T, Nout), 83, 1e-3)
    _, dW = mx.linear_bwd(dY.cuda(), X.cuda(), W.cuda(), fmt, wgrad_hadamard=True,
                          wgrad_dy_rounding="sr", seed=seed, stream_id=sid, need_dx=False)
    ra = orc.quantize(bits(dY), fmt, "col", rounding="sr", seed=seed, stream_id=sid, hadamard=True)
    rb = orc.quantize(bits(X), fmt, "col", hadamard=True)
    ref, cabs = orc.gemm(ra, rb, extra_alpha=1.0 / 32)
    assert_gemm_close(dW, ref, cabs, f"wgrad {fmt} H32+SR")
    # and the result estimates the exact dY^T X
    exact = (dY.double().t() @ X.double()).numpy()
    rel = np.linalg.norm(dW.cpu().double().numpy() - exact) / np.linalg.norm(exact)
    assert rel < 0.25


def test_workspace_too_small(mx):
    X = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.linear_fwd(X, W, "mxfp8", workspace=ws)
    assert e.value.code == mx.MX_ERR_WORKSPACE


@pytest.mark.parametrize("fmt", ["mxfp8", "moss"])
def test_e4m3_wgrad_stochastic_rounding(mx, fmt):
    """E4M3 formats take SR on the weight gradient's dY^T too (same Philox stream)."""
    T, Kin, Nout = 512, 256, 384
    X = workloads.draw("normal", (T, Kin), 86)
    W = workloads.draw("normal", (Nout, Kin), 87, 0.02)
    dY = workloads.draw("student_t3", (T, Nout), 88, 1e-3)
    _, dW = mx.linear_bwd(dY.cuda(), X.cuda(), W.cuda(), fmt, wgrad_dy_rounding="sr", seed=9, stream_id=2,
                          need_dx=False)
    ra = orc.quantize(bits(dY), fmt, "col", rounding="sr", seed=9, stream_id=2)
    rb = orc.quantize(bits(X), fmt, "col")
    ref, cabs = orc.gemm(ra, rb)
    assert_gemm_close(dW, ref, cabs, f"wgrad {fmt} SR")


# --------------------------------------------- saved backward state (one read per tensor)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("hadamard,rounding", [(False, "rne"), (True, "sr")])
def test_saved_state_path_equals_the_plain_layer(mx, fmt, hadamard, rounding):
    """mx_linear_fwd_save + mx_linear_bwd_saved read X, W and dY once each and
    give bit for bit what mx_linear_fwd + mx_linear_bwd give, and the oracle's
    composition of the same quantizations and GEMMs."""
    if hadamard and fmt not in ("mxfp8", "mxfp4", "nvfp4"):
        pytest.skip("the Hadamard transform is offered on the MX formats and NVFP4")
    T, Kin, Nout = 512, 256, 768
    X = workloads.draw("student_t3", (T, Kin), 171).cuda()
    W = workloads.draw("normal", (Nout, Kin), 172, 0.02).cuda()
    dY = workloads.draw("student_t3", (T, Nout), 173, 1e-3).cuda()
    kw = dict(wgrad_hadamard=hadamard, wgrad_dy_rounding=rounding, seed=42, stream_id=3)
    Y0 = mx.linear_fwd(X, W, fmt, out_dtype=torch.float32)
    dX0, dW0 = mx.linear_bwd(dY, X, W, fmt, dx_dtype=torch.float32, **kw)
    Y1, saved = mx.linear_fwd_save(X, W, fmt, out_dtype=torch.float32, **kw)
    dX1, dW1 = mx.linear_bwd_saved(dY, saved, Kin, fmt, dx_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK
    assert torch.equal(Y0, Y1) and torch.equal(dX0, dX1) and torch.equal(dW0, dW1)
    # one of the three against the oracle (the others are checked by the plain-layer tests)
    ra = orc.quantize(bits(dY.cpu()), fmt, "col", rounding=rounding, seed=42, stream_id=3, hadamard=hadamard)
    rb = orc.quantize(bits(X.cpu()), fmt, "col", hadamard=hadamard)
    ref, cabs = orc.gemm(ra, rb, extra_alpha=(1.0 / 32 if hadamard else 1.0))
    assert_gemm_close(dW1, ref, cabs, f"wgrad from saved state {fmt}")


@pytest.mark.parametrize("fmt", ["nvfp4", "moss"])
def test_saved_state_path_with_caller_amax(mx, fmt):
    """A caller-supplied tensor amax skips the amax passes: with the true maxima
    the results are those of the plain layer; with a larger amax they are the
    oracle's quantization at that amax."""
    T, Kin, Nout = 256, 512, 512  # every GEMM's K a multiple of 256, as FP4 requires
    X = workloads.draw("student_t3", (T, Kin), 181).cuda()
    W = workloads.draw("normal", (Nout, Kin), 182, 0.02).cuda()
    dY = workloads.draw("student_t3", (T, Nout), 183, 1e-3).cuda()
    am = lambda t: t.float().abs().max().reshape(1)  # noqa: E731
    Y0 = mx.linear_fwd(X, W, fmt, out_dtype=torch.float32)
    dX0, dW0 = mx.linear_bwd(dY, X, W, fmt, dx_dtype=torch.float32)
    Y1, saved = mx.linear_fwd_save(X, W, fmt, out_dtype=torch.float32, x_amax=am(X), w_amax=am(W))
    dX1, dW1 = mx.linear_bwd_saved(dY, saved, Kin, fmt, dx_dtype=torch.float32, dy_amax=am(dY))
    assert torch.equal(Y0, Y1) and torch.equal(dX0, dX1) and torch.equal(dW0, dW1)
    big = am(X) * 4
    Y2, _ = mx.linear_fwd_save(X, W, fmt, out_dtype=torch.float32, x_amax=big)
    ref, cabs = orc.gemm(orc.quantize(bits(X.cpu()), fmt, amax_in=float(big)), orc.quantize(bits(W.cpu()), fmt))
    assert_gemm_close(Y2, ref, cabs, f"fwd with caller amax {fmt}")


def test_saved_state_buffers_too_small(mx):
    X = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.linear_fwd_save(X, W, "mxfp8", saved=torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.code == mx.MX_ERR_WORKSPACE
    _, sv = mx.linear_fwd_save(X, W, "mxfp8")
    with pytest.raises(mx.MXError) as e:
        mx.linear_bwd_saved(X, sv[:1024], 256, "mxfp8")
    assert e.value.code == mx.MX_ERR_WORKSPACE


def _bwd_inputs(T, Kin, Nout, seed):
    X = workloads.draw("student_t3", (T, Kin), seed).cuda()
    W = workloads.draw("normal", (Nout, Kin), seed + 1, 0.02).cuda()
    dY = workloads.draw("student_t3", (T, Nout), seed + 2, 1e-3).cuda()
    return X, W, dY


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
def test_gradient_fork_equals_one_stream(mx, fmt):
    """The weight gradient on the library's side stream gives bit for bit what
    the two gradients give one after the other on the caller's stream, for the
    plain and the saved-state backward, launched eagerly and replayed from a
    captured graph (many tiles per GEMM, so the two really run side by side)."""
    T, Kin, Nout = 2048, 1024, 1536
    X, W, dY = _bwd_inputs(T, Kin, Nout, 181)
    kw = dict(wgrad_hadamard=fmt == "mxfp4", wgrad_dy_rounding="sr" if fmt == "mxfp4" else "rne", seed=7,
              stream_id=1)
    _, saved = mx.linear_fwd_save(X, W, fmt, **kw)
    mx.set_bwd_fork(False)
    try:
        ref = mx.linear_bwd(dY, X, W, fmt, **kw) + mx.linear_bwd_saved(dY, saved, Kin, fmt, **kw)
    finally:
        mx.set_bwd_fork(True)
    got = mx.linear_bwd(dY, X, W, fmt, **kw) + mx.linear_bwd_saved(dY, saved, Kin, fmt, **kw)
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    ws = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "bwd_saved"), dtype=torch.uint8, device="cuda")
    dX = torch.full_like(got[2], float("nan"))
    dW = torch.full_like(got[3], float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.linear_bwd_saved(dY, saved, Kin, fmt, workspace=ws, dX=dX, dW=dW, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dX, ref[2]) and torch.equal(dW, ref[3])


def test_gradient_fork_first_captured_call_in_a_thread(mx):
    """A thread whose first backward call is made under graph capture (before
    its side stream exists) runs both gradients on the capturing stream and
    gives the same results."""
    import threading

    T, Kin, Nout, fmt = 1024, 512, 768, "nvfp4"
    X, W, dY = _bwd_inputs(T, Kin, Nout, 191)
    ref = mx.linear_bwd(dY, X, W, fmt)
    ws = torch.empty(mx.workspace_bytes(T, Kin, Nout, fmt, "bwd"), dtype=torch.uint8, device="cuda")
    dX, dW = torch.empty_like(ref[0]), torch.empty_like(ref[1])
    torch.cuda.synchronize()
    out = {}

    def body():
        try:
            torch.cuda.set_device(0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                mx.linear_bwd(dY, X, W, fmt, workspace=ws, dX=dX, dW=dW)
            g.replay()
            torch.cuda.synchronize()
            out["ok"] = True
        except Exception as e:  # reported below, in the test's own thread
            out["err"] = e

    t = threading.Thread(target=body)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    assert torch.equal(dX, ref[0]) and torch.equal(dW, ref[1])
