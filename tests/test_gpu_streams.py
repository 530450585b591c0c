"""Launches go to the caller's stream: a GEMM on a side stream, and the same
GEMM captured into a CUDA graph on that stream and replayed, give the
default-stream result bit for bit."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_gemm_on_side_stream_and_in_a_graph(mx, fmt):
    M, N, K = 4096, 4096, 1024  # enough tiles for the CTA-pair kernel
    qa = mx.quantize(workloads.draw("student_t3", (M, K), 5).cuda(), fmt)
    qb = mx.quantize(workloads.draw("normal", (N, K), 6, 0.02).cuda(), fmt)
    ref = mx.gemm(qa, qb, out_dtype=torch.float32)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    out = torch.zeros_like(ref)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mx.gemm(qa, qb, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

    out2 = torch.zeros_like(ref)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.gemm(qa, qb, out=out2, stream=s)
    torch.cuda.synchronize()
    assert not out2.any()  # capture records, it does not run
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)
    assert mx.last_device_status() == mx.MX_OK


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_linear_layer_captured_in_a_graph(mx, fmt):
    """The whole layer (quantize producers, amax, GEMMs) for forward and backward,
    captured on a side stream with caller-owned workspace and outputs, replays
    to the eagerly computed result bit for bit."""
    T, Kin, Nout = 1024, 1024, 1536
    X = workloads.draw("student_t3", (T, Kin), 21).cuda()
    W = workloads.draw("normal", (Nout, Kin), 22, 0.02).cuda()
    dY = workloads.draw("student_t3", (T, Nout), 23, 1e-3).cuda()
    ws = torch.empty(max(mx.workspace_bytes(T, Kin, Nout, fmt, "fwd"), mx.workspace_bytes(T, Kin, Nout, fmt, "bwd")),
                     dtype=torch.uint8, device="cuda")
    Y_ref = mx.linear_fwd(X, W, fmt, workspace=ws)
    dX_ref, dW_ref = mx.linear_bwd(dY, X, W, fmt, workspace=ws)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    Y = torch.zeros_like(Y_ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.linear_fwd(X, W, fmt, workspace=ws, out=Y, stream=s)
        dX, dW = mx.linear_bwd(dY, X, W, fmt, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y, Y_ref)
    assert torch.equal(dX, dX_ref)
    assert torch.equal(dW, dW_ref)
    assert mx.last_device_status() == mx.MX_OK
