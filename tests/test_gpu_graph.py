"""The library's calls under CUDA-graph capture: a quantize + GEMM sequence
captured once and replayed gives bit for bit what the same calls give when
launched one by one (every call launches on the capturing stream, allocates
nothing and synchronises nothing), and the replay keeps doing so after the
inputs change in place."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

FMTS = ["mxfp8", "mxfp4", "nvfp4", "moss", "nvfp4_local"]


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


def _sequence(mx, fmt, X, W, qx, qxt, qw, Y):
    mx.quantize_dual(X, fmt, row_out=qx, col_out=qxt)
    mx.quantize(W, fmt, "row", out=qw)
    mx.gemm(qx, qw, out=Y)


@pytest.mark.parametrize("fmt", FMTS)
def test_graph_replay_equals_eager_launches(mx, fmt):
    T, Kin, Nout = 512, 1024, 768
    X = workloads.draw("student_t3", (T, Kin), 201).cuda()
    W = workloads.draw("normal", (Nout, Kin), 202, 0.02).cuda()
    dev = X.device
    outs = [(mx.MXTensor(fmt, T, Kin, dev), mx.MXTensor(fmt, Kin, T, dev), mx.MXTensor(fmt, Nout, Kin, dev),
             torch.empty(T, Nout, dtype=torch.bfloat16, device=dev)) for _ in range(2)]
    eager, graphed = outs
    _sequence(mx, fmt, X, W, *eager)  # also the first call of every kernel (one-time setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _sequence(mx, fmt, X, W, *graphed)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK

    def same(a, b):
        for qa, qb in zip(a[:3], b[:3]):
            assert torch.equal(qa.codes, qb.codes) and torch.equal(qa.sf, qb.sf)
            assert torch.equal(qa.scalars, qb.scalars)
        assert torch.equal(a[3], b[3])

    same(eager, graphed)
    # new input values, same buffers: the replay recomputes everything from them
    X.copy_(workloads.draw("student_t3", (T, Kin), 203).cuda())
    _sequence(mx, fmt, X, W, *eager)
    g.replay()
    torch.cuda.synchronize()
    same(eager, graphed)
