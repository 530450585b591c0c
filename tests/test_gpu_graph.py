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


@pytest.mark.parametrize("streams", [2, 3])
def test_multi_stream_step_graph_equals_eager_step(mx, streams):
    """The bench's step captured on two or three streams (each layer's dY
    producer and gradient GEMMs on further streams, events for the
    cross-stream reads) gives bit for bit the outputs of the same calls issued
    one by one on one stream: small layers, both schemes of the layer-linears
    workload."""
    import bench

    gl = []
    for i, (kin, nout) in enumerate(((512, 768), (768, 512), (512, 1024))):
        gl.append(workloads.Gemm(f"l{i}", 256, kin, nout, x=workloads._t(f"X{i}", (256, kin), "student_t3"),
                                 w=workloads._t(f"W{i}", (nout, kin), "normal", 0.02),
                                 dy=workloads._t(f"dY{i}", (256, nout), "student_t3", 1e-3),
                                 passes=("fwd", "dgrad", "wgrad")))
    wl = workloads.Workload(0, "small_layers", ("mxfp8", "nvfp4"), gl)
    dev = torch.device("cuda", 0)
    inputs = workloads.materialize(wl, device=dev)
    plans = [bench.Plan(mx, wl, fmt, dev) for fmt in wl.formats]

    def outputs():
        return [t.clone() for p in plans for e in p.gemms for t in (e["Y"], e["dX"], e["dW"])]

    for p in plans:
        for c in p.calls(inputs):
            c[1]()
    torch.cuda.synchronize()
    eager = outputs()
    for p in plans:  # clear, so that the graph's replay must write everything again
        for e in p.gemms:
            for k in ("Y", "dX", "dW"):
                e[k].fill_(float("nan"))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    role_calls = [(p.fmt,) + c for p in plans for c in p.roles(inputs)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if streams == 2:
            bench.issue_two_streams(role_calls, s1)
        else:
            bench.issue_three_streams(role_calls, s1, s2)
    g.replay()
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK
    for a, b in zip(eager, outputs()):
        assert torch.equal(a, b)
