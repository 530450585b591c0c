"""The GEMM epilogue's output amax (mx_gemm_amax): the absolute maximum of the
output as written equals torch's max |C| over the same tensor bit for bit, in
every kernel variant, for fp32 and bf16 outputs and ragged shapes; columns of
the row stride past N and rows past M do not count; the word is zeroed by the
call; and it serves as the next quantization's tensor amax."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

VARIANTS = ["cta_n128", "cta_n256", "pair", "pair_ws"]


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    yield m
    m.set_gemm_variant("auto")


def _operands(mx, fmt, M, N, K, seed):
    a = workloads.draw("student_t3", (M, K), seed).cuda()
    b = workloads.draw("normal", (N, K), seed + 1, 0.02).cuda()
    return mx.quantize(a, fmt), mx.quantize(b, fmt)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mnk", [(256, 256, 512), (200, 136, 512), (130, 520, 256), (1000, 1048, 1024)])
def test_amax_equals_max_abs_of_output(mx, fmt, variant, out_dtype, mnk):
    M, N, K = mnk
    qa, qb = _operands(mx, fmt, M, N, K, 300 + M)
    mx.set_gemm_variant(variant)
    am = torch.full((1,), 123.0, device="cuda")
    c = mx.gemm(qa, qb, out_dtype=out_dtype, amax_out=am)
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK
    ref = c.abs().max().float()
    assert am.item() == ref.item(), (variant, am.item(), ref.item())
    # the same call without the amax writes the same output
    assert torch.equal(mx.gemm(qa, qb, out_dtype=out_dtype), c)


@pytest.mark.parametrize("variant", VARIANTS)
def test_amax_in_ragged_corner_and_strided_output(mx, variant):
    """The largest product sits at the last row and column of a ragged shape;
    the output is a view into wider rows prefilled with larger values, which
    must neither be written nor counted."""
    M, N, K = 200, 136, 512
    a = workloads.draw("normal", (M, K), 310).cuda()
    b = workloads.draw("normal", (N, K), 311).cuda()
    a[M - 1] = 4.0
    b[N - 1] = 4.0
    qa, qb = mx.quantize(a, "mxfp8"), mx.quantize(b, "mxfp8")
    wide = torch.full((M + 8, N + 24), -1e30, device="cuda")
    out = wide[:M, :N]
    am = torch.zeros(1, device="cuda")
    mx.set_gemm_variant(variant)
    mx.gemm(qa, qb, out=out, amax_out=am)
    torch.cuda.synchronize()
    assert (wide[:, N:] == -1e30).all() and (wide[M:] == -1e30).all()
    assert am.item() == out.abs().max().item() == abs(out[M - 1, N - 1].item())


def test_amax_of_empty_products_is_zero(mx):
    qa, qb = _operands(mx, "mxfp8", 128, 128, 256, 320)
    q0 = mx.quantize(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), "mxfp8")
    am = torch.full((1,), 7.0, device="cuda")
    mx.gemm(q0, qb, amax_out=am)
    torch.cuda.synchronize()
    assert am.item() == 0.0
    am.fill_(7.0)
    mx.gemm(qa, q0, amax_out=am)
    torch.cuda.synchronize()
    assert am.item() == 0.0


def test_amax_rezeroed_on_every_call(mx):
    """A second call with a smaller output reports its own amax, not the first's."""
    qa, qb = _operands(mx, "nvfp4", 256, 256, 512, 330)
    am = torch.zeros(1, device="cuda")
    big = mx.gemm(qa, qb, extra_alpha=64.0, amax_out=am)
    torch.cuda.synchronize()
    assert am.item() == big.abs().max().item()
    small = mx.gemm(qa, qb, extra_alpha=0.5, amax_out=am)
    torch.cuda.synchronize()
    assert am.item() == small.abs().max().item() < big.abs().max().item()


@pytest.mark.parametrize("fmt", ["nvfp4", "moss"])
def test_amax_feeds_the_next_quantization(mx, fmt):
    """Y's epilogue amax given to the next producer as amax_in gives the same
    codes, scales and tensor scale as the producer's own amax pass over Y."""
    T, Kin, Nout = 512, 1024, 768
    qx, qw = _operands(mx, "nvfp4", T, Nout, Kin, 340)
    am = torch.zeros(1, device="cuda")
    y = mx.gemm(qx, qw, out_dtype=torch.bfloat16, amax_out=am)
    q_own = mx.quantize(y, fmt)
    q_fed = mx.quantize(y, fmt, amax_in=am)
    torch.cuda.synchronize()
    assert torch.equal(q_own.codes, q_fed.codes) and torch.equal(q_own.sf, q_fed.sf)
    assert torch.equal(q_own.scalars, q_fed.scalars)


def test_amax_under_graph_replay(mx):
    """The zeroing and the GEMM captured into a CUDA graph: every replay reports
    the amax of the current inputs."""
    M, N, K = 512, 384, 512
    a = workloads.draw("student_t3", (M, K), 350).cuda()
    b = workloads.draw("normal", (N, K), 351, 0.02).cuda()
    qa, qb = mx.MXTensor("mxfp8", M, K, a.device), mx.MXTensor("mxfp8", N, K, a.device)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    am = torch.zeros(1, device="cuda")

    def seq():
        mx.quantize(a, "mxfp8", out=qa)
        mx.quantize(b, "mxfp8", out=qb)
        mx.gemm(qa, qb, out=y, amax_out=am)

    seq()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        seq()
    for scale in (1.0, 0.25):
        a.copy_(workloads.draw("student_t3", (M, K), 352).cuda() * scale)
        g.replay()
        torch.cuda.synchronize()
        assert am.item() == y.abs().max().float().item()


def test_amax_word_must_be_aligned(mx):
    """A misaligned amax word is refused on the host, before anything launches."""
    import ctypes as C

    qa, qb = _operands(mx, "mxfp8", 128, 128, 256, 360)
    c = torch.empty(128, 128, device="cuda")
    buf = torch.zeros(8, dtype=torch.float32, device="cuda")
    ca, cb = qa._c(), qb._c()
    rc = mx.lib().mx_gemm_amax(C.byref(ca), C.byref(cb), 1.0, C.c_void_p(c.data_ptr()), 128, 0,
                               C.c_void_p(buf.data_ptr() + 2), None)
    assert rc == mx.MX_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.equal(buf, torch.zeros_like(buf))
