"""Parity of the tcgen05 block-scaled GEMM with the oracle's fp64 GEMM over the
dequantised operands (and bit-exact where fp32 accumulation is exact)."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads
from parity import assert_gemm_close, assert_quant_equal, bits

pytestmark = pytest.mark.gpu

FMTS = ["mxfp8", "mxfp4", "nvfp4", "moss", "nvfp4_local"]
FP4 = ("mxfp4", "nvfp4", "nvfp4_local")


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    yield m
    m.set_gemm_variant("auto")


def quant_pair(mx, a, b, fmt, **kw):
    qa, qb = mx.quantize(a.cuda(), fmt, **kw), mx.quantize(b.cuda(), fmt, **kw)
    ra, rb = orc.quantize(bits(a), fmt, **kw), orc.quantize(bits(b), fmt, **kw)
    return qa, qb, ra, rb


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("variant", ["cta_n128", "cta_n256", "pair", "pair_ws"])
def test_exact_small_integers(mx, fmt, variant):
    """Small-integer codes with power-of-two scales: every partial sum is exact in
    fp32, so the tensor core must reproduce the fp64 oracle bit for bit."""
    mx.set_gemm_variant(variant)
    rng = np.random.default_rng(1)
    vals = np.array([-6, -4, -3, -2, -1, 0, 1, 2, 3, 4, 6])
    a = torch.tensor(rng.choice(vals, (256, 512)), dtype=torch.float32).to(torch.bfloat16)
    b = torch.tensor(rng.choice(vals, (384, 512)), dtype=torch.float32).to(torch.bfloat16)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt, rule="ceil")
    c = mx.gemm(qa, qb)
    ref, _ = orc.gemm(ra, rb)
    assert np.array_equal(c.cpu().numpy().astype(np.float64), ref)
    assert np.array_equal(ref, (a.double() @ b.double().t()).numpy())


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("variant", ["cta_n128", "cta_n256", "pair", "pair_ws"])
def test_scale_factor_layout_one_hot(mx, fmt, variant):
    """Pins the swizzled scale layout against the hardware: with all-ones inputs,
    raise single scale bytes of A and of B in the GPU buffers (at the offsets the
    layout definition gives) and check every output against the oracle GEMM
    computed with the same raised logical scales."""
    mx.set_gemm_variant(variant)
    M, N, K = 256, 384, 1024 if fmt in FP4 else 512
    a = torch.ones(M, K, dtype=torch.bfloat16)
    b = torch.ones(N, K, dtype=torch.bfloat16)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    rng = np.random.default_rng(3)
    for q, r in ((qa, ra), (qb, rb)):
        kb = r.sf_logical.shape[1]
        sf = q.sf.cpu().numpy()
        for row in range(r.rows):
            blk = int(rng.integers(0, kb))
            # E8M0: +1 doubles the scale; UE4M3 (0x7E here): -8 halves it
            new = int(r.sf_logical[row, blk]) + (1 if fmt not in ("nvfp4", "nvfp4_local") else -8)
            r.sf_logical[row, blk] = new
            sf[orc.sf_index(row, blk, kb)] = new
        q.sf.copy_(torch.from_numpy(sf))
    c = mx.gemm(qa, qb)
    ref, cabs = orc.gemm(ra, rb)
    assert_gemm_close(c, ref, cabs, f"one-hot {fmt}", tol=1e-6)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mnk", [(256, 256, 256), (200, 136, 512), (384, 640, 1024), (130, 520, 256)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_random_gemm(mx, fmt, mnk, out_dtype):
    M, N, K = mnk
    if fmt in FP4 and K % 256:
        K = 256 * ((K + 255) // 256)
    a = workloads.draw("student_t3", (M, K), 40 + M)
    b = workloads.draw("normal", (N, K), 41 + N, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    for variant in ("cta_n128", "cta_n256", "pair", "pair_ws"):
        mx.set_gemm_variant(variant)
        c = mx.gemm(qa, qb, out_dtype=out_dtype)
        ref, cabs = orc.gemm(ra, rb)
        assert_gemm_close(c, ref, cabs, f"{fmt} {mnk} {variant}")


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
def test_hadamard_alpha(mx, fmt):
    mx.set_gemm_variant("auto")
    """Both operands transformed: the epilogue applies the 1/32 of (Ha)^T(Hb) = 32 a^T b."""
    dy = workloads.draw("student_t3", (512, 256), 51, 1e-3)
    x = workloads.draw("normal", (512, 384), 52)
    qa = mx.quantize(dy.cuda(), fmt, "col", hadamard=True)
    qb = mx.quantize(x.cuda(), fmt, "col", hadamard=True)
    ra = orc.quantize(bits(dy), fmt, "col", hadamard=True)
    rb = orc.quantize(bits(x), fmt, "col", hadamard=True)
    c = mx.gemm(qa, qb, extra_alpha=0.5)
    ref, cabs = orc.gemm(ra, rb, extra_alpha=0.5 / 32)
    assert_gemm_close(c, ref, cabs, f"H32 {fmt}")


def test_mixed_hadamard_rejected(mx):
    x = workloads.draw("normal", (256, 256), 1).cuda()
    qa = mx.quantize(x, "mxfp8", "col", hadamard=True)
    qb = mx.quantize(x, "mxfp8", "col")
    with pytest.raises(mx.MXError) as e:
        mx.gemm(qa, qb)
    assert e.value.code == mx.MX_ERR_INVALID_ARG


def test_gemm_k_alignment_rejected(mx):
    x = workloads.draw("normal", (128, 96), 1).cuda()
    q = mx.quantize(x, "mxfp8")
    with pytest.raises(mx.MXError) as e:
        mx.gemm(q, q)
    assert e.value.code == mx.MX_ERR_ALIGNMENT
    assert mx.last_device_status() == mx.MX_OK


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("pv", ["pair", "pair_ws"])
def test_pair_kernel_many_tiles_and_tails(mx, pv, fmt):
    """Enough 256 x 256 tiles that every cluster runs several (persistent
    loop, accumulator hand-off between tiles), with ragged M and N tails."""
    mx.set_gemm_variant(pv)
    M, N, K = 1280 + 72, 1536 + 40, 512
    a = workloads.draw("student_t3", (M, K), 77)
    b = workloads.draw("normal", (N, K), 78, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    rows = np.r_[0:40, M - 80:M]
    for out_dtype in (torch.float32, torch.bfloat16):
        c = mx.gemm(qa, qb, out_dtype=out_dtype)
        ref, cabs = orc.gemm(ra, rb, rows=rows)
        assert_gemm_close(c[torch.as_tensor(rows, device=c.device)], ref, cabs, f"pair {fmt}")
    mx.set_gemm_variant("auto")


# ------------------------------------------------ quantized epilogue (next layer)
@pytest.mark.parametrize("in_fmt", FMTS)
@pytest.mark.parametrize("out_fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("variant", ["cta_n128", "cta_n256", "pair", "pair_ws"])
def test_gemm_quantized_epilogue(mx, in_fmt, out_fmt, variant):
    """The operand the epilogue writes equals the oracle's rowwise MX quantization
    of the same kernel's fp32 output, bit for bit: both runs issue the same MMAs
    in the same order, so the fp32 sums are identical."""
    mx.set_gemm_variant(variant)
    M, N, K = 424, 640, 512
    a = workloads.draw("student_t3", (M, K), 91)
    b = workloads.draw("normal", (N, K), 92, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, in_fmt)
    c32 = mx.gemm(qa, qb, extra_alpha=0.75, out_dtype=torch.float32)
    q = mx.gemm_quantized(qa, qb, out_fmt, extra_alpha=0.75)
    torch.cuda.synchronize()
    assert (q.rows, q.k) == (M, N)
    # the fp32 result the epilogue quantizes is itself the oracle GEMM within 1e-3
    ref, cabs = orc.gemm(ra, rb, extra_alpha=0.75)
    assert_gemm_close(c32, ref, cabs, f"{in_fmt} fp32 before the epilogue quantizer {variant}")
    assert_quant_equal(q, orc.quantize_rows_f32(c32.cpu().numpy(), out_fmt), f"{in_fmt}->{out_fmt} {variant}")
    mx.set_gemm_variant("auto")


@pytest.mark.parametrize("out_fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("pv", ["pair", "pair_ws"])
def test_gemm_quantized_many_tiles_feeds_next_gemm(mx, pv, out_fmt):
    """Pair kernel over many 256 x 256 tiles with a ragged M tail; the result is a
    valid operand: a second GEMM consuming it matches the oracle GEMM of the
    oracle-quantized first result."""
    mx.set_gemm_variant(pv)
    # N is the next GEMM's K (a multiple of 128 / 256); 1408 leaves a ragged 256-column tile
    M, N, K = 1280 + 72, (1408 if out_fmt == "mxfp8" else 1792), 512
    a = workloads.draw("student_t3", (M, K), 93)
    b = workloads.draw("normal", (N, K), 94, 0.02)
    qa, qb, _, _ = quant_pair(mx, a, b, "mxfp8")
    c32 = mx.gemm(qa, qb, out_dtype=torch.float32)
    q = mx.gemm_quantized(qa, qb, out_fmt)
    ref = orc.quantize_rows_f32(c32.cpu().numpy(), out_fmt)
    assert_quant_equal(q, ref, f"many tiles -> {out_fmt}")
    w2 = workloads.draw("normal", (256, N), 95, 0.02)
    q2 = mx.quantize(w2.cuda(), out_fmt)
    r2 = orc.quantize(bits(w2), out_fmt)
    y = mx.gemm(q, q2)
    yref, yabs = orc.gemm(ref, r2)
    assert_gemm_close(y, yref, yabs, "second GEMM on the epilogue operand")
    mx.set_gemm_variant("auto")


def test_gemm_quantized_rejects(mx):
    x = workloads.draw("normal", (256, 256), 1).cuda()
    q = mx.quantize(x, "mxfp8")
    qn = mx.quantize(workloads.draw("normal", (48, 256), 2).cuda(), "mxfp8")  # N = 48: not whole blocks
    with pytest.raises(mx.MXError) as e:  # the C entry checks N % 32 itself
        mx.gemm_quantized(q, qn, "mxfp8", out=mx.MXTensor("mxfp8", 256, 64))
    assert e.value.code == mx.MX_ERR_ALIGNMENT
    with pytest.raises(mx.MXError) as e:
        mx.gemm_quantized(q, q, "nvfp4")
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
    assert mx.last_device_status() == mx.MX_OK


@pytest.mark.parametrize("fmt,K", [("mxfp8", 384), ("mxfp8", 1280), ("mxfp4", 768), ("mxfp4", 1536)])
@pytest.mark.parametrize("pv", ["pair", "pair_ws"])
def test_pair_kernel_both_stage_depths(mx, pv, fmt, K):
    """K a multiple of 256 bytes takes the three-stage ring of 256-byte K-stages,
    otherwise the five-stage ring of 128-byte stages: both against the oracle."""
    mx.set_gemm_variant(pv)
    M, N = 512 + 64, 768 + 32
    a = workloads.draw("student_t3", (M, K), 101)
    b = workloads.draw("normal", (N, K), 102, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    c = mx.gemm(qa, qb)
    ref, cabs = orc.gemm(ra, rb)
    assert_gemm_close(c, ref, cabs, f"{fmt} K={K}")
    mx.set_gemm_variant("auto")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mnk", [(33, 40, 256), (300, 1000, 512), (257, 264, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("pv", ["pair", "pair_ws"])
def test_pair_output_stays_inside_a_strided_view(mx, pv, fmt, mnk, out_dtype):
    """The CTA-pair kernel writes its bf16 / fp32 output (TMA stores of 32-row
    boxes, clipped at M and N) into a view of a wider, taller buffer: every
    element of the view matches the oracle and nothing past column N or row M
    is touched."""
    M, N, K = mnk
    a = workloads.draw("student_t3", (M, K), 90 + M)
    b = workloads.draw("normal", (N, K), 91 + N, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    ld = ((N + 24 + 7) // 8) * 8
    buf = torch.full((M + 16, ld), float("nan"), dtype=out_dtype, device="cuda")
    out = buf[:M, :N]
    mx.set_gemm_variant(pv)
    try:
        mx.gemm(qa, qb, out=out)
    finally:
        mx.set_gemm_variant("auto")
    ref, cabs = orc.gemm(ra, rb)
    assert_gemm_close(out, ref, cabs, f"pair strided {fmt} {mnk}")
    assert torch.isnan(buf[:M, N:]).all()
    assert torch.isnan(buf[M:, :]).all()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("K", [256, 512])
@pytest.mark.parametrize("pv", ["pair", "pair_ws"])
def test_pair_kernel_short_k_many_tiles(mx, pv, fmt, K):
    """Every cluster runs several tiles of one or two K-stages, so the
    epilogue warps' scale stores run ahead across several future tiles and the
    accumulator changes hands every stage or two."""
    M, N = 4096 + 40, 4096
    a = workloads.draw("student_t3", (M, K), 95 + K)
    b = workloads.draw("normal", (N, K), 96 + K, 0.02)
    qa, qb, ra, rb = quant_pair(mx, a, b, fmt)
    rows = np.r_[0:32, 2048:2080, M - 64:M]
    mx.set_gemm_variant(pv)
    try:
        for out_dtype in (torch.float32, torch.bfloat16):
            c = mx.gemm(qa, qb, out_dtype=out_dtype)
            ref, cabs = orc.gemm(ra, rb, rows=rows)
            assert_gemm_close(c[torch.as_tensor(rows, device=c.device)], ref, cabs, f"pair short K {fmt} {K}")
    finally:
        mx.set_gemm_variant("auto")
