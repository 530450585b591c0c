"""Parity of the CUDA quantize producer with the oracle: bit-exact codes, scale
bytes (in the tensor core's layout), amax and tensor scale."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads
from parity import assert_quant_equal, bits, sf_valid_mask

pytestmark = pytest.mark.gpu

FMTS = ["mxfp8", "mxfp4", "nvfp4", "moss"]


@pytest.fixture(scope="module", params=["auto", "direct", "tile"])
def mx(request):
    """The library, once per producer implementation (outputs must not depend on it)."""
    import fp4_precision_gemms_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    m.set_quant_impl(request.param)
    yield m
    m.set_quant_impl("auto")


def run_both(mx, x, fmt, direction="row", **kw):
    q = mx.quantize(x.cuda(), fmt, direction, **kw)
    torch.cuda.synchronize()
    ref = orc.quantize(bits(x), fmt, direction, **kw)
    return q, ref


def test_status_word_starts_clear(mx):
    assert mx.last_device_status() == mx.MX_OK


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("direction", ["row", "col"])
def test_every_bf16_pattern(mx, fmt, direction):
    """All 65280 finite bf16 values, seeded-shuffled so every block mixes binades."""
    pats = workloads.all_bf16_patterns()
    g = torch.Generator().manual_seed(0)
    pats = pats[torch.randperm(pats.numel(), generator=g)]
    x = torch.zeros(512 * 128, dtype=torch.bfloat16)
    x[:pats.numel()] = pats
    x = x.view(512, 128)
    q, ref = run_both(mx, x, fmt, direction)
    assert_quant_equal(q, ref, f"{fmt}/{direction}")


@pytest.mark.parametrize("fmt,rule", [(f, r) for f in ("mxfp8", "mxfp4", "moss")
                                      for r in ("floor", "ceil", "nearest")])
def test_scale_rules(mx, fmt, rule):
    x = workloads.draw("outliers", (256, 256), 11)
    for direction in ("row", "col"):
        q, ref = run_both(mx, x, fmt, direction, rule=rule)
        assert_quant_equal(q, ref, f"{fmt}/{rule}/{direction}")


SHAPES = [(416, 544), (128, 4096), (32, 32), (4096, 64)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind", ["student_t3", "lognormal_cols", "outliers"])
def test_random_tensors(mx, fmt, shape, kind):
    x = workloads.draw(kind, shape, 100 + shape[0])
    for direction in ("row", "col"):
        q, ref = run_both(mx, x, fmt, direction)
        assert_quant_equal(q, ref, f"{fmt}/{kind}/{shape}/{direction}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("direction", ["row", "col"])
@pytest.mark.parametrize("seed,stream_id", [(42, 0), (7, 3), (2**40 + 5, 9)])
def test_stochastic_rounding(mx, fmt, direction, seed, stream_id):
    x = workloads.draw("student_t3", (416, 544), 5, 1e-3)
    q, ref = run_both(mx, x, fmt, direction, rounding="sr", seed=seed, stream_id=stream_id)
    assert_quant_equal(q, ref, f"SR {fmt}/{direction}/{seed}")


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("direction", ["row", "col"])
def test_hadamard(mx, fmt, direction):
    x = workloads.draw("outliers", (416, 544), 6)
    q, ref = run_both(mx, x, fmt, direction, hadamard=True)
    assert_quant_equal(q, ref, f"H32 {fmt}/{direction}")
    if True:
        q, ref = run_both(mx, x, fmt, direction, hadamard=True, rounding="sr", seed=42)
        assert_quant_equal(q, ref, f"H32+SR {fmt}/{direction}")


@pytest.mark.parametrize("fmt", ["nvfp4", "moss"])
def test_amax_kernel_and_precomputed_amax(mx, fmt):
    x = workloads.draw("student_t3", (416, 544), 8)
    xg = x.cuda()
    a = mx.amax(xg)
    torch.cuda.synchronize()
    assert np.float32(a.item()) == np.float32(orc.amax_bf16(bits(x)))
    # a caller-supplied amax (here twice the true one) replaces the amax pass
    a2 = a * 2
    q = mx.quantize(xg, fmt, "col", amax_in=a2)
    ref = orc.quantize(bits(x), fmt, "col", amax_in=float(a2.item()))
    torch.cuda.synchronize()
    assert_quant_equal(q, ref, f"amax_in {fmt}")


def test_strided_rows(mx):
    big = workloads.draw("student_t3", (256, 640), 9)
    view = big.cuda()[:, :576]
    for fmt in FMTS:
        for direction in ("row", "col"):
            q = mx.quantize(view, fmt, direction)
            ref = orc.quantize(bits(big[:, :576]), fmt, direction)
            torch.cuda.synchronize()
            assert_quant_equal(q, ref, f"strided {fmt}/{direction}")


@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize(mx, fmt):
    x = workloads.draw("student_t3", (128, 256), 12)
    q, ref = run_both(mx, x, fmt)
    d = mx.dequantize(q).cpu().numpy().astype(np.float64)
    want = ref.dequantize() * (ref.tensor_scale if ref.tensor_scale is not None else 1.0)
    assert np.array_equal(d.astype(np.float32), want.astype(np.float32))


def test_zero_tensor_and_empty(mx):
    x = torch.zeros(128, 64, dtype=torch.bfloat16)
    for fmt in FMTS:
        q, ref = run_both(mx, x, fmt)
        assert_quant_equal(q, ref, f"zeros {fmt}")
        assert (q.codes.cpu() == 0).all()
    e = mx.quantize(torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"), "nvfp4")
    torch.cuda.synchronize()
    assert e.rows == 0 and float(e.scalars[1]) == 1.0


def test_argument_errors(mx):
    x = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.quantize(x, "moss", hadamard=True)
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
    with pytest.raises(mx.MXError) as e:  # NVFP4 blocks of 16, but the transform needs whole 32-groups
        mx.quantize(torch.zeros(64, 48, dtype=torch.bfloat16, device="cuda"), "nvfp4", hadamard=True)
    assert e.value.code == mx.MX_ERR_ALIGNMENT
    with pytest.raises(mx.MXError) as e:  # one caller amax cannot serve two differently transformed operands
        mx.quantize_dual(x, "nvfp4", col_hadamard=True, amax_in=torch.ones(1, device="cuda"))
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
    with pytest.raises(mx.MXError) as e:
        mx.quantize(torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda"), "mxfp8", "col")
    assert e.value.code in (mx.MX_ERR_ALIGNMENT, mx.MX_ERR_INVALID_ARG)
    with pytest.raises(mx.MXError) as e:
        mx.quantize(torch.zeros(64, 48, dtype=torch.bfloat16, device="cuda"), "mxfp8")
    assert e.value.code in (mx.MX_ERR_ALIGNMENT, mx.MX_ERR_INVALID_ARG)


def test_bounded_wait_gives_up_and_reports(mx):
    assert mx.last_device_status() == mx.MX_OK
    rc = mx.selftest_bounded_wait(2_000_000)  # 2 ms
    assert rc == mx.MX_ERR_TIMEOUT
    assert mx.last_device_status() == mx.MX_ERR_TIMEOUT  # read and cleared
    assert mx.last_device_status() == mx.MX_OK
    # the context is still usable afterwards
    x = workloads.draw("normal", (64, 64), 1)
    q, ref = run_both(mx, x, "mxfp8")
    assert_quant_equal(q, ref, "after timeout")


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_tile_producer_wait_gives_up_and_reports(mx, request, fmt):
    """A stage wait of the tile producer that runs out (forced by the test hook
    on one thread of every CTA, at its third tile) ends the pass with
    MX_ERR_TIMEOUT in the status word, with no fault and no hang: the CTA
    leaves together after its barrier vote, once its copies have landed.  The
    next pass is exact."""
    if request.node.callspec.params.get("mx") == "direct":
        pytest.skip("the direct producers have no stage waits")
    x = workloads.draw("normal", (4096, 4096), 5).cuda()
    assert mx.last_device_status() == mx.MX_OK
    mx.set_tile_fail_at(2)
    try:
        mx.quantize_dual(x, fmt)
        torch.cuda.synchronize()
    finally:
        mx.set_tile_fail_at(-1)
    assert mx.last_device_status() == mx.MX_ERR_TIMEOUT
    assert mx.last_device_status() == mx.MX_OK
    xs = workloads.draw("student_t3", (256, 512), 6)
    qr, qc = mx.quantize_dual(xs.cuda(), fmt)
    torch.cuda.synchronize()
    assert_quant_equal(qr, orc.quantize(bits(xs), fmt, "row"), f"{fmt} row after a forced timeout")
    assert_quant_equal(qc, orc.quantize(bits(xs), fmt, "col"), f"{fmt} col after a forced timeout")


# ------------------------------------------------------------ dual producer
DUAL_SHAPES = [(416, 544), (256, 4096), (4096, 96), (96, 288)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", DUAL_SHAPES)
def test_dual_producer_matches_two_single_passes(mx, fmt, shape):
    x = workloads.draw("outliers" if fmt == "mxfp8" else "student_t3", shape, 300 + shape[1])
    qr, qc = mx.quantize_dual(x.cuda(), fmt)
    torch.cuda.synchronize()
    assert_quant_equal(qr, orc.quantize(bits(x), fmt, "row"), f"dual row {fmt} {shape}")
    assert_quant_equal(qc, orc.quantize(bits(x), fmt, "col"), f"dual col {fmt} {shape}")


@pytest.mark.parametrize("fmt", FMTS + ["nvfp4_local"])
@pytest.mark.parametrize("shape", [(416, 544), (96, 288)])
def test_scale_padding_is_left_unwritten(mx, fmt, shape):
    """Ragged tiles (rows past R, columns and K-blocks past C) write only the
    real positions of the scale-factor layout: a sentinel in every padding
    byte survives both producers and the dual pass."""
    x = workloads.draw("student_t3", shape, 77).cuda()
    R, Cc = shape
    pairs = []
    qr, qc = mx.MXTensor(fmt, R, Cc), mx.MXTensor(fmt, Cc, R)
    for q in (qr, qc):
        q.sf.fill_(0xA5)
    mx.quantize_dual(x, fmt, row_out=qr, col_out=qc)
    pairs += [(qr, "dual row"), (qc, "dual col")]
    for d in ("row", "col"):
        q = mx.MXTensor(fmt, *((R, Cc) if d == "row" else (Cc, R)))
        q.sf.fill_(0xA5)
        mx.quantize(x, fmt, d, out=q)
        pairs.append((q, d))
    torch.cuda.synchronize()
    for q, what in pairs:
        mask = sf_valid_mask(q.rows, q.k // q.block)
        got = q.sf.cpu().numpy()
        real = np.zeros(got.size, dtype=bool)
        real[:mask.size] = mask
        assert (got[~real] == 0xA5).all(), f"{fmt} {shape} {what}: padding bytes written"
        assert (got[real] != 0xA5).any()


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8", "nvfp4"])
def test_dual_producer_direction_options(mx, fmt):
    """The weight-gradient pattern: dY rowwise with RNE for dgrad and colwise
    with SR and the Hadamard transform for wgrad, from one call (NVFP4: each
    direction with its own tensor amax)."""
    x = workloads.draw("student_t3", (512, 384), 31, 1e-3)
    sr = "sr"
    had = True
    qr, qc = mx.quantize_dual(x.cuda(), fmt, seed=42, stream_id=1, col_rounding=sr, col_hadamard=had)
    torch.cuda.synchronize()
    assert_quant_equal(qr, orc.quantize(bits(x), fmt, "row"), f"dual row {fmt}")
    ref = orc.quantize(bits(x), fmt, "col", rounding=sr, seed=42, stream_id=1, hadamard=had)
    assert_quant_equal(qc, ref, f"dual col {fmt}")
    qr2, qc2 = mx.quantize_dual(x.cuda(), fmt, row_hadamard=had, row_rounding=sr, seed=7)
    torch.cuda.synchronize()
    assert_quant_equal(qr2, orc.quantize(bits(x), fmt, "row", hadamard=had, rounding=sr, seed=7), f"dual row opts {fmt}")
    assert_quant_equal(qc2, orc.quantize(bits(x), fmt, "col"), f"dual col plain {fmt}")


def test_dual_producer_rejects_ragged_rows(mx):
    with pytest.raises(mx.MXError) as e:
        mx.quantize_dual(torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda"), "mxfp8")
    assert e.value.code in (mx.MX_ERR_ALIGNMENT, mx.MX_ERR_INVALID_ARG)


# ------------------------------------------- product-for-quotient certificate
# NVFP4 and MOSS divide by a tensor-dependent scale; the producer multiplies by
# the reciprocal only where it has certified that no bf16 input can land near a
# rounding boundary, and divides exactly elsewhere.  These cases sweep tensor
# scales across magnitudes, including power-of-two ones where every boundary
# is hit exactly and the exact division must take over.
AMAX_CASES = [None, 2688.0, 2688.0 * 2.0**-9, 2688.0 * 2.0**20, 448.0, 448.0 * 3, 448.0 * 2.0**-5,
              3.1415927, 1.0e-3, 7.0e-3, 12345.678, 1.0e30, 1.0e-30, 3.0e38, 266.0, 224.0, 0.59375]


@pytest.mark.parametrize("fmt", ["nvfp4", "moss"])
@pytest.mark.parametrize("amax", AMAX_CASES)
def test_tensor_scale_sweep(mx, fmt, amax):
    x = workloads.draw("student_t3", (256, 512), 17)
    if amax is not None:
        x = (x.float() * (amax / x.float().abs().max())).to(torch.bfloat16)
    a_in = None if amax is None else torch.tensor([amax], dtype=torch.float32, device="cuda")
    for direction in ("row", "col"):
        q = mx.quantize(x.cuda(), fmt, direction, amax_in=a_in)
        torch.cuda.synchronize()
        ref = orc.quantize(bits(x), fmt, direction, amax_in=None if amax is None else float(np.float32(amax)))
        assert_quant_equal(q, ref, f"{fmt}/{direction}/amax={amax}")


@pytest.mark.parametrize("k", [-9, 0, 7])
def test_nvfp4_ties_at_every_scale_byte(mx, k):
    """Tensor scale 2^k: for every scale byte s_b the block holds 6 dec(s_b) 2^k
    (which selects s_b) and every E2M1 midpoint times dec(s_b) 2^k, so each
    quotient is an exact tie that a product with the rounded reciprocal could
    push the wrong way."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    dec = np.array([orc.decode("e4m3", c) for c in range(128)])
    rows = []
    rng = np.random.default_rng(k + 100)
    for sb in range(1, 127):
        d = dec[sb] * 2.0**k
        blk = np.array([6 * d] + [m * d for m in mids] + [-m * d for m in mids] + [0.0])
        rows.append(np.concatenate([rng.permutation(blk) for _ in range(16)]))
    rows += rows[:2]
    x = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(x.double().numpy(), np.array(rows))  # every value is exact in bf16
    a_in = torch.tensor([2688.0 * 2.0**k], dtype=torch.float32, device="cuda")
    for xx, direction in ((x, "row"), (x.t().contiguous(), "col")):
        q = mx.quantize(xx.cuda(), "nvfp4", direction, amax_in=a_in)
        torch.cuda.synchronize()
        ref = orc.quantize(bits(xx), "nvfp4", direction, amax_in=2688.0 * 2.0**k)
        assert_quant_equal(q, ref, f"ties k={k} {direction}")


# ----------------------------------------------------- CTA-local NVFP4 (f2)
LOCAL_SHAPES = [(416, 544), (256, 4096), (4096, 96), (96, 288), (320, 128)]


@pytest.mark.parametrize("shape", LOCAL_SHAPES)
@pytest.mark.parametrize("kind", ["student_t3", "lognormal_cols"])
def test_nvfp4_local_row_col_dual(mx, shape, kind):
    """One FP32 scale per 128 operand rows (ragged last region): codes, scale
    bytes and the amax / tensor-scale arrays equal the oracle's, rowwise,
    colwise and from the dual pass (row regions and column regions of x)."""
    x = workloads.draw(kind, shape, 500 + shape[0])
    for direction in ("row", "col"):
        q, ref = run_both(mx, x, "nvfp4_local", direction)
        assert_quant_equal(q, ref, f"local/{direction}/{shape}")
    qr, qc = mx.quantize_dual(x.cuda(), "nvfp4_local")
    torch.cuda.synchronize()
    assert_quant_equal(qr, orc.quantize(bits(x), "nvfp4_local", "row"), f"local dual row {shape}")
    assert_quant_equal(qc, orc.quantize(bits(x), "nvfp4_local", "col"), f"local dual col {shape}")


@pytest.mark.parametrize("direction", ["row", "col"])
def test_nvfp4_local_sr_and_amax_in(mx, direction):
    x = workloads.draw("student_t3", (384, 512), 33, 1e-3)
    q, ref = run_both(mx, x, "nvfp4_local", direction, rounding="sr", seed=5, stream_id=1)
    assert_quant_equal(q, ref, f"local SR {direction}")
    n = -(-(384 if direction == "row" else 512) // 128)
    ain = torch.linspace(1e-3, 4e-3, n, dtype=torch.float32)
    q = mx.quantize(x.cuda(), "nvfp4_local", direction, amax_in=ain.cuda())
    torch.cuda.synchronize()
    ref = orc.quantize(bits(x), "nvfp4_local", direction, amax_in=ain.numpy())
    assert_quant_equal(q, ref, f"local amax_in {direction}")
    with pytest.raises(mx.MXError) as e:  # the dual pass computes its own region maxima
        mx.quantize_dual(x.cuda(), "nvfp4_local", amax_in=ain.cuda())
    assert e.value.code == mx.MX_ERR_UNSUPPORTED


@pytest.mark.parametrize("direction", ["row", "col"])
def test_nvfp4_hadamard_amax_is_of_the_transformed_operand(mx, direction):
    """NVFP4 with the transform: the tensor amax is max |H32 x| over the operand
    (not max |x|), and a caller amax is taken as given."""
    x = workloads.draw("student_t3", (512, 640), 41)
    q, ref = run_both(mx, x, "nvfp4", direction, hadamard=True)
    assert_quant_equal(q, ref, f"nvfp4 H32 {direction}")
    assert ref.amax > float(x.float().abs().max())
    big = torch.tensor([ref.amax * 3], dtype=torch.float32, device="cuda")
    q2 = mx.quantize(x.cuda(), "nvfp4", direction, hadamard=True, amax_in=big)
    assert_quant_equal(q2, orc.quantize(bits(x), "nvfp4", direction, hadamard=True, amax_in=ref.amax * 3),
                       f"nvfp4 H32 caller amax {direction}")
