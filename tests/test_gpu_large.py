"""Index arithmetic past 2^31 elements: a producer pass over a 65600 x 32768
bf16 tensor (2.15e9 elements, a ragged last row tile) and a GEMM whose A
operand holds 2.15e9 codes.  The parts of the results that lie past 2^31
elements must equal what the same calls give on a slice holding just those
rows (blocks are independent, and the tensor scale is passed in), so any
32-bit offset that wraps shows up as a mismatch."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


def _randn_bf16(rows, cols, seed):
    """Seeded N(0, 1) bf16 on the GPU, drawn in row chunks (no 2x fp32 copy)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    for r in range(0, rows, 4096):
        n = min(4096, rows - r)
        x[r:r + n] = torch.randn(n, cols, generator=g, device="cuda").to(torch.bfloat16)
    return x


def _sf_logical(q, rows, kbs):
    """Scale bytes of operand rows `rows` and K-blocks `kbs` (logical order),
    gathered from the swizzled layout: 512-byte tiles of 128 rows x 4 K-blocks."""
    kblocks = q.k // q.block
    kg = (kblocks + 3) // 4
    r = torch.as_tensor(rows, device="cuda", dtype=torch.int64)[:, None]
    kb = torch.as_tensor(kbs, device="cuda", dtype=torch.int64)[None, :]
    idx = ((r >> 7) * kg + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3)
    return q.sf[idx]


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_dual_producer_past_2g_elements(mx, fmt):
    R, C, tail = 65600, 32768, 64
    x = _randn_bf16(R, C, 11)
    am = mx.amax(x) if fmt == "nvfp4" else None
    qr, qc = mx.quantize_dual(x, fmt, amax_in=am)
    sr, sc = mx.quantize_dual(x[R - tail:].contiguous(), fmt, amax_in=am)
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MX_OK
    fp4 = fmt == "nvfp4"
    # rowwise operand: the last rows
    assert torch.equal(qr.codes[R - tail:], sr.codes)
    kb_row = range(C // qr.block)
    assert torch.equal(_sf_logical(qr, range(R - tail, R), kb_row), _sf_logical(sr, range(tail), kb_row))
    # colwise operand: the last K positions of every row (input column)
    k0 = (R - tail) // 2 if fp4 else R - tail
    assert torch.equal(qc.codes[:, k0:], sc.codes)
    nb = tail // qc.block
    cols = range(0, C, 97)  # a spread of operand rows (input columns)
    assert torch.equal(_sf_logical(qc, cols, range((R - tail) // qc.block, (R - tail) // qc.block + nb)),
                       _sf_logical(sc, cols, range(nb)))
    if am is not None:
        assert torch.equal(qr.scalars, sr.scalars) and torch.equal(qc.scalars, sc.scalars)


def test_gemm_past_2g_operand(mx):
    M, N, K, tail = 65536, 256, 32768, 256
    a = _randn_bf16(M, K, 12)
    b = _randn_bf16(N, K, 13)
    qa, qb = mx.quantize(a, "mxfp8"), mx.quantize(b, "mxfp8")
    qs = mx.quantize(a[M - tail:].contiguous(), "mxfp8")
    mx.set_gemm_variant("pair_ws")
    try:
        c = mx.gemm(qa, qb)
        cs = mx.gemm(qs, qb)
        torch.cuda.synchronize()
    finally:
        mx.set_gemm_variant("auto")
    assert mx.last_device_status() == mx.MX_OK
    assert torch.isfinite(c).all()
    assert torch.equal(c[M - tail:], cs)  # the same tiles, the same K order
