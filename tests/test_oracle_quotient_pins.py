"""Pins for the quotients by the tensor scale: NVFP4's block-scale byte and
element divisor, and MOSS's level-1 division.

The pages fix these steps only in words: MOSS ("MOSS: 用微缩放和自动缩放实现无损
FP8 训练", section 两级缩放实现) divides the tensor by its FP32 tensor scale
amax / 448 before the power-of-two micro scale; NVFP4 ("格式感知融合:让FP4预训练
提速两倍的工程实践", section FP4加速为何常常"纸上富贵") scales each 16-element
block by an E4M3 block scale under a global FP32 scale.  The reading taken:

  NVFP4  s_t = fl32(amax / 2688); s_b = UE4M3_RNE(fl32(b / fl32(6 * s_t)));
         d = fl32(dec(s_b) * s_t); code = E2M1_RNE(fl32(x / d)) (sign-kept 0
         when d == 0).
  MOSS   s_t = fl32(amax / 448); y = fl32(x / s_t); e = CEIL(max |y| of the
         32-block); code = E4M3_RNE(fl32(y * 2^-e)).

Each reading is restated here in numpy float32 arithmetic (IEEE
round-to-nearest-even per operation), with the UE4M3 / E4M3 rounding taken
from torch's float8_e4m3fn cast and the E2M1 rounding by brute force over the
grid {0, .5, 1, 1.5, 2, 3, 4, 6}.  None of it calls the oracle's arithmetic.
The oracle must match byte for byte, on random tensors and on stress tensors
built by search so that each plausible alternative (a ceiling scale byte,
6 * s_t formed in double precision, dividing twice, a reciprocal product)
changes at least one byte; the test asserts that it does, so a mistake of that
kind in the oracle cannot pass.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
F32 = np.float32


def bf16_values(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_bf16_bits(v):
    """float32 values that are exact bf16 values -> their bit patterns."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert ((u & 0xFFFF) == 0).all()
    return (u >> 16).astype(np.uint16)


POS_BF16 = bf16_values(np.arange(1, 0x7F80, dtype=np.uint32))  # every positive finite bf16


def e4m3_rne_bytes(v):
    """RNE to E4M3 (saturating at 448, sign kept) through torch's float8 cast."""
    v = np.asarray(v, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(np.clip(v, -448.0, 448.0).reshape(-1)))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(v.shape)


def e4m3_ceil_bytes(v):
    """The smallest non-negative E4M3 value >= v (a wrong reading of the scale byte)."""
    grid = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    return np.searchsorted(grid, np.minimum(np.asarray(v, dtype=np.float64), 448.0), side="left").astype(np.uint8)


def e4m3_decode(b):
    b = np.asarray(b, dtype=np.uint8)
    t = torch.from_numpy(np.ascontiguousarray(b.reshape(-1)))
    return t.view(torch.float8_e4m3fn).float().numpy().reshape(b.shape)


def e2m1_rne_codes(v):
    """Nearest E2M1 grid point to |v| (ties to the even code, saturating at 6), sign kept."""
    v = np.asarray(v, dtype=np.float32)
    a = np.minimum(np.abs(v.astype(np.float64)), 6.0)
    d = np.abs(a[..., None] - E2M1_GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # two candidates only on an exact tie: take the even code
    idx = np.where(cand.sum(-1) > 1, np.argmax(cand & (np.arange(8) % 2 == 0), axis=-1), np.argmax(cand, axis=-1))
    return (idx | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


# --------------------------------------------------------------- NVFP4 ---
def nvfp4_reference(x, amax=None, variant="page"):
    """NVFP4 codes [rows, K] (one code per element, unpacked) and scale bytes
    [rows, K/16] of a row-major float32 matrix of bf16 values, in numpy float32.

    variant "page" is the reading above; the others are the alternatives the
    pins must tell apart from it."""
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    if amax is None:
        amax = np.abs(x).max()
    amax = F32(amax)
    st = F32(amax / F32(2688.0)) if amax != 0 else F32(1.0)
    blk = x.reshape(rows, K // 16, 16)
    b = np.abs(blk).max(axis=-1)
    if variant == "denom_f64":
        q = (b.astype(np.float64) / (6.0 * np.float64(st))).astype(np.float32)
    else:
        q = b / F32(F32(6.0) * st)
    sb = e4m3_ceil_bytes(q) if variant == "ceil_scale" else e4m3_rne_bytes(q)
    d = F32(1.0) * e4m3_decode(sb).astype(np.float32) * st  # float32 product
    dd = d[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        if variant == "divide_twice":
            v = (blk / st) / e4m3_decode(sb).astype(np.float32)[..., None]
        elif variant == "reciprocal":
            v = blk * (F32(1.0) / dd)
        else:
            v = blk / dd
    v = np.where(dd == 0, np.where(np.signbit(blk), F32(-0.0), F32(0.0)), v).astype(np.float32)
    codes = e2m1_rne_codes(v)
    return codes.reshape(rows, K), sb


def unpack_fp4(codes_packed):
    lo = codes_packed & 0xF
    hi = codes_packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes_packed.shape[0], -1)


def oracle_nvfp4(x_bits, fmt="nvfp4", amax_in=None):
    q = orc.quantize(x_bits, fmt, "row", amax_in=amax_in)
    return unpack_fp4(q.codes), q.sf_logical, q


E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def bf16_neighbours(v):
    """The bf16 values just below and just above each positive float64 v."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32) >> 16
    lo = bf16_values(u)
    hi = bf16_values(u + 1)
    return np.concatenate([lo, hi])


def nvfp4_stress_tensors():
    """Tensors (one per tensor amax) whose 16-element blocks are built by search
    so that the alternatives to the page reading give other bytes.

    The tensor amax runs over the 128 bf16 values of one binade (the tensor
    scale's significand depends on nothing else).  For each:
      - block maxima b whose UE4M3 byte changes when 6 * s_t is formed in double
        precision instead of fl32;
      - for every scale byte, the bf16 values next to d * m for each E2M1
        decision boundary m (d = fl32(dec(s_b) * s_t)), kept where dividing by
        s_t and then by dec(s_b), or multiplying by fl32(1 / d), gives another
        E2M1 code than fl32(x / d)."""
    out = []
    for amax in bf16_values(np.arange(0x40C0, 0x4100, dtype=np.uint32)):  # [6, 8)
        st = F32(amax / F32(2688.0))
        D = F32(F32(6.0) * st)
        cand = POS_BF16[POS_BF16 <= amax]
        sb_all = e4m3_rne_bytes(cand / D)
        blocks = []
        q_f64 = (cand.astype(np.float64) / (6.0 * np.float64(st))).astype(np.float32)
        for b in cand[np.flatnonzero(sb_all != e4m3_rne_bytes(q_f64))][:16]:
            blk = np.full(16, b * F32(0.5), dtype=np.float32)
            blk[0] = b
            blocks.append(blk)
        for sb in np.unique(sb_all):
            bmax = cand[sb_all == sb].max()
            dec = e4m3_decode(sb).astype(np.float32)
            d = F32(dec * st)
            if d == 0:
                continue
            xs = bf16_neighbours(E2M1_MIDPOINTS * np.float64(d))
            xs = xs[(xs > 0) & (xs <= bmax)]
            page = e2m1_rne_codes(xs / d)
            twice = e2m1_rne_codes((xs / st) / dec)
            recip = e2m1_rne_codes(xs * (F32(1.0) / d))
            hit = xs[(page != twice) | (page != recip)]
            for i in range(0, len(hit), 15):
                blk = np.zeros(16, dtype=np.float32)
                blk[0] = bmax
                blk[1:1 + len(hit[i:i + 15])] = hit[i:i + 15]
                blocks.append(blk)
        if not blocks:
            continue
        head = np.zeros(16, dtype=np.float32)
        head[0] = amax  # the tensor amax, in a block of its own
        blocks.insert(0, head)
        while len(blocks) % 4:
            blocks.append(np.zeros(16, dtype=np.float32))
        signs = np.where(np.arange(len(blocks) * 16) % 3 == 2, -1.0, 1.0).astype(np.float32)
        signs[::16] = 1.0  # keep every block maximum positive (the sign plays no part in it)
        body = (np.stack(blocks).reshape(-1) * signs).reshape(-1, 64)
        out.append(body)
    assert out, "no amax found where the quotient's form matters"
    return out


def ties_tensor():
    """amax = 2688 * 2^-4 gives s_t = 2^-4 exactly; every block maximum b =
    6 * s_t * m for an E4M3 midpoint m (a UE4M3 tie) or a grid value, and the
    other elements sit on E2M1 midpoints d * {0.25, 0.75, ..., 5} (E2M1 ties)."""
    st = 2.0 ** -4
    amax = 2688.0 * st  # 168, a bf16 value
    grid = e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    rows = []
    for m in np.concatenate([grid, mids]):
        b = 6.0 * st * m
        if b > amax or b != float(np.float32(b)) or float(to_bf16_bits_safe(b)) != b:
            continue
        sb = e4m3_rne_bytes(np.float32(b / (6.0 * st)))
        d = float(e4m3_decode(sb)) * st
        blk = [b] + [d * t for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.5, 3.0)]
        blk = [v if float(to_bf16_bits_safe(v)) == v else 0.0 for v in blk]
        blk += [0.0] * (16 - len(blk))
        rows.append(blk)
    while len(rows) % 4:
        rows.append([0.0] * 16)
    body = np.array(rows, dtype=np.float32).reshape(-1, 64)
    body[0, 15] = amax
    return body


def to_bf16_bits_safe(v):
    """The bf16 value nearest to v when v is exactly representable, else NaN."""
    f = np.float32(v)
    u = np.array([f]).view(np.uint32)[0]
    return float(f) if (u & 0xFFFF) == 0 and float(f) == v else float("nan")


@pytest.mark.parametrize("kind", ["student_t3", "normal", "outliers"])
def test_nvfp4_oracle_matches_page_reading_on_random_tensors(kind):
    x = workloads.draw(kind, (64, 256), 31, 0.02 if kind == "normal" else 1.0)
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    codes, sf, _ = oracle_nvfp4(xb)
    rc, rs = nvfp4_reference(bf16_values(xb))
    assert np.array_equal(sf, rs)
    assert np.array_equal(codes, rc)
    # a ceiling scale byte changes the bytes of ordinary random data
    _, cs = nvfp4_reference(bf16_values(xb), variant="ceil_scale")
    assert not np.array_equal(cs, sf)


def test_nvfp4_oracle_matches_page_reading_on_stress_tensors():
    tensors = nvfp4_stress_tensors()
    separated = set()
    for xf in tensors:
        xb = to_bf16_bits(xf)
        codes, sf, q = oracle_nvfp4(xb)
        assert np.float32(q.tensor_scale) == F32(F32(np.abs(xf).max()) / F32(2688.0))
        rc, rs = nvfp4_reference(xf)
        assert np.array_equal(sf, rs)
        assert np.array_equal(codes, rc)
        for variant in ("denom_f64", "divide_twice", "reciprocal", "ceil_scale"):
            ac, as_ = nvfp4_reference(xf, variant=variant)
            if not (np.array_equal(as_, sf) and np.array_equal(ac, codes)):
                separated.add(variant)
    # each alternative reading gives other bytes on some stress tensor
    assert separated == {"denom_f64", "divide_twice", "reciprocal", "ceil_scale"}, separated


def test_nvfp4_oracle_matches_page_reading_on_exact_ties():
    xf = ties_tensor()
    xb = to_bf16_bits(xf)
    codes, sf, q = oracle_nvfp4(xb)
    assert q.tensor_scale == 2.0 ** -4
    rc, rs = nvfp4_reference(xf)
    assert np.array_equal(sf, rs)
    assert np.array_equal(codes, rc)


def test_nvfp4_local_matches_page_reading_per_region():
    """CTA-local NVFP4: every 128-row region is the page reading with that
    region's own amax."""
    x = workloads.draw("student_t3", (300, 128), 33)
    x[130:140] *= 40  # regions with very different maxima
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    xf = bf16_values(xb)
    codes, sf, q = oracle_nvfp4(xb, "nvfp4_local")
    for g, r0 in enumerate(range(0, 300, 128)):
        r1 = min(r0 + 128, 300)
        amax = np.abs(xf[r0:r1]).max()
        assert q.amax[g] == amax and q.tensor_scale[g] == F32(F32(amax) / F32(2688.0))
        rc, rs = nvfp4_reference(xf[r0:r1], amax=amax)
        assert np.array_equal(sf[r0:r1], rs)
        assert np.array_equal(codes[r0:r1], rc)


def test_nvfp4_caller_amax_is_used_as_given():
    x = workloads.draw("student_t3", (32, 128), 34)
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    xf = bf16_values(xb)
    amax = F32(np.abs(xf).max() * 3.0)  # a larger, caller-chosen amax
    codes, sf, _ = oracle_nvfp4(xb, amax_in=amax)
    rc, rs = nvfp4_reference(xf, amax=amax)
    assert np.array_equal(sf, rs) and np.array_equal(codes, rc)


# ---------------------------------------------------------------- MOSS ---
def moss_reference(x, variant="page"):
    """MOSS codes [rows, K] and E8M0 bytes [rows, K/32] in numpy float32."""
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    amax = F32(np.abs(x).max())
    st = F32(amax / F32(448.0)) if amax != 0 else F32(1.0)
    if variant == "reciprocal":
        y = x * (F32(1.0) / st)
    elif variant == "inverse_scale":
        y = x * (F32(448.0) / amax)
    else:
        y = x / st
    y = y.astype(np.float32)
    blk = y.reshape(rows, K // 32, 32)
    b = np.abs(blk).max(axis=-1).astype(np.float64)
    # CEIL rule: the smallest e with b * 2^-e <= 448 (b = 0: e = 0)
    e = np.zeros(b.shape, dtype=np.int64)
    nz = b > 0
    e[nz] = np.ceil(np.log2(b[nz] / 448.0)).astype(np.int64)
    for _ in range(3):  # exact fix-up of the floating log2
        up = nz & (np.ldexp(b, -e) > 448.0)
        e[up] += 1
        down = nz & (np.ldexp(b, -(e - 1)) <= 448.0)
        e[down] -= 1
    e = np.clip(e, -127, 127)
    scaled = np.ldexp(blk, -e[..., None]).astype(np.float32)
    return e4m3_rne_bytes(scaled).reshape(rows, K), (e + 127).astype(np.uint8)


def moss_stress_tensors():
    """Tensors (one per tensor amax) of 32-element blocks whose maximum is the
    tensor amax itself, so the micro scale is the CEIL exponent e of
    fl32(amax / s_t) (within an ulp of 448: e = 0 or 1), filled with the bf16
    values next to s_t * m * 2^e for every E4M3 decision boundary m, kept where
    a reciprocal product gives another code than fl32(x / s_t)."""
    grid = e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    out = []
    for amax in bf16_values(np.arange(0x40C0, 0x4100, dtype=np.uint32)):  # [6, 8)
        st = F32(amax / F32(448.0))
        e = 0 if F32(amax / st) <= F32(448.0) else 1
        xs = bf16_neighbours(mids * np.ldexp(np.float64(st), e))
        xs = xs[(xs > 0) & (xs < amax)]
        page = e4m3_rne_bytes(np.ldexp(xs / st, -e))
        hit = np.zeros(len(xs), dtype=bool)
        for alt in (xs * (F32(1.0) / st), xs * (F32(448.0) / amax)):
            hit |= page != e4m3_rne_bytes(np.ldexp(alt.astype(np.float32), -e))
        vals = xs[hit]
        if not len(vals):
            continue
        rows = []
        for i in range(0, len(vals), 31):
            blk = np.zeros(32, dtype=np.float32)
            blk[0] = amax
            chunk = vals[i:i + 31]
            blk[1:1 + len(chunk)] = chunk
            rows.append(blk)
        while len(rows) % 4:
            rows.append(np.zeros(32, dtype=np.float32))
        out.append(np.stack(rows).reshape(-1, 128))
    assert out, "no amax found where the division form matters"
    return out


@pytest.mark.parametrize("kind", ["lognormal_cols", "student_t3"])
def test_moss_oracle_matches_page_reading_on_random_tensors(kind):
    x = workloads.draw(kind, (64, 256), 41)
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    q = orc.quantize(xb, "moss", "row")
    rc, rs = moss_reference(bf16_values(xb))
    assert np.array_equal(q.sf_logical, rs)
    assert np.array_equal(q.codes, rc)


def test_moss_oracle_matches_page_reading_on_stress_tensors():
    separated = set()
    for xf in moss_stress_tensors():
        xb = to_bf16_bits(xf)
        q = orc.quantize(xb, "moss", "row")
        assert np.float32(q.tensor_scale) == F32(F32(np.abs(xf).max()) / F32(448.0))
        rc, rs = moss_reference(xf)
        assert np.array_equal(q.sf_logical, rs)
        assert np.array_equal(q.codes, rc)
        for variant in ("reciprocal", "inverse_scale"):
            ac, as_ = moss_reference(xf, variant=variant)
            if not (np.array_equal(ac, q.codes) and np.array_equal(as_, q.sf_logical)):
                separated.add(variant)
    # each alternative reading gives other bytes on some stress tensor
    assert separated == {"reciprocal", "inverse_scale"}, separated


# ------------------------------------------------- NVFP4 with Hadamard-32 ---
def _exact_transform_input(shape, seed):
    """bf16 values k / 16, |k| <= 8: every butterfly of the 32-point transform
    is exact in fp32, so the transformed block equals H32 x computed in fp64."""
    rng = np.random.default_rng(seed)
    return (rng.integers(-8, 9, size=shape) / 16.0).astype(np.float32)


@pytest.mark.parametrize("direction", ["row", "col"])
def test_nvfp4_hadamard_is_the_page_reading_on_transformed_blocks(direction):
    """NVFP4 with the transform: y = H32 x per 32 operand elements along K
    (scipy's Sylvester matrix, fp64), the tensor amax over all y, then the
    NVFP4 reading on y.  The oracle must give the same bytes, and its amax must
    be the transformed one (larger than max |x| here)."""
    from scipy.linalg import hadamard
    H = hadamard(32).astype(np.float64)
    x = _exact_transform_input((64, 128), 51)
    xb = to_bf16_bits(x)
    q = orc.quantize(xb, "nvfp4", direction, hadamard=True)
    op = x if direction == "row" else x.T  # operand rows along K
    y = (op.reshape(op.shape[0], -1, 32).astype(np.float64) @ H.T).reshape(op.shape).astype(np.float32)
    assert np.float32(q.amax) == np.abs(y).max() > np.abs(x).max()
    rc, rs = nvfp4_reference(y)
    assert np.array_equal(q.sf_logical, rs)
    assert np.array_equal(unpack_fp4(q.codes), rc)
    # a caller amax is taken as the transformed tensor's amax, as given
    q2 = orc.quantize(xb, "nvfp4", direction, hadamard=True, amax_in=float(np.abs(y).max()) * 2)
    rc2, rs2 = nvfp4_reference(y, amax=np.abs(y).max() * 2)
    assert np.array_equal(q2.sf_logical, rs2) and np.array_equal(unpack_fp4(q2.codes), rc2)


def test_nvfp4_hadamard_wgrad_identity():
    """(H a)^T (H b) = 32 a^T b: the weight gradient from transformed NVFP4
    operands, scaled by 1/32, estimates dY^T X (quantization error only)."""
    dy = workloads.draw("student_t3", (256, 128), 52, 1e-3)
    xx = workloads.draw("normal", (256, 96), 53)
    ra = orc.quantize(dy.contiguous().view(torch.int16).numpy().view(np.uint16), "nvfp4", "col", hadamard=True)
    rb = orc.quantize(xx.contiguous().view(torch.int16).numpy().view(np.uint16), "nvfp4", "col", hadamard=True)
    c, _ = orc.gemm(ra, rb, extra_alpha=1.0 / 32)
    exact = dy.double().t().numpy() @ xx.double().numpy()
    rel = np.linalg.norm(c - exact) / np.linalg.norm(exact)
    assert rel < 0.25
