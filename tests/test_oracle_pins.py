"""Pins that tie the CPU oracle to the pages and to mathematics, not to itself.

Each test checks an oracle function against something independent of its own
code: values printed on the pages (tests/golden), a library routine (torch's
float8 cast, scipy's Hadamard matrix, numpy's fp64 matmul and float32
arithmetic), closed forms, invariants, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def minifloat_values(ebits, mbits, nan_all_ones=False):
    """Generic sign/exponent/mantissa decoder with IEEE-style bias, subnormals and
    no infinities; written independently of the oracle's per-format decoders."""
    bias = 2 ** (ebits - 1) - 1
    vals = {}
    for code in range(2 ** (1 + ebits + mbits)):
        s = code >> (ebits + mbits)
        e = (code >> mbits) & ((1 << ebits) - 1)
        m = code & ((1 << mbits) - 1)
        if nan_all_ones and e == (1 << ebits) - 1 and m == (1 << mbits) - 1:
            vals[code] = float("nan")
            continue
        if e == 0:
            mag = m * 2.0 ** (1 - bias - mbits)
        else:
            mag = (1 + m / 2.0 ** mbits) * 2.0 ** (e - bias)
        vals[code] = -mag if s else mag
    return vals


# ------------------------------------------------------------------ formats ---
def test_e4m3_grid_matches_generic_minifloat_and_page_range():
    g = gold("e4m3_range.json")
    ref = minifloat_values(4, 3, nan_all_ones=True)
    for code in range(256):
        v = orc.decode("e4m3", code)
        if math.isnan(ref[code]):
            assert math.isnan(v), code
        else:
            assert v == ref[code], code
    finite = [abs(orc.decode("e4m3", c)) for c in range(256) if not math.isnan(orc.decode("e4m3", c))]
    assert max(finite) == g["max"]
    mn = min(v for v in finite if v > 0)
    assert round(mn, 5) == g["min_printed"] and mn == 2.0 ** -9
    ratio = max(finite) / mn
    assert ratio == 229376 and abs(ratio - g["range_printed"]) / g["range_printed"] < 0.2
    assert orc.decode("e4m3", 0x7E) == 448.0 and math.isnan(orc.decode("e4m3", 0x7F))
    assert math.isnan(orc.decode("e4m3", 0xFF))


def test_e2m1_grid_from_page_bit_layout():
    lay = gold("fp4_layouts.json")["E2M1"]
    ref = minifloat_values(lay["exponent"], lay["mantissa"])
    got = {c: orc.decode("e2m1", c) for c in range(16)}
    assert got == ref
    assert sorted({abs(v) for v in got.values()}) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e8m0_is_power_of_two():
    for b in range(255):
        assert orc.decode("e8m0", b) == math.ldexp(1.0, b - 127)
    assert math.isnan(orc.decode("e8m0", 255))


def test_power_of_two_dequant_is_exact_shift():
    g = gold("pow2_shift.json")
    # the page's example: value 50, k = 3
    assert g["value"] * 2 ** g["k"] == g["result"]
    assert math.ldexp(g["value"], g["k"]) == g["result"]
    for elem in ("e4m3", "e2m1"):
        for code in range(256 if elem == "e4m3" else 16):
            v = orc.decode(elem, code)
            if math.isnan(v):
                continue
            for k in range(-20, 21):
                s = orc.decode("e8m0", 127 + k)
                assert np.float32(v) * np.float32(s) == math.ldexp(v, k)


# ------------------------------------------------------------- RNE casting ---
def test_e4m3_rne_matches_torch_float8_on_every_bf16():
    x = workloads.all_bf16_patterns().float()
    ref = x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.encode_rne("e4m3", float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("elem,nmax", [("e4m3", 0x7E), ("e2m1", 7)])
def test_rne_midpoints_ties_even_and_saturation(elem, nmax):
    grid = [orc.decode(elem, c) for c in range(nmax + 1)]
    for c in range(nmax):
        lo, hi = grid[c], grid[c + 1]
        mid = (lo + hi) / 2
        below = np.nextafter(np.float32(mid), np.float32(-1))
        above = np.nextafter(np.float32(mid), np.float32(1e9))
        assert orc.encode_rne(elem, below) == c
        assert orc.encode_rne(elem, above) == c + 1
        assert orc.encode_rne(elem, mid) == (c if c % 2 == 0 else c + 1)
        neg = orc.encode_rne(elem, -float(above))
        assert neg == (c + 1) | (0x80 if elem == "e4m3" else 0x8)
    top = grid[nmax]
    for v in (top, top * 1.01, top * 2, 3.0e38):
        assert orc.encode_rne(elem, v) == nmax
    sign = 0x80 if elem == "e4m3" else 0x8
    assert orc.encode_rne(elem, -0.0) == sign
    assert orc.encode_rne(elem, -1e-30) == sign
    assert orc.encode_rne(elem, 0.0) == 0


def test_e2m1_rne_brute_force_random_values():
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), rng.normal(0, 1, 4000)]).astype(np.float32)
    grid = np.array([orc.decode("e2m1", c) for c in range(8)])
    for v in vals:
        a = min(abs(float(v)), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        assert orc.encode_rne("e2m1", v) == (c | (0x8 if np.signbit(v) else 0))


# ------------------------------------------------------------ scale rules ---
def _bs():
    rng = np.random.default_rng(5)
    b = np.concatenate([np.exp2(rng.uniform(-140, 127, 3000)), [448, 6, 449, 447.9, 2 ** -133,
                                                               3.38e38, 1.0, 5.99, 6.01]])
    return b.astype(np.float32)


@pytest.mark.parametrize("elem,Q,emax", [("e4m3", 448.0, 8), ("e2m1", 6.0, 2)])
def test_scale_rules_properties(elem, Q, emax):
    for b in _bs():
        b = float(b)
        e = orc.pow2_exponent(b, "floor", elem)
        if -127 <= math.floor(math.log2(b)) - emax <= 127:
            s = math.ldexp(b, -e)
            assert 2.0 ** emax <= s < 2.0 ** (emax + 1), (b, e)
        e = orc.pow2_exponent(b, "ceil", elem)
        if -127 < e < 127:
            assert math.ldexp(b, -e) <= Q < math.ldexp(b, -(e - 1)), (b, e)
        e = orc.pow2_exponent(b, "nearest", elem)
        if -127 < e < 127:
            assert abs(math.log2(b / Q) - e) <= 0.5 + 1e-12, (b, e)
    for rule in ("floor", "ceil", "nearest"):
        assert orc.pow2_exponent(0.0, rule, elem) == 0
        assert orc.pow2_exponent(2.0 ** -140, rule, elem) == -127


# -------------------------------------------------------------- Philox/SR ---
def test_philox_statistics_and_counter_sensitivity():
    key = np.array([42, 0], dtype=np.uint32)
    outs = np.array([orc.philox4x32_10([i, 0, 0, 0], key) for i in range(4096)], dtype=np.uint32)
    # bit balance of 4096*4 words: each of 32 bits is set ~half the time
    bits = ((outs.reshape(-1, 1) >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 0.02)
    # 16-bit halves are uniform (chi-square over 64 bins)
    u16 = np.concatenate([outs.reshape(-1) & 0xFFFF, outs.reshape(-1) >> 16])
    h = np.bincount(u16 >> 10, minlength=64)
    exp = len(u16) / 64
    chi2 = ((h - exp) ** 2 / exp).sum()
    assert chi2 < 130  # 63 dof: p ~ 1e-6
    # every counter word and key word changes the output (avalanche)
    base = orc.philox4x32_10([7, 8, 9, 10], [1, 2])
    for i in range(4):
        c = [7, 8, 9, 10]
        c[i] ^= 1
        flips = np.unpackbits((orc.philox4x32_10(c, [1, 2]) ^ base).view(np.uint8)).sum()
        assert 30 < flips < 98
    for i in range(2):
        k = [1, 2]
        k[i] ^= 1
        flips = np.unpackbits((orc.philox4x32_10([7, 8, 9, 10], k) ^ base).view(np.uint8)).sum()
        assert 30 < flips < 98


def _curand_host():
    """cuRAND's host-side (CPU) generator library, if the toolkit ships it."""
    import ctypes

    for name in ("libcurand.so", "libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """The oracle's Philox4x32-10 against a library implementation of the same
    published generator: cuRAND's host Philox4_32_10 generator, which runs on the
    CPU.  With a 64-bit seed s it emits output block j (four words) as
    Philox4x32-10 with key (s mod 2^32, s div 2^32) and counter
    (j div 65536, 0, j mod 65536, 0).  That covers both key words and counter
    words 0 and 2, the words the stochastic-rounding counter uses."""
    import ctypes

    L = _curand_host()
    if L is None:
        pytest.skip("cuRAND is not installed")
    gen = ctypes.c_void_p()
    if L.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:  # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        n_blocks = 65536 + 1024
        for seed in (0x0123456789ABCDEF, 42, 2 ** 64 - 1):
            assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert L.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0  # restart the stream
            out = np.zeros(4 * n_blocks, dtype=np.uint32)
            assert L.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(out.size)) == 0
            blocks = out.reshape(-1, 4)
            key = [seed & 0xFFFFFFFF, seed >> 32]
            rng = np.random.default_rng(seed & 0xFFFF)
            picks = list(range(64)) + list(range(65536, 65536 + 64)) + list(rng.integers(0, n_blocks, 64))
            for j in picks:
                j = int(j)
                want = orc.philox4x32_10([j // 65536, 0, j % 65536, 0], key)
                assert np.array_equal(blocks[j], want), (seed, j)
    finally:
        L.curandDestroyGenerator(gen)


def test_sr_unbiased_and_probability():
    grid = [orc.decode("e2m1", c) for c in range(8)]
    rng = np.random.default_rng(11)
    for v in [0.2, 0.74, 1.1, 1.9, 2.25, 3.5, 4.001, 5.9, -2.6, -0.01]:
        n = 4000
        us = rng.integers(0, 65536, n)
        codes = np.array([orc.encode_e2m1_sr(v, int(u)) for u in us])
        dec = np.array([orc.decode("e2m1", int(c)) for c in codes])
        a = abs(v)
        lo = max(g for g in grid if g <= a)
        hi = min(g for g in grid if g > a)
        p = (a - lo) / (hi - lo)
        assert set(np.abs(dec)) <= {lo, hi}
        frac_up = np.mean(np.abs(dec) == hi)
        assert abs(frac_up - p) < 4 * math.sqrt(p * (1 - p) / n) + 1e-3
        sd = (hi - lo) * math.sqrt(p * (1 - p) / n)
        assert abs(dec.mean() - v) < 4 * sd + 1e-4
    # deterministic edges: u16 = 0 always rounds an off-grid value up,
    # grid points and saturated values never move
    assert orc.decode("e2m1", orc.encode_e2m1_sr(0.25, 0)) == 0.5
    assert orc.decode("e2m1", orc.encode_e2m1_sr(0.25, 32768)) == 0.0
    assert orc.decode("e2m1", orc.encode_e2m1_sr(0.25, 32767)) == 0.5
    for g in grid:
        for u in (0, 65535):
            assert orc.decode("e2m1", orc.encode_e2m1_sr(g, u)) == g
    assert orc.decode("e2m1", orc.encode_e2m1_sr(9.0, 0)) == 6.0


def test_sr_bits_use_one_philox_block_per_8_elements():
    seed, sid = 42, 3
    vals = [orc.sr_u16(seed, sid, L) for L in range(64)]
    assert len(set(vals)) > 56
    # the 8 elements of a group are distinct halves of one 128-bit block
    for g in range(8):
        blk = orc.philox4x32_10([g, 0, sid, 0], [seed, 0])
        halves = []
        for w in blk:
            halves += [int(w) & 0xFFFF, int(w) >> 16]
        assert vals[8 * g:8 * g + 8] == halves


# -------------------------------------------------------------- Hadamard ---
def test_fwht_equals_scipy_hadamard_exactly():
    from scipy.linalg import hadamard
    H = hadamard(32).astype(np.float64)
    assert np.array_equal(H @ H.T, 32 * np.eye(32))
    rng = np.random.default_rng(2)
    for _ in range(200):
        x = rng.integers(-1000, 1000, 32).astype(np.float32)
        assert np.array_equal(orc.fwht32(x).astype(np.float64), H @ x.astype(np.float64))
    x = rng.integers(-50, 50, 32).astype(np.float32)
    assert np.array_equal(orc.fwht32(orc.fwht32(x)), 32 * x)


# ------------------------------------------------------------ SF layout ---
def test_sf_layout_is_a_bijection_onto_512_byte_tiles():
    for rows, kb in ((128, 4), (256, 8), (130, 3), (384, 12)):
        n = orc.sf_bytes(rows, kb)
        assert n == math.ceil(rows / 128) * math.ceil(kb / 4) * 512
        seen = set()
        for r in range(rows):
            for b in range(kb):
                i = orc.sf_index(r, b, kb)
                assert 0 <= i < n and i not in seen
                seen.add(i)
                # same 16-byte row for rows r, r+32, r+64, r+96 of a tile
                assert (i % 512) // 16 == r % 32
    # a tile is contiguous: all scales of rows 0..127, blocks 0..3 fill bytes 0..511
    assert sorted(orc.sf_index(r, b, 8) for r in range(128) for b in range(4)) == list(range(512))


# ------------------------------------------------------------- quantizer ---
def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_colwise_is_rowwise_of_transpose():
    x = workloads.draw("student_t3", (96, 64), 1)
    for fmt in ("mxfp8", "mxfp4", "nvfp4", "moss"):
        a = orc.quantize(_bits(x), fmt, "col")
        b = orc.quantize(_bits(x.t().contiguous()), fmt, "row")
        assert np.array_equal(a.codes, b.codes) and np.array_equal(a.sf_logical, b.sf_logical)
        assert a.amax == b.amax and a.tensor_scale == b.tensor_scale


def test_mx_quantize_is_nearest_at_the_chosen_scale():
    """Brute force on tiny blocks: every code is the nearest grid point to
    x * 2^-e (ties even, saturating) and the scale byte is the FLOOR rule."""
    x = workloads.draw("outliers", (4, 64), 7)
    xf = x.float().numpy().astype(np.float64)
    for fmt, elem, nmax in (("mxfp8", "e4m3", 0x7E), ("mxfp4", "e2m1", 7)):
        q = orc.quantize(_bits(x), fmt, "row")
        grid = np.array([orc.decode(elem, c) for c in range(nmax + 1)])
        for r in range(4):
            for kb in range(2):
                blk = xf[r, 32 * kb:32 * kb + 32]
                e = int(q.sf_logical[r, kb]) - 127
                assert e == math.floor(math.log2(np.abs(blk).max())) - (8 if elem == "e4m3" else 2)
                for i, v in enumerate(blk):
                    k = 32 * kb + i
                    c = q.codes[r, k] if elem == "e4m3" else (q.codes[r, k // 2] >> (4 * (k % 2))) & 0xF
                    a = min(abs(math.ldexp(v, -e)), grid[-1])
                    d = np.abs(grid - a)
                    best = np.flatnonzero(d == d.min())
                    want = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
                    sign = (0x80 if elem == "e4m3" else 0x8) if np.signbit(v) else 0
                    assert c == want | sign


def test_moss_two_level_scales():
    g = gold("moss_two_level.json")
    x = workloads.draw("lognormal_cols", (64, 128), 9)
    xf = x.float().numpy()
    q = orc.quantize(_bits(x), "moss", "row")
    amax = np.float32(np.abs(xf).max())
    assert q.amax == amax
    assert np.float32(q.tensor_scale) == np.float32(amax) / np.float32(g["fp8_max"])
    e = q.sf_logical.astype(int) - 127
    assert e.max() <= 1  # micro scales: fine adjustment below the tensor scale
    dq = q.dequantize() * q.tensor_scale
    # E4M3 keeps 4 significant bits: relative error <= 2^-4 above the subnormal range
    big = np.abs(xf) > 2.0 ** -6 * q.tensor_scale * 2.0 ** e.repeat(32, axis=1)
    rel = np.abs(dq - xf)[big] / np.abs(xf)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-9


def test_nvfp4_scales():
    x = workloads.draw("student_t3", (32, 64), 4)
    xf = x.float().numpy()
    q = orc.quantize(_bits(x), "nvfp4", "row")
    amax = np.float32(np.abs(xf).max())
    assert np.float32(q.tensor_scale) == np.float32(amax) / np.float32(2688.0)
    sfv = np.array([[orc.decode("e4m3", s) for s in row] for row in q.sf_logical])
    assert sfv.max() <= 448 and (q.sf_logical < 0x80).all()
    dq = q.dequantize() * q.tensor_scale
    blkmax = np.abs(xf).reshape(32, 4, 16).max(axis=2)
    # E2M1 step is at most 2^-1 of the block's top binade: error <= block max / 4 * (1 + 1/8)
    err = np.abs(dq - xf).reshape(32, 4, 16).max(axis=2)
    assert np.all(err <= blkmax / 4 * 1.126 + 1e-12)


def test_quantize_rejects_unsupported():
    x = _bits(workloads.draw("normal", (32, 32), 1))
    for fmt in ("moss", "nvfp4_local"):  # the transform is offered on the MX formats and NVFP4
        with pytest.raises(ValueError):
            orc.quantize(x, fmt, hadamard=True)
    with pytest.raises(ValueError):  # NVFP4 blocks of 16, but the transform needs whole 32-groups
        orc.quantize(_bits(workloads.draw("normal", (32, 48), 1)), "nvfp4", hadamard=True)
    with pytest.raises(ValueError):
        orc.quantize(_bits(workloads.draw("normal", (32, 24), 1)), "mxfp8")


def test_hadamard_wgrad_identity():
    """(H a)^T (H b) = 32 a^T b: transforming both operands along K and scaling
    the product by 1/32 leaves dW unchanged up to quantization error."""
    dy = workloads.draw("student_t3", (64, 32), 21, 1e-3)
    xx = workloads.draw("normal", (64, 48), 22)
    exact = dy.double().t() @ xx.double()
    qa = orc.quantize(_bits(dy), "mxfp4", "col", hadamard=True)
    qb = orc.quantize(_bits(xx), "mxfp4", "col", hadamard=True)
    c, _ = orc.gemm(qa, qb, extra_alpha=1.0 / 32)
    rel = np.linalg.norm(c - exact.numpy()) / np.linalg.norm(exact.numpy())
    assert rel < 0.3
    qa0 = orc.quantize(_bits(dy), "mxfp8", "col", hadamard=True)
    qb0 = orc.quantize(_bits(xx), "mxfp8", "col", hadamard=True)
    c0, _ = orc.gemm(qa0, qb0, extra_alpha=1.0 / 32)
    assert np.linalg.norm(c0 - exact.numpy()) / np.linalg.norm(exact.numpy()) < 0.05


# ------------------------------------------------------------------ GEMM ---
@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4", "moss"])
def test_gemm_matches_numpy_fp64_matmul(fmt):
    a = workloads.draw("student_t3", (40, 64), 31)
    b = workloads.draw("normal", (24, 64), 32, 0.02)
    qa, qb = orc.quantize(_bits(a), fmt), orc.quantize(_bits(b), fmt)
    c, cabs = orc.gemm(qa, qb, extra_alpha=0.5)
    alpha = np.float32(np.float32(np.float32(qa.tensor_scale or 1) * np.float32(qb.tensor_scale or 1)) * np.float32(0.5))
    ref = float(alpha) * (qa.dequantize() @ qb.dequantize().T)
    assert np.allclose(c, ref, rtol=1e-12, atol=1e-300)
    assert np.allclose(cabs, abs(float(alpha)) * (np.abs(qa.dequantize()) @ np.abs(qb.dequantize()).T), rtol=1e-12)
    rows, cols = [3, 17, 39], [0, 5, 23]
    cs, _ = orc.gemm(qa, qb, extra_alpha=0.5, rows=rows, cols=cols)
    assert np.array_equal(cs, c[np.ix_(rows, cols)])


def test_gemm_exact_on_small_integers():
    # codes that are small integers with unit scales: every partial sum exact
    rng = np.random.default_rng(8)
    vals = np.array([-6, -4, -3, -2, -1, 0, 1, 2, 3, 4, 6])  # representable in E2M1 too
    a = torch.tensor(rng.choice(vals, (16, 64)), dtype=torch.float32).to(torch.bfloat16)
    b = torch.tensor(rng.choice(vals, (8, 64)), dtype=torch.float32).to(torch.bfloat16)
    exact = (a.double() @ b.double().t()).numpy()
    for fmt in ("mxfp8", "mxfp4"):
        qa = orc.quantize(_bits(a), fmt, rule="ceil")
        qb = orc.quantize(_bits(b), fmt, rule="ceil")
        assert np.array_equal(qa.dequantize(), a.double().numpy())
        c, _ = orc.gemm(qa, qb)
        assert np.array_equal(c, exact)


# ---------------------------------------- fp32 rowwise MX (GEMM epilogue) ---
def test_e4m3_rne_matches_torch_float8_on_random_fp32():
    """The encoder on fp32 values off the bf16 grid (an epilogue quantizes fp32 sums)."""
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(0, 50, 20000), np.exp2(rng.uniform(-12, 9.5, 20000)) *
                        rng.choice([-1, 1], 20000)]).astype(np.float32)
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.encode_rne("e4m3", float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_quantize_rows_f32_equals_bf16_quantize_on_bf16_values(fmt):
    """On values that bf16 holds exactly, the fp32 entry reproduces the pinned
    bf16 quantizer code for code and scale for scale (every finite bf16 value,
    shuffled, plus a heavy-tailed matrix)."""
    pats = workloads.all_bf16_patterns()
    g = torch.Generator().manual_seed(1)
    x = torch.zeros(510 * 128, dtype=torch.bfloat16)
    x[:pats.numel()] = pats[torch.randperm(pats.numel(), generator=g)]
    for xb in (x.view(510, 128), workloads.draw("outliers", (96, 320), 3)):
        bits = xb.contiguous().view(torch.int16).numpy().view(np.uint16)
        a = orc.quantize(bits, fmt)
        b = orc.quantize_rows_f32(xb.float().numpy(), fmt)
        assert np.array_equal(a.codes, b.codes) and np.array_equal(a.sf_logical, b.sf_logical)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_quantize_rows_f32_is_nearest_at_the_floor_scale(fmt):
    """Off the bf16 grid: each block's scale is 2^(floor(log2 max|y|) - emax) and
    each code decodes to a nearest grid value of y at that scale (brute force)."""
    elem, emax = ("e4m3", 8) if fmt == "mxfp8" else ("e2m1", 2)
    rng = np.random.default_rng(4)
    y = (rng.standard_t(3, (8, 64)) * np.exp2(rng.integers(-20, 20, (8, 1)))).astype(np.float32)
    q = orc.quantize_rows_f32(y, fmt)
    deq = q.dequantize()
    grid = np.array(sorted({orc.decode(elem, c) for c in range(0x7F if elem == "e4m3" else 8)}))
    for r in range(8):
        for kb in range(2):
            blk = y[r, kb * 32:(kb + 1) * 32].astype(np.float64)
            e = math.floor(math.log2(np.abs(blk).max())) - emax
            assert q.sf_logical[r, kb] == e + 127
            s = 2.0 ** e
            for v, dv in zip(blk, deq[r, kb * 32:(kb + 1) * 32]):
                a = min(abs(v) / s, grid[-1])
                assert abs(abs(dv) / s - a) <= np.abs(grid - a).min() + 1e-12


# ------------------------------------------------- E4M3 stochastic rounding ---
def test_e4m3_sr_unbiased_and_probability():
    """E4M3 SR rounds |v| up to the next grid value with probability
    (|v| - lo) / (hi - lo): the empirical frequency and mean over uniform u16
    match, in every binade, the subnormals and at saturation."""
    grid = sorted({orc.decode("e4m3", c) for c in range(0x7F)})
    rng = np.random.default_rng(12)
    for v in [1e-4, 0.0029, 0.013, 0.9, 1.0625, 3.3, 17.0, 100.5, 300.0, 447.0, -6.1, -0.3]:
        n = 4000
        us = rng.integers(0, 65536, n)
        dec = np.array([orc.decode("e4m3", orc.encode_e4m3_sr(v, int(u))) for u in us])
        a = abs(v)
        lo = max(g for g in grid if g <= a)
        hi = min(g for g in grid if g > a)
        p = (a - lo) / (hi - lo)
        assert set(np.abs(dec)) <= {lo, hi}
        assert np.all(np.sign(dec[dec != 0]) == np.sign(v))
        frac_up = np.mean(np.abs(dec) == hi)
        assert abs(frac_up - p) < 4 * math.sqrt(p * (1 - p) / n) + 1e-3
        sd = (hi - lo) * math.sqrt(p * (1 - p) / n)
        assert abs(dec.mean() - v) < 4 * sd + 1e-6
    for g in grid[::7] + [448.0]:
        for u in (0, 65535):
            assert orc.decode("e4m3", orc.encode_e4m3_sr(g, u)) == g
    assert orc.decode("e4m3", orc.encode_e4m3_sr(1000.0, 0)) == 448.0
    # exact threshold: halfway between 1.0 and 1.125 rounds up iff u16 < 32768
    assert orc.encode_e4m3_sr(1.0625, 32767) == 0x39 and orc.encode_e4m3_sr(1.0625, 32768) == 0x38


@pytest.mark.parametrize("fmt", ["mxfp8", "moss"])
def test_e4m3_sr_quantize_is_unbiased_at_the_chosen_scale(fmt):
    """Quantize with SR: per element the code is one of the two grid neighbours
    of the scaled value (the RNE result's scale), and averaged over seeds the
    dequantized tensor approaches the scaled input."""
    x = workloads.draw("student_t3", (32, 64), 21)
    xb = _bits(x)
    rne = orc.quantize(xb, fmt)
    acc = np.zeros((32, 64))
    n = 64
    for seed in range(n):
        q = orc.quantize(xb, fmt, rounding="sr", seed=seed)
        assert np.array_equal(q.sf_logical, rne.sf_logical)
        acc += q.dequantize()  # code x block scale (the tensor scale is applied in the GEMM epilogue)
    y = x.double().numpy()
    if fmt == "moss":
        y = (x.float() / np.float32(rne.tensor_scale)).double().numpy()
    grid = np.array(sorted({orc.decode("e4m3", c) for c in range(0x7F)}))
    s = np.repeat(np.exp2(rne.sf_logical.astype(np.float64) - 127), 32, axis=1)
    a = np.minimum(np.abs(y) / s, 448.0)
    hi = grid[np.minimum(np.searchsorted(grid, a, side="right"), len(grid) - 1)]
    lo = grid[np.maximum(np.searchsorted(grid, a, side="right") - 1, 0)]
    bound = 5 * s * (hi - lo) / (2 * math.sqrt(n)) + 1e-12
    sat = np.abs(y) / s >= 448.0  # the FLOOR rule lets a block max land in (448, 512): it saturates
    assert np.all(np.abs(acc / n - y)[~sat] <= bound[~sat])
    assert np.allclose(np.abs(acc / n)[sat], 448.0 * s[sat])


# ------------------------------------------------ CTA-local NVFP4 (regions) ---
@pytest.mark.parametrize("direction", ["row", "col"])
def test_nvfp4_local_is_global_nvfp4_per_region(direction):
    """nvfp4_local = the pinned global NVFP4 quantizer applied to each region of
    128 operand rows on its own (last region ragged), codes, scales, amax and
    tensor scale alike."""
    x = workloads.draw("lognormal_cols", (320, 416), 7)
    xb = _bits(x)
    q = orc.quantize(xb, "nvfp4_local", direction)
    rows = q.rows
    assert q.tensor_scale.shape == (-(-rows // 128),)
    for g in range(q.tensor_scale.shape[0]):
        sl = slice(128 * g, min(128 * (g + 1), rows))
        part = xb[sl] if direction == "row" else np.ascontiguousarray(xb[:, sl])
        ref = orc.quantize(part, "nvfp4", direction)
        assert np.array_equal(ref.codes, q.codes[sl]) and np.array_equal(ref.sf_logical, q.sf_logical[sl])
        assert np.float32(ref.amax) == q.amax[g] and np.float32(ref.tensor_scale) == q.tensor_scale[g]
    # a caller's per-region amax replaces the computed one
    ain = q.amax * 2
    q2 = orc.quantize(xb, "nvfp4_local", direction, amax_in=ain)
    assert np.array_equal(q2.amax, ain.astype(np.float32))
    part = xb[:128] if direction == "row" else np.ascontiguousarray(xb[:, :128])
    ref = orc.quantize(part, "nvfp4", direction, amax_in=float(ain[0]))
    assert np.array_equal(ref.codes, q2.codes[:128])


def test_nvfp4_local_gemm_matches_numpy_with_region_scales():
    """Region scales are constant along K, so they factor out of each output:
    C[i, j] = s_A[i // 128] s_B[j // 128] sum_k dq(A)[i, k] dq(B)[j, k]."""
    a = workloads.draw("student_t3", (300, 256), 8)
    b = workloads.draw("normal", (260, 256), 9, 0.02)
    qa, qb = orc.quantize(_bits(a), "nvfp4_local"), orc.quantize(_bits(b), "nvfp4_local")
    c, _ = orc.gemm(qa, qb, extra_alpha=0.5)
    ta = np.repeat(qa.tensor_scale.astype(np.float64), 128)[:300]
    tb = np.repeat(qb.tensor_scale.astype(np.float64), 128)[:260]
    ref = (qa.dequantize() * ta[:, None]) @ (qb.dequantize() * tb[:, None]).T * 0.5
    assert np.allclose(c, ref, rtol=1e-6, atol=0)
