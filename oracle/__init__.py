"""CPU oracle for the block-scaled (microscaling) low-precision linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library (``fp4_precision_gemms_gb300``) and never
imports it.

The arithmetic lives in ``mx_oracle.c`` (plain C, fp64 where the pages fix no
precision); this module only builds it with gcc and marshals numpy arrays.
Citations of the pages are in ``mx_oracle.h``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")

# Oracle-private enum values (mirror mx_oracle.h).
FMT = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2, "moss": 3, "nvfp4_local": 4}
LOCAL_REGION = 128  # operand rows per FP32 scale in nvfp4_local
ROUND = {"rne": 0, "sr": 1}
RULE = {"default": 0, "floor": 1, "ceil": 2, "nearest": 3}
DIR = {"row": 0, "col": 1}
ELEM = {"e4m3": 0, "e2m1": 1}
BLOCK = {"mxfp8": 32, "mxfp4": 32, "nvfp4": 16, "moss": 32, "nvfp4_local": 16}
FP4 = {"mxfp4", "nvfp4", "nvfp4_local"}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liborc.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mx_oracle.h"))):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off"]
    tmp = _LIB + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base + extra + [_SRC, "-o", tmp, "-lm"], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB)
            return _LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            p, i64, u64, u32, i32 = C.c_void_p, C.c_int64, C.c_uint64, C.c_uint32, C.c_int
            L.orc_bf16_to_f32.restype = C.c_float
            L.orc_bf16_to_f32.argtypes = [C.c_uint16]
            L.orc_f32_to_bf16_rne.restype = C.c_uint16
            L.orc_f32_to_bf16_rne.argtypes = [C.c_float]
            for n in ("orc_decode_e4m3", "orc_decode_e2m1", "orc_decode_e8m0"):
                getattr(L, n).restype = C.c_double
                getattr(L, n).argtypes = [C.c_uint]
            for n in ("orc_encode_e4m3_rne", "orc_encode_e2m1_rne"):
                getattr(L, n).restype = C.c_uint
                getattr(L, n).argtypes = [C.c_float]
            L.orc_encode_e2m1_sr.restype = C.c_uint
            L.orc_encode_e2m1_sr.argtypes = [C.c_float, C.c_uint]
            L.orc_encode_e4m3_sr.restype = C.c_uint
            L.orc_encode_e4m3_sr.argtypes = [C.c_float, C.c_uint]
            L.orc_pow2_exponent.restype = i32
            L.orc_pow2_exponent.argtypes = [C.c_float, i32, i32]
            L.orc_philox4x32_10.restype = None
            L.orc_philox4x32_10.argtypes = [p, p, p]
            L.orc_sr_u16.restype = C.c_uint
            L.orc_sr_u16.argtypes = [u64, u32, u64]
            L.orc_fwht32.restype = None
            L.orc_fwht32.argtypes = [p]
            L.orc_sf_index.restype = i64
            L.orc_sf_index.argtypes = [i64, i64, i64]
            L.orc_sf_bytes.restype = i64
            L.orc_sf_bytes.argtypes = [i64, i64]
            L.orc_sf_swizzle.restype = None
            L.orc_sf_swizzle.argtypes = [p, i64, i64, p]
            L.orc_amax_bf16.restype = C.c_float
            L.orc_amax_bf16.argtypes = [p, i64, i64, i64]
            L.orc_quantize.restype = i32
            L.orc_quantize.argtypes = [p, i64, i64, i64, i32, i32, i32, i32, i32, u64, u32, i32,
                                       p, p, p, p, p]
            L.orc_quantize_rows_f32.restype = i32
            L.orc_quantize_rows_f32.argtypes = [p, i64, i64, i64, i32, p, p]
            L.orc_dequantize.restype = None
            L.orc_dequantize.argtypes = [p, p, i64, i64, i32, i32, p]
            L.orc_gemm_alpha.restype = C.c_float
            L.orc_gemm_alpha.argtypes = [p, p, C.c_float]
            L.orc_gemm_q.restype = None
            L.orc_gemm_q.argtypes = [p, p, p, p, i32, i32, i64, i64, i64, C.c_double,
                                     p, i64, p, i64, p, p]
            L.orc_num_threads.restype = i32
            L.orc_num_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- scalars ---
def decode(elem: str, code: int) -> float:
    return {"e4m3": lib().orc_decode_e4m3, "e2m1": lib().orc_decode_e2m1,
            "e8m0": lib().orc_decode_e8m0}[elem](int(code))


def encode_rne(elem: str, v: float) -> int:
    f = lib().orc_encode_e4m3_rne if elem == "e4m3" else lib().orc_encode_e2m1_rne
    return int(f(float(np.float32(v))))


def encode_e2m1_sr(v: float, u16: int) -> int:
    return int(lib().orc_encode_e2m1_sr(float(np.float32(v)), int(u16)))


def encode_e4m3_sr(v: float, u16: int) -> int:
    return int(lib().orc_encode_e4m3_sr(float(np.float32(v)), int(u16)))


def pow2_exponent(block_amax: float, rule: str, elem: str) -> int:
    return int(lib().orc_pow2_exponent(float(np.float32(block_amax)), RULE[rule], ELEM[elem]))


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_u16(seed: int, stream_id: int, L: int) -> int:
    return int(lib().orc_sr_u16(seed, stream_id, L))


def fwht32(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32).copy()
    assert a.shape == (32,)
    lib().orc_fwht32(_ptr(a))
    return a


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_rne(x) -> int:
    return int(lib().orc_f32_to_bf16_rne(float(np.float32(x))))


# ----------------------------------------------------------------- layout ---
def sf_index(r: int, kb: int, kblocks: int) -> int:
    return int(lib().orc_sf_index(r, kb, kblocks))


def sf_bytes(rows: int, kblocks: int) -> int:
    return int(lib().orc_sf_bytes(rows, kblocks))


def sf_swizzle(sf_logical: np.ndarray, fill: int = 0) -> np.ndarray:
    s = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    rows, kblocks = s.shape
    out = np.full(sf_bytes(rows, kblocks), fill, dtype=np.uint8)
    lib().orc_sf_swizzle(_ptr(s), rows, kblocks, _ptr(out))
    return out


# -------------------------------------------------------------- quantizer ---
class OracleQuant:
    """Result of oracle.quantize: K-major codes and logical block scales."""

    def __init__(self, fmt, rows, k, codes, sf_logical, amax, tensor_scale, hadamard):
        self.fmt, self.rows, self.k = fmt, rows, k
        self.block = BLOCK[fmt]
        self.codes, self.sf_logical = codes, sf_logical
        self.amax, self.tensor_scale, self.hadamard = amax, tensor_scale, hadamard

    def sf_swizzled(self, fill: int = 0) -> np.ndarray:
        return sf_swizzle(self.sf_logical, fill)

    def dequantize(self) -> np.ndarray:
        out = np.empty((self.rows, self.k), dtype=np.float64)
        lib().orc_dequantize(_ptr(self.codes), _ptr(self.sf_logical), self.rows, self.k,
                             FMT[self.fmt], self.block, _ptr(out))
        return out


def amax_bf16(x_bits: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, Cc = x.shape
    return float(lib().orc_amax_bf16(_ptr(x), R, Cc, Cc))


def quantize(x_bits: np.ndarray, fmt: str, direction: str = "row", rounding: str = "rne",
             rule: str = "default", seed: int = 0, stream_id: int = 0, hadamard: bool = False,
             amax_in: float | None = None) -> OracleQuant:
    """Quantize a bf16 matrix given as uint16 bit patterns [R, C]."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, Cc = x.shape
    rows, k = (R, Cc) if direction == "row" else (Cc, R)
    block = BLOCK[fmt]
    kbytes = k // 2 if fmt in FP4 else k
    codes = np.zeros((rows, kbytes), dtype=np.uint8)
    sf = np.zeros((rows, k // block), dtype=np.uint8)
    nreg = max(1, -(-rows // LOCAL_REGION)) if fmt == "nvfp4_local" else 1
    amax = np.zeros(nreg, dtype=np.float32)
    ts = np.ones(nreg, dtype=np.float32)
    ain = None if amax_in is None else np.atleast_1d(np.asarray(amax_in, dtype=np.float32))
    rc = lib().orc_quantize(_ptr(x), R, Cc, Cc, DIR[direction], FMT[fmt], block, ROUND[rounding],
                            RULE[rule], seed, stream_id, int(bool(hadamard)), _ptr(ain),
                            _ptr(codes), _ptr(sf), _ptr(amax), _ptr(ts))
    if rc != 0:
        raise ValueError(f"oracle quantize rejected the arguments (code {rc})")
    if fmt == "nvfp4_local":  # one FP32 scale per region of LOCAL_REGION operand rows
        return OracleQuant(fmt, rows, k, codes, sf, amax.copy(), ts.copy(), bool(hadamard))
    tsv = float(ts[0]) if fmt in ("moss", "nvfp4") else None
    return OracleQuant(fmt, rows, k, codes, sf, float(amax[0]), tsv, bool(hadamard))


def quantize_rows_f32(x: np.ndarray, fmt: str) -> OracleQuant:
    """Rowwise MXFP8 / MXFP4 quantization (FLOOR rule, RNE) of an fp32 matrix [R, C]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, Cc = x.shape
    kbytes = Cc // 2 if fmt in FP4 else Cc
    codes = np.zeros((R, kbytes), dtype=np.uint8)
    sf = np.zeros((R, Cc // 32), dtype=np.uint8)
    rc = lib().orc_quantize_rows_f32(_ptr(x), R, Cc, Cc, FMT[fmt], _ptr(codes), _ptr(sf))
    if rc != 0:
        raise ValueError(f"oracle quantize_rows_f32 rejected the arguments (code {rc})")
    return OracleQuant(fmt, R, Cc, codes, sf, 0.0, None, False)


def gemm_alpha(ts_a: float | None, ts_b: float | None, extra: float = 1.0) -> float:
    a = None if ts_a is None else np.array([ts_a], dtype=np.float32)
    b = None if ts_b is None else np.array([ts_b], dtype=np.float32)
    return float(lib().orc_gemm_alpha(_ptr(a), _ptr(b), float(np.float32(extra))))


def gemm(A: OracleQuant, B: OracleQuant, extra_alpha: float = 1.0, rows=None, cols=None):
    """fp64 C = alpha * dq(A) dq(B)^T over the selected rows/cols; returns (C, Cabs)."""
    assert A.fmt == B.fmt and A.k == B.k
    if A.fmt == "nvfp4_local":
        # alpha varies with the region pair (row // LOCAL_REGION, col // LOCAL_REGION): the
        # scales are constant along K, so they factor out of each output's K-sum
        r = np.arange(A.rows) if rows is None else np.asarray(rows, dtype=np.int64)
        c = np.arange(B.rows) if cols is None else np.asarray(cols, dtype=np.int64)
        # the same codes and block scales read as NVFP4 without a tensor scale (alpha 1)
        ones = OracleQuant("nvfp4", A.rows, A.k, A.codes, A.sf_logical, 0.0, None, A.hadamard)
        onesb = OracleQuant("nvfp4", B.rows, B.k, B.codes, B.sf_logical, 0.0, None, B.hadamard)
        c1, a1 = gemm(ones, onesb, 1.0, r, c)
        al = np.array([[gemm_alpha(float(A.tensor_scale[i // LOCAL_REGION]), float(B.tensor_scale[j // LOCAL_REGION]),
                                   extra_alpha) for j in range(0, B.rows, LOCAL_REGION)]
                       for i in range(0, A.rows, LOCAL_REGION)], dtype=np.float64)
        alpha = al[np.ix_(r // LOCAL_REGION, c // LOCAL_REGION)]
        return alpha * c1, np.abs(alpha) * a1
    alpha = gemm_alpha(A.tensor_scale, B.tensor_scale, extra_alpha)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = A.rows if r is None else len(r)
    nc = B.rows if c is None else len(c)
    out = np.zeros((nr, nc), dtype=np.float64)
    oabs = np.zeros((nr, nc), dtype=np.float64)
    lib().orc_gemm_q(_ptr(A.codes), _ptr(A.sf_logical), _ptr(B.codes), _ptr(B.sf_logical),
                     FMT[A.fmt], A.block, A.rows, B.rows, A.k, alpha, _ptr(r), nr, _ptr(c), nc,
                     _ptr(out), _ptr(oabs))
    return out, oabs


def num_threads() -> int:
    return int(lib().orc_num_threads())
