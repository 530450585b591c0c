"""GB300-native block-scaled (MXFP8 / MXFP4 / NVFP4 / MOSS two-level FP8) linear layer.

A thin ctypes binding over ``libmx_gb300.so`` (C ABI in ``include/mx.h``).  This
module only marshals arguments: every step of quantize, GEMM and the linear
layer's passes runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.  There is no CPU fallback: without the built library (see
``build()``) or an sm_103 GPU every call raises ``MXError``.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmx_gb300.so")

FORMATS = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2, "moss": 3, "nvfp4_local": 4}
BLOCK = {"mxfp8": 32, "mxfp4": 32, "nvfp4": 16, "moss": 32, "nvfp4_local": 16}
FP4 = ("mxfp4", "nvfp4", "nvfp4_local")
ROUNDING = {"rne": 0, "sr": 1}
RULES = {"default": 0, "floor": 1, "ceil": 2, "nearest": 3}
DIRS = {"row": 0, "col": 1}
OUT = {torch.float32: 0, torch.bfloat16: 1}

MX_OK, MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED, MX_ERR_ALIGNMENT = 0, 1, 2, 3
MX_ERR_CUDA, MX_ERR_TIMEOUT, MX_ERR_NO_DEVICE, MX_ERR_WORKSPACE = 4, 5, 6, 7

EXPORTED = ("mx_codes_bytes", "mx_sf_bytes", "mx_scale_count", "mx_amax", "mx_quantize", "mx_quantize_dual", "mx_dequantize", "mx_gemm",
            "mx_gemm_amax", "mx_gemm_quantized",
            "mx_linear_workspace_bytes", "mx_linear_fwd", "mx_linear_fwd_noalloc", "mx_linear_bwd",
            "mx_linear_saved_bytes", "mx_linear_fwd_save", "mx_linear_bwd_saved", "mx_strerror",
            "mx_last_device_status", "mx_selftest_bounded_wait", "mx_launch_count",
            "mx_debug_divide", "mx_debug_set_quant_impl", "mx_debug_set_tile_fail_at", "mx_debug_set_bwd_fork", "mx_debug_set_gemm_variant",
            "mx_debug_last_gemm_variant")


class MXError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (mx_status {code})" if what else strerror(code))


class _CTensor(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("sf", C.c_void_p), ("amax", C.c_void_p),
                ("tensor_scale", C.c_void_p), ("rows", C.c_int64), ("k", C.c_int64),
                ("fmt", C.c_int32), ("block", C.c_int32), ("hadamard", C.c_int32),
                ("reserved", C.c_int32)]


class _CBwdOpts(C.Structure):
    _fields_ = [("wgrad_hadamard", C.c_int32), ("wgrad_dy_rounding", C.c_int32),
                ("seed", C.c_uint64), ("stream_id", C.c_uint32), ("reserved", C.c_int32)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libmx_gb300.so in-tree for sm_103a (nvcc)."""
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise MXError(MX_ERR_NO_DEVICE, f"{LIB_PATH} is not built (call build())")
            L = C.CDLL(LIB_PATH)
            p, i64, i32, u64, u32, sz = C.c_void_p, C.c_int64, C.c_int, C.c_uint64, C.c_uint32, C.c_size_t
            L.mx_codes_bytes.restype = sz
            L.mx_codes_bytes.argtypes = [i32, i64, i64]
            L.mx_sf_bytes.restype = sz
            L.mx_sf_bytes.argtypes = [i32, i64, i64]
            L.mx_scale_count.restype = sz
            L.mx_scale_count.argtypes = [i32, i64]
            L.mx_amax.restype = i32
            L.mx_amax.argtypes = [p, i64, i64, i64, p, p]
            L.mx_quantize.restype = i32
            L.mx_quantize.argtypes = [p, i64, i64, i64, i32, i32, i32, i32, i32, u64, u32, i32, p,
                                      C.POINTER(_CTensor), p]
            L.mx_quantize_dual.restype = i32
            L.mx_quantize_dual.argtypes = [p, i64, i64, i64, i32, i32, i32, u64, u32, i32, i32, i32, i32, p,
                                           C.POINTER(_CTensor), C.POINTER(_CTensor), p]
            L.mx_debug_set_quant_impl.restype = None
            L.mx_debug_set_quant_impl.argtypes = [i32]
            L.mx_debug_set_tile_fail_at.restype = None
            L.mx_debug_set_tile_fail_at.argtypes = [i64]
            L.mx_debug_set_bwd_fork.restype = None
            L.mx_debug_set_bwd_fork.argtypes = [i32]
            L.mx_dequantize.restype = i32
            L.mx_dequantize.argtypes = [C.POINTER(_CTensor), p, p]
            L.mx_gemm.restype = i32
            L.mx_gemm.argtypes = [C.POINTER(_CTensor), C.POINTER(_CTensor), C.c_float, p, i64, i32, p]
            L.mx_gemm_amax.restype = i32
            L.mx_gemm_amax.argtypes = [C.POINTER(_CTensor), C.POINTER(_CTensor), C.c_float, p, i64, i32, p, p]
            L.mx_gemm_quantized.restype = i32
            L.mx_gemm_quantized.argtypes = [C.POINTER(_CTensor), C.POINTER(_CTensor), C.c_float,
                                            C.POINTER(_CTensor), p]
            L.mx_linear_workspace_bytes.restype = sz
            L.mx_linear_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
            L.mx_linear_fwd.restype = i32
            L.mx_linear_fwd.argtypes = [p, p, i64, i64, i64, i32, p, i32, p, sz, p]
            L.mx_linear_fwd_noalloc.restype = i32
            L.mx_linear_fwd_noalloc.argtypes = [p, p, i64, i64, i64, i32, p, i32, p]
            L.mx_linear_bwd.restype = i32
            L.mx_linear_bwd.argtypes = [p, p, p, i64, i64, i64, i32, C.POINTER(_CBwdOpts), p, i32, p,
                                        i32, p, sz, p]
            L.mx_linear_saved_bytes.restype = sz
            L.mx_linear_saved_bytes.argtypes = [i64, i64, i64, i32]
            L.mx_linear_fwd_save.restype = i32
            L.mx_linear_fwd_save.argtypes = [p, p, i64, i64, i64, i32, p, p, C.POINTER(_CBwdOpts), p, i32, p, sz,
                                             p, sz, p]
            L.mx_linear_bwd_saved.restype = i32
            L.mx_linear_bwd_saved.argtypes = [p, i64, i64, i64, i32, p, C.POINTER(_CBwdOpts), p, sz, p, i32, p, i32,
                                              p, sz, p]
            L.mx_strerror.restype = C.c_char_p
            L.mx_strerror.argtypes = [i32]
            L.mx_last_device_status.restype = i32
            L.mx_last_device_status.argtypes = [p]
            L.mx_selftest_bounded_wait.restype = i32
            L.mx_selftest_bounded_wait.argtypes = [u64, p]
            L.mx_launch_count.restype = u64
            L.mx_launch_count.argtypes = []
            L.mx_debug_divide.restype = i32
            L.mx_debug_divide.argtypes = [p, p, i64, p, p, p]
            L.mx_debug_set_gemm_variant.restype = None
            L.mx_debug_set_gemm_variant.argtypes = [i32]
            L.mx_debug_last_gemm_variant.restype = i32
            L.mx_debug_last_gemm_variant.argtypes = []
            _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().mx_strerror(int(code)).decode()
    except Exception:
        return f"mx_status {code}"


def _check(rc: int, what: str):
    if rc != MX_OK:
        raise MXError(rc, what)


def _stream(stream=None):
    if stream is None:
        if not torch.cuda.is_available():
            return None  # the library reports MX_ERR_NO_DEVICE
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _on_gpu(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise MXError(MX_ERR_NO_DEVICE if not torch.cuda.is_available() else MX_ERR_INVALID_ARG,
                          "tensors must live on a CUDA device (there is no CPU path)")


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


class MXTensor:
    """A quantized K-major operand: codes, swizzled block scales, amax and tensor scale."""

    def __init__(self, fmt: str, rows: int, k: int, device=None):
        device = device or torch.device("cuda")
        self.fmt, self.rows, self.k = fmt, int(rows), int(k)
        self.block = BLOCK[fmt]
        self.hadamard = False
        L = lib()
        nc = L.mx_codes_bytes(FORMATS[fmt], self.rows, self.k)
        ns = L.mx_sf_bytes(FORMATS[fmt], self.rows, self.k)
        if (nc == 0 or ns == 0) and self.rows * self.k > 0:
            raise MXError(MX_ERR_INVALID_ARG, f"operand shape {rows}x{k} for {fmt}")
        kb = self.k // 2 if fmt in FP4 else self.k
        self.codes = torch.empty((self.rows, kb), dtype=torch.uint8, device=device)
        self.sf = torch.empty(max(ns, 1), dtype=torch.uint8, device=device)
        # amax and tensor scale: one each, or one per 128-row region (nvfp4_local)
        self.nscale = max(1, int(L.mx_scale_count(FORMATS[fmt], self.rows)))
        self.scalars = torch.zeros(2 * self.nscale, dtype=torch.float32, device=device)

    @property
    def amax(self):
        return self.scalars[0:self.nscale]

    @property
    def tensor_scale(self):
        return self.scalars[self.nscale:2 * self.nscale]

    def _c(self) -> _CTensor:
        t = _CTensor()
        _on_gpu(self.codes, self.sf, self.scalars)  # the library only reads and writes device memory
        t.codes = self.codes.data_ptr()
        t.sf = self.sf.data_ptr()
        t.amax = self.scalars.data_ptr()
        t.tensor_scale = self.scalars.data_ptr() + 4 * self.nscale
        t.rows, t.k = self.rows, self.k
        t.fmt, t.block, t.hadamard = FORMATS[self.fmt], self.block, int(self.hadamard)
        return t


def amax(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    _on_gpu(x, out)
    out = out if out is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().mx_amax(_ptr(x), x.shape[0], x.shape[1], x.stride(0), _ptr(out), _stream(stream)),
           "mx_amax")
    return out


def quantize(x: torch.Tensor, fmt: str, direction: str = "row", rounding: str = "rne",
             rule: str = "default", seed: int = 0, stream_id: int = 0, hadamard: bool = False,
             amax_in: torch.Tensor | None = None, out: MXTensor | None = None, stream=None) -> MXTensor:
    """bf16 [R, C] -> block-scaled K-major operand (rowwise: [R, C]; colwise: [C, R])."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    _on_gpu(x, amax_in)
    R, Cc = x.shape
    rows, k = (R, Cc) if direction == "row" else (Cc, R)
    q = out if out is not None else MXTensor(fmt, rows, k, x.device)
    ct = q._c()
    rc = lib().mx_quantize(_ptr(x), R, Cc, x.stride(0), DIRS[direction], FORMATS[fmt], BLOCK[fmt],
                           ROUNDING[rounding], RULES[rule], seed, stream_id, int(bool(hadamard)),
                           _ptr(amax_in), C.byref(ct), _stream(stream))
    _check(rc, "mx_quantize")
    q.rows, q.k, q.hadamard = ct.rows, ct.k, bool(ct.hadamard)
    return q


def quantize_dual(x: torch.Tensor, fmt: str, rule: str = "default", seed: int = 0, stream_id: int = 0,
                  row_rounding: str = "rne", row_hadamard: bool = False, col_rounding: str = "rne",
                  col_hadamard: bool = False, amax_in: torch.Tensor | None = None,
                  row_out: MXTensor | None = None, col_out: MXTensor | None = None, stream=None):
    """One read of bf16 x [R, C] -> (rowwise operand [R, C], colwise operand [C, R])."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    _on_gpu(x, amax_in)
    R, Cc = x.shape
    qr = row_out if row_out is not None else MXTensor(fmt, R, Cc, x.device)
    qc = col_out if col_out is not None else MXTensor(fmt, Cc, R, x.device)
    cr, cc = qr._c(), qc._c()
    rc = lib().mx_quantize_dual(_ptr(x), R, Cc, x.stride(0), FORMATS[fmt], BLOCK[fmt], RULES[rule], seed,
                                stream_id, ROUNDING[row_rounding], int(bool(row_hadamard)),
                                ROUNDING[col_rounding], int(bool(col_hadamard)), _ptr(amax_in),
                                C.byref(cr), C.byref(cc), _stream(stream))
    _check(rc, "mx_quantize_dual")
    qr.rows, qr.k, qr.hadamard = cr.rows, cr.k, bool(cr.hadamard)
    qc.rows, qc.k, qc.hadamard = cc.rows, cc.k, bool(cc.hadamard)
    return qr, qc


QUANT_IMPLS = {"auto": 0, "direct": 1, "tile": 2}


def set_quant_impl(impl: str) -> None:
    """Choose the producer implementation (tests and tuning)."""
    lib().mx_debug_set_quant_impl(QUANT_IMPLS[impl])


def set_tile_fail_at(tile: int) -> None:
    """Test hook: the tile producer gives up its wait on this tile of each CTA (-1: off)."""
    lib().mx_debug_set_tile_fail_at(int(tile))


def set_bwd_fork(on: bool) -> None:
    """Whether linear_bwd / linear_bwd_saved run the weight gradient on the
    library's side stream (the default) or after the data gradient on the
    caller's stream.  Per host thread."""
    lib().mx_debug_set_bwd_fork(int(on))


def dequantize(q: MXTensor, stream=None) -> torch.Tensor:
    out = torch.empty((q.rows, q.k), dtype=torch.float32, device=q.codes.device)
    ct = q._c()
    _check(lib().mx_dequantize(C.byref(ct), _ptr(out), _stream(stream)), "mx_dequantize")
    return out


def gemm(a: MXTensor, b: MXTensor, extra_alpha: float = 1.0, out_dtype=torch.float32,
         out: torch.Tensor | None = None, stream=None, amax_out: torch.Tensor | None = None) -> torch.Tensor:
    """C[M, N] = alpha * dq(a) dq(b)^T on the tensor cores.  amax_out: an
    optional one-element fp32 device tensor that receives max |C| as written,
    reduced in the GEMM's epilogue."""
    _on_gpu(out, amax_out)
    out = out if out is not None else torch.empty((a.rows, b.rows), dtype=out_dtype,
                                                  device=a.codes.device)
    ca, cb = a._c(), b._c()
    if amax_out is None:
        rc = lib().mx_gemm(C.byref(ca), C.byref(cb), float(extra_alpha), _ptr(out), out.stride(0),
                           OUT[out.dtype], _stream(stream))
        _check(rc, "mx_gemm")
    else:
        if amax_out.dtype != torch.float32 or amax_out.numel() < 1:
            raise ValueError("amax_out must be a float32 tensor with at least one element")
        rc = lib().mx_gemm_amax(C.byref(ca), C.byref(cb), float(extra_alpha), _ptr(out), out.stride(0),
                                OUT[out.dtype], _ptr(amax_out), _stream(stream))
        _check(rc, "mx_gemm_amax")
    return out


def gemm_quantized(a: MXTensor, b: MXTensor, fmt: str = "mxfp8", extra_alpha: float = 1.0,
                   out: MXTensor | None = None, stream=None) -> MXTensor:
    """alpha * dq(a) dq(b)^T quantized in the GEMM epilogue into the rowwise MX
    operand (rows M = a.rows, K = N = b.rows) of format fmt (mxfp8 or mxfp4)."""
    out = out if out is not None else MXTensor(fmt, a.rows, b.rows, a.codes.device)
    ca, cb, co = a._c(), b._c(), out._c()
    _check(lib().mx_gemm_quantized(C.byref(ca), C.byref(cb), float(extra_alpha), C.byref(co), _stream(stream)),
           "mx_gemm_quantized")
    return out


PASSES = {"fwd": 0, "bwd": 1, "bwd_saved": 2}


def workspace_bytes(T: int, Kin: int, Nout: int, fmt: str, pass_: str = "fwd") -> int:
    return int(lib().mx_linear_workspace_bytes(T, Kin, Nout, FORMATS[fmt], PASSES[pass_]))


def saved_bytes(T: int, Kin: int, Nout: int, fmt: str) -> int:
    """Bytes of one layer's saved backward state (X^T and W^T operands)."""
    return int(lib().mx_linear_saved_bytes(T, Kin, Nout, FORMATS[fmt]))


def linear_fwd(X: torch.Tensor, W: torch.Tensor, fmt: str, out_dtype=torch.bfloat16,
               workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Y = X W^T with X [T, Kin], W [Nout, Kin] (bf16, contiguous)."""
    _on_gpu(X, W, workspace, out)
    T, Kin = X.shape
    Nout = W.shape[0]
    n = workspace_bytes(T, Kin, Nout, fmt, "fwd")
    ws = workspace if workspace is not None else torch.empty(n, dtype=torch.uint8, device=X.device)
    Y = out if out is not None else torch.empty((T, Nout), dtype=out_dtype, device=X.device)
    rc = lib().mx_linear_fwd(_ptr(X), _ptr(W), T, Kin, Nout, FORMATS[fmt], _ptr(Y), OUT[Y.dtype],
                             _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mx_linear_fwd")
    return Y


def linear_fwd_noalloc(X: torch.Tensor, W: torch.Tensor, fmt: str, out_dtype=torch.bfloat16,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """linear_fwd without a workspace: the library's fixed device array holds the
    quantized operands (for callers that cannot allocate; up to 32 MiB)."""
    _on_gpu(X, W, out)
    T, Kin = X.shape
    Nout = W.shape[0]
    Y = out if out is not None else torch.empty((T, Nout), dtype=out_dtype, device=X.device)
    rc = lib().mx_linear_fwd_noalloc(_ptr(X), _ptr(W), T, Kin, Nout, FORMATS[fmt], _ptr(Y),
                                     OUT[Y.dtype], _stream(stream))
    _check(rc, "mx_linear_fwd_noalloc")
    return Y


def linear_bwd(dY: torch.Tensor, X: torch.Tensor, W: torch.Tensor, fmt: str,
               wgrad_hadamard: bool = False, wgrad_dy_rounding: str = "rne", seed: int = 0,
               stream_id: int = 0, dx_dtype=torch.bfloat16, dw_dtype=torch.float32,
               need_dx: bool = True, need_dw: bool = True, workspace: torch.Tensor | None = None,
               dX: torch.Tensor | None = None, dW: torch.Tensor | None = None, stream=None):
    """dX = dY W and dW = dY^T X for the layer Y = X W^T."""
    _on_gpu(dY, X, W, workspace, dX, dW)
    T, Kin = X.shape
    Nout = W.shape[0]
    n = workspace_bytes(T, Kin, Nout, fmt, "bwd")
    ws = workspace if workspace is not None else torch.empty(n, dtype=torch.uint8, device=X.device)
    if need_dx and dX is None:
        dX = torch.empty((T, Kin), dtype=dx_dtype, device=X.device)
    if need_dw and dW is None:
        dW = torch.empty((Nout, Kin), dtype=dw_dtype, device=X.device)
    o = _CBwdOpts(int(bool(wgrad_hadamard)), ROUNDING[wgrad_dy_rounding], seed, stream_id, 0)
    rc = lib().mx_linear_bwd(_ptr(dY), _ptr(X), _ptr(W), T, Kin, Nout, FORMATS[fmt], C.byref(o),
                             _ptr(dX) if need_dx else None, OUT[dX.dtype] if need_dx else 0,
                             _ptr(dW) if need_dw else None, OUT[dW.dtype] if need_dw else 0,
                             _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mx_linear_bwd")
    return dX, dW


def _bwd_opts(wgrad_hadamard, wgrad_dy_rounding, seed, stream_id):
    return _CBwdOpts(int(bool(wgrad_hadamard)), ROUNDING[wgrad_dy_rounding], seed, stream_id, 0)


def linear_fwd_save(X: torch.Tensor, W: torch.Tensor, fmt: str, out_dtype=torch.bfloat16,
                    wgrad_hadamard: bool = False, wgrad_dy_rounding: str = "rne", seed: int = 0,
                    stream_id: int = 0, x_amax: torch.Tensor | None = None, w_amax: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, saved: torch.Tensor | None = None,
                    out: torch.Tensor | None = None, stream=None):
    """Y = X W^T plus the layer's saved backward state (one read each of X and W).
    Returns (Y, saved); pass `saved` and the same backward options to linear_bwd_saved."""
    _on_gpu(X, W, x_amax, w_amax, workspace, saved, out)
    T, Kin = X.shape
    Nout = W.shape[0]
    ws = workspace if workspace is not None else torch.empty(workspace_bytes(T, Kin, Nout, fmt, "fwd"),
                                                             dtype=torch.uint8, device=X.device)
    sv = saved if saved is not None else torch.empty(saved_bytes(T, Kin, Nout, fmt), dtype=torch.uint8,
                                                     device=X.device)
    Y = out if out is not None else torch.empty((T, Nout), dtype=out_dtype, device=X.device)
    o = _bwd_opts(wgrad_hadamard, wgrad_dy_rounding, seed, stream_id)
    rc = lib().mx_linear_fwd_save(_ptr(X), _ptr(W), T, Kin, Nout, FORMATS[fmt], _ptr(x_amax), _ptr(w_amax),
                                  C.byref(o), _ptr(Y), OUT[Y.dtype], _ptr(ws), ws.numel(), _ptr(sv), sv.numel(),
                                  _stream(stream))
    _check(rc, "mx_linear_fwd_save")
    return Y, sv


def linear_bwd_saved(dY: torch.Tensor, saved: torch.Tensor, Kin: int, fmt: str,
                     wgrad_hadamard: bool = False, wgrad_dy_rounding: str = "rne", seed: int = 0,
                     stream_id: int = 0, dy_amax: torch.Tensor | None = None, dx_dtype=torch.bfloat16,
                     dw_dtype=torch.float32, need_dx: bool = True, need_dw: bool = True,
                     workspace: torch.Tensor | None = None, dX: torch.Tensor | None = None,
                     dW: torch.Tensor | None = None, stream=None):
    """dX = dY W and dW = dY^T X from the state linear_fwd_save kept (one read of dY)."""
    _on_gpu(dY, saved, dy_amax, workspace, dX, dW)
    T, Nout = dY.shape
    ws = workspace if workspace is not None else torch.empty(workspace_bytes(T, Kin, Nout, fmt, "bwd_saved"),
                                                             dtype=torch.uint8, device=dY.device)
    if need_dx and dX is None:
        dX = torch.empty((T, Kin), dtype=dx_dtype, device=dY.device)
    if need_dw and dW is None:
        dW = torch.empty((Nout, Kin), dtype=dw_dtype, device=dY.device)
    o = _bwd_opts(wgrad_hadamard, wgrad_dy_rounding, seed, stream_id)
    rc = lib().mx_linear_bwd_saved(_ptr(dY), T, Kin, Nout, FORMATS[fmt], _ptr(dy_amax), C.byref(o), _ptr(saved),
                                   saved.numel(), _ptr(dX) if need_dx else None, OUT[dX.dtype] if need_dx else 0,
                                   _ptr(dW) if need_dw else None, OUT[dW.dtype] if need_dw else 0,
                                   _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mx_linear_bwd_saved")
    return dX, dW


def last_device_status(stream=None) -> int:
    return int(lib().mx_last_device_status(_stream(stream)))


def selftest_bounded_wait(limit_ns: int, stream=None) -> int:
    return int(lib().mx_selftest_bounded_wait(int(limit_ns), _stream(stream)))


def launch_count() -> int:
    """Kernels the library has launched so far in this process."""
    return int(lib().mx_launch_count())


def debug_divide(v: torch.Tensor, d: torch.Tensor):
    """(fast, ieee) quotients of the quantizer's shared-divisor division."""
    _on_gpu(v, d)
    fast, ieee = torch.empty_like(v), torch.empty_like(v)
    _check(lib().mx_debug_divide(_ptr(v), _ptr(d), v.numel(), _ptr(fast), _ptr(ieee), _stream()),
           "mx_debug_divide")
    return fast, ieee


GEMM_VARIANTS = {"auto": 0, "cta_n128": 1, "cta_n256": 2, "pair": 3, "pair_ws": 4}


def set_gemm_variant(variant: str) -> None:
    """Force one GEMM kernel variant (tests and tuning); "auto" restores the default."""
    lib().mx_debug_set_gemm_variant(GEMM_VARIANTS[variant])


def last_gemm_variant() -> str:
    """The GEMM variant the most recent GEMM launch used (a GEMM_VARIANTS key)."""
    v = lib().mx_debug_last_gemm_variant()
    return {i: k for k, i in GEMM_VARIANTS.items()}.get(v, "none")
