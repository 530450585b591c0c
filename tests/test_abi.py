"""The C-ABI library builds, loads, and exports every function include/mx.h declares.

These run without a GPU: only size queries, error strings and the no-device /
argument-error paths are called (nothing is launched).
"""
import ctypes as C
import os
import re

import pytest
import torch

import fp4_precision_gemms_gb300 as mx
from conftest import gpu_available

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mx_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    mx.build()
    return mx.lib()


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mx.EXPORTED)


def test_size_queries(lib):
    f = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2, "moss": 3}
    assert lib.mx_codes_bytes(f["mxfp8"], 256, 256) == 65536
    assert lib.mx_codes_bytes(f["mxfp4"], 256, 256) == 32768
    assert lib.mx_codes_bytes(f["nvfp4"], 3, 33) == 0  # odd K cannot be packed
    # scale tiles: 128 rows x 4 blocks per 512 bytes, padded
    assert lib.mx_sf_bytes(f["mxfp8"], 256, 256) == 2 * 2 * 512
    assert lib.mx_sf_bytes(f["nvfp4"], 130, 64) == 2 * 1 * 512
    assert lib.mx_sf_bytes(f["moss"], 11008, 4096) == 86 * 32 * 512
    assert lib.mx_sf_bytes(f["mxfp8"], 8, 48) == 0  # K not a multiple of the block
    assert lib.mx_sf_bytes(9, 8, 64) == 0
    assert lib.mx_linear_workspace_bytes(8192, 4096, 6144, f["nvfp4"], 0) > 8192 * 2048 + 6144 * 2048


def test_strerror(lib):
    for code in range(8):
        s = lib.mx_strerror(code).decode()
        assert s and s != "unknown status"
    assert lib.mx_strerror(99).decode() == "unknown status"


@pytest.mark.skipif(gpu_available(), reason="checks the no-GPU error path")
def test_calls_without_a_gpu_fail_loudly(lib):
    t = mx._CTensor()
    rc = lib.mx_quantize(None, 0, 0, 0, 0, 0, 32, 0, 0, 0, 0, 0, None, C.byref(t), None)
    assert rc == mx.MX_ERR_NO_DEVICE
    assert lib.mx_gemm(C.byref(t), C.byref(t), 1.0, None, 0, 0, None) == mx.MX_ERR_NO_DEVICE
    amax = C.c_float(0.0)
    assert lib.mx_gemm_amax(C.byref(t), C.byref(t), 1.0, None, 0, 0, C.byref(amax), None) == mx.MX_ERR_NO_DEVICE
    # a missing amax word is an argument error, found before the device is looked at
    assert lib.mx_gemm_amax(C.byref(t), C.byref(t), 1.0, None, 0, 0, None, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_last_device_status(None) == mx.MX_ERR_NO_DEVICE
    with pytest.raises(mx.MXError):
        mx.quantize(torch.zeros(32, 32, dtype=torch.bfloat16), "mxfp8")


def test_size_queries_agree_with_the_oracle_layout(lib):
    """The library's buffer sizes against the oracle's independently written
    layout (512-byte tiles of 128 rows x 4 scale blocks) on many shapes, and the
    tensor-scale entry counts against the format table."""
    import oracle as orc

    fmts = {"mxfp8": (0, 32, 1.0), "mxfp4": (1, 32, 0.5), "nvfp4": (2, 16, 0.5), "moss": (3, 32, 1.0),
            "nvfp4_local": (4, 16, 0.5)}
    for name, (f, block, code_bytes) in fmts.items():
        for rows in (1, 31, 127, 128, 129, 300, 4096, 14336):
            for k in (block, 2 * block, 4 * block, 5 * block, 256, 4160, 14336):
                assert lib.mx_codes_bytes(f, rows, k) == int(rows * k * code_bytes), (name, rows, k)
                assert lib.mx_sf_bytes(f, rows, k) == orc.sf_bytes(rows, k // block), (name, rows, k)
            want = {"nvfp4": 1, "moss": 1, "nvfp4_local": max(1, -(-rows // 128))}.get(name, 0)
            assert lib.mx_scale_count(f, rows) == want, (name, rows)


def test_host_memory_is_refused_before_the_library_is_called():
    """The library reads and writes device memory only: operands, outputs and
    workspaces in host memory are refused by the binding (no launch happens)."""
    q = mx.MXTensor("mxfp8", 128, 64, "cpu")  # allocated in host memory
    with pytest.raises(mx.MXError):
        mx.gemm(q, q)
    with pytest.raises(mx.MXError):
        mx.dequantize(q)
    x = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(mx.MXError):
        mx.linear_fwd(x, x, "mxfp8", out=torch.zeros(64, 64, dtype=torch.bfloat16))


def test_saved_state_sizes(lib):
    """The saved backward state is the colwise operands X^T [Kin, T] and W^T
    [Kin, Nout]; the saved-state backward's workspace is dY and dY^T.  Each
    operand is its codes, scale bytes and two scalar arrays, each padded."""
    def operand(f, rows, k):
        pad = lambda v, a: -(-v // a) * a  # noqa: E731
        n = max(1, lib.mx_scale_count(f, rows))
        return pad(lib.mx_codes_bytes(f, rows, k), 256) + pad(lib.mx_sf_bytes(f, rows, k), 256) + 2 * pad(4 * n, 128)
    for f in range(5):
        for T, Kin, Nout in ((8192, 4096, 6144), (256, 512, 384), (4096, 14336, 4096)):
            assert lib.mx_linear_saved_bytes(T, Kin, Nout, f) == operand(f, Kin, T) + operand(f, Kin, Nout)
            assert lib.mx_linear_workspace_bytes(T, Kin, Nout, f, 2) == operand(f, T, Nout) + operand(f, Nout, T)
            assert lib.mx_linear_workspace_bytes(T, Kin, Nout, f, 3) == 0
    assert lib.mx_linear_saved_bytes(256, 256, 256, 9) == 0
