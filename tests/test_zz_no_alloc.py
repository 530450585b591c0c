"""mx_linear_fwd_noalloc, the forward for callers that cannot allocate device
memory (allocator callbacks, fully pre-reserved processes, plugin interfaces
that pass only inputs and outputs): it must give what mx_linear_fwd gives,
call after call, while its quantized operands live in the library's fixed
device array.  Collected last so a stop-at-first-failure run has already run
every other test."""
import ctypes as C

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-3  # the relative GEMM tolerance of the other parity tests


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4", "moss", "nvfp4_local"])
def test_noalloc_forward_matches_linear_fwd_twice(mx, fmt):
    T, Kin, Nout = 512, 1024, 768
    X = workloads.draw("student_t3", (T, Kin), 91).cuda()
    W = workloads.draw("normal", (Nout, Kin), 92, 0.02).cuda()
    ref = mx.linear_fwd(X, W, fmt, out_dtype=torch.float32)
    L = mx.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        Y = torch.full((T, Nout), float("nan"), dtype=torch.float32, device="cuda")
        rc = L.mx_linear_fwd_noalloc(C.c_void_p(X.data_ptr()), C.c_void_p(W.data_ptr()), T, Kin, Nout,
                                     mx.FORMATS[fmt], C.c_void_p(Y.data_ptr()), 0, stream)
        assert rc == mx.MX_OK, mx.strerror(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(Y).all()
        err = (Y.double() - ref.double()).abs()
        assert (err <= TOL * ref.double().abs().max()).all()
        assert torch.equal(Y, ref)  # same kernels on the same inputs
    assert mx.last_device_status() == mx.MX_OK


def test_noalloc_rejects_sizes_beyond_its_array(mx):
    X = torch.zeros(8192, 4096, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.linear_fwd_noalloc(X, W, "mxfp8")
    assert e.value.code == mx.MX_ERR_WORKSPACE
