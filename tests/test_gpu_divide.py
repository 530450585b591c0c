"""The quantizer divides many elements by one shared divisor (the MOSS tensor
scale, the NVFP4 block scale times the tensor scale) using the divisor's
correctly rounded reciprocal plus residual corrections.  It must return exactly
what CUDA's IEEE division returns, bit for bit, including signed zeros."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import fp4_precision_gemms_gb300 as m
    m.build()
    return m


def same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def check(mx, v, d):
    fast, ieee = mx.debug_divide(v.contiguous(), d.contiguous())
    torch.cuda.synchronize()
    bad = (fast.view(torch.int32) != ieee.view(torch.int32)).nonzero()
    assert bad.numel() == 0, (f"{bad.numel()} quotients differ; first v={v.flatten()[bad[0]].item()!r} "
                              f"d={d.flatten()[bad[0]].item()!r}")
    # the IEEE reference is also what numpy's float32 division gives
    with np.errstate(all="ignore"):
        ref = (v.cpu().numpy() / d.cpu().numpy()).astype(np.float32)
    assert np.array_equal(ieee.cpu().numpy().view(np.int32), ref.view(np.int32))


def test_every_bf16_numerator_against_many_divisors(mx):
    v = workloads.all_bf16_patterns().float().cuda()
    g = torch.Generator().manual_seed(5)
    ds = torch.cat([torch.exp2(torch.empty(48).uniform_(-40, 40, generator=g)),
                    torch.tensor([1.0, 3.0, 448.0 / 2688.0, 1.0 / 6.0, 2.0 ** -100, 2.0 ** 100, 2.0 ** -120,
                                  2.0 ** 120, 1.9999999, 1.0000001, 0.7, 1e-30, 3e30])]).float()
    for dv in ds:
        check(mx, v, torch.full_like(v, float(dv)))


def test_random_pairs(mx):
    g = torch.Generator(device="cuda").manual_seed(9)
    n = 1 << 22
    bits = torch.randint(0, 0x7F800000, (n,), generator=g, device="cuda", dtype=torch.int64)  # finite
    sign = torch.randint(0, 2, (n,), generator=g, device="cuda", dtype=torch.int64) << 31
    bits = torch.where(sign != 0, bits - 2 ** 31, bits).to(torch.int32)  # sign bit set where sign != 0
    v = bits.view(torch.float32)
    d = torch.exp2(torch.empty(n, device="cuda").uniform_(-110, 110, generator=g)) * \
        (1 + torch.rand(n, device="cuda", generator=g))
    check(mx, v, d)


def test_quotients_at_e2m1_rounding_thresholds(mx):
    """Numerators whose exact quotient sits within a few ulps of an E2M1 RNE
    midpoint, where a wrongly rounded quotient would change the code."""
    g = torch.Generator().manual_seed(3)
    d = torch.exp2(torch.empty(4096).uniform_(-20, 10, generator=g)).float()
    vs = []
    for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 448.0):
        base = (torch.tensor(t, dtype=torch.float64) * d.double()).float().view(torch.int32)
        for k in range(-3, 4):  # k ulps away from the rounded product t * d
            vs.append((base + k).view(torch.float32))
    v = torch.cat(vs)
    dd = d.repeat(len(vs))
    check(mx, v.cuda(), dd.cuda())
    check(mx, (-v).cuda(), dd.cuda())
