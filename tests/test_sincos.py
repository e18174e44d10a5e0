"""The sine and cosine behind the sin/cos random features ("Kernel Feature
Maps", section 3 "Random Fourier Features") on the tensor-core path: the argument is
reduced by 2 pi in three parts and the fast hardware sincos takes the
remainder.  The reduction must hold up for large projections, so the device
values are compared with float64 sin and cos of the same fp32 arguments, up
to |x| ~ 4e5 (2^16 periods, where the exact product n p1 ends).

Bound: after the reduction the remainder carries at most a few fp32 roundings
of a value in [-pi, pi] (about 2.4e-7 each), and the hardware sincos has an
absolute error of about 2^-21.4 (3.6e-7) there, so 1e-6 leaves room while a
two-part reduction, which loses n * 1e-11 of the argument, fails it from
|x| ~ 1e5 on (n ~ 1.6e4)."""
import math

import numpy as np
import pytest

import favor_random_feature_gb300 as fv
from favor_random_feature_gb300 import build as fbuild

TOL = 1e-6


def _arguments():
    rng = np.random.default_rng(20261202)
    parts = [
        rng.uniform(-math.pi, math.pi, 4096),                       # already reduced
        rng.uniform(-64.0, 64.0, 4096),                             # typical projections
        np.sign(rng.standard_normal(8192)) * np.exp(rng.uniform(0.0, math.log(4.0e5), 8192)),
        np.arange(-2000, 2001) * (math.pi / 2),                     # zeros and extrema of sin, cos
        np.arange(-2000, 2001) * (math.pi / 2) + 1e-3,
        np.array([0.0, -0.0, 1e-30, -1e-30, 4.0e5, -4.0e5, 2 * math.pi * 65535]),
    ]
    return np.concatenate(parts).astype(np.float32)


def test_reduction_constants_sum_to_two_pi():
    """p1 + p2 + p3 (the fp32 constants the kernels hold) equals 2 pi to
    ~3e-19; p1 has 8 significant bits.  Checked with exact rationals."""
    from fractions import Fraction
    p1, p2, p3 = (np.float32(6.28125), np.float32(1.935307169e-3), np.float32(1.025337627e-11))
    two_pi = Fraction("6.28318530717958647692528676655900576839433879875")
    resid = two_pi - Fraction(float(p1)) - Fraction(float(p2)) - Fraction(float(p3))
    assert abs(resid) < Fraction(1, 10 ** 18)
    assert Fraction(float(p1)) * 32 == 201            # 201 < 2^8
    assert 201 * 65535 < 2 ** 24                      # n p1 exact for |n| < 2^16


@pytest.mark.gpu
def test_sincos_against_float64():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fbuild.build()
    x_host = _arguments()
    n = x_host.size
    x = torch.from_numpy(x_host).cuda()
    s = torch.empty_like(x)
    c = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    assert fv.favor_check_sincos(x, s, c, n, stream) == fv.FAVOR_OK
    assert fv.favor_get_device_status(stream) == fv.FAVOR_OK
    xd = x_host.astype(np.float64)
    es = np.abs(s.cpu().numpy().astype(np.float64) - np.sin(xd))
    ec = np.abs(c.cpu().numpy().astype(np.float64) - np.cos(xd))
    worst = int(np.argmax(np.maximum(es, ec)))
    assert max(es.max(), ec.max()) <= TOL, (float(x_host[worst]), float(es[worst]), float(ec[worst]))
    # empty input: nothing launched
    assert fv.favor_check_sincos(x, s, c, 0, stream) == fv.FAVOR_OK


def test_sincos_rejects_bad_arguments():
    fbuild.build()
    assert fv.favor_check_sincos(None, None, None, -1, None) == fv.FAVOR_ERR_INVALID_ARG
    assert fv.favor_check_sincos(None, None, None, 0, None) == fv.FAVOR_OK
