"""GPU: the per-pair phasor of the sums on its own (fhd_test_phasor), against
fp64 sin and cos.

- Accurate mode (compensated reduced phase, accurate FMA-pipe polynomial):
  the error stays within one bound for every |k.x| up to 1e5 cycles, because
  each product is reduced on its own before the sum.
- The accurate polynomial against CUDA's sincospif on the same reduced
  arguments.
- Fast mode: the phase is one float32 FMA chain, reduced to t = p - rint(p)
  before the hardware sin/cos.  Its error is the chain's own rounding (a bound
  computed per pair) plus the hardware approximation on [-pi, pi], at every
  |k.x|: the approximation is never given a large argument ("Case study -
  iterative MRI reconstruction", section 17.3.5).  The fast polynomial share
  is checked the same way.
"""
import math

import numpy as np
import pytest

from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu

ACCURATE, FAST_MUFU, FAST_POLY, SINCOSPIF, ACCURATE_POLY_OF_T = 0, 1, 2, 3, 4
U = 2.0 ** -24  # float32 unit roundoff


@pytest.fixture(scope="module")
def lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    torch.cuda.set_device(0)
    return load()


@pytest.fixture(scope="module")
def pairs():
    """2^20 pairs: k components of magnitude 10^0 .. 10^5 cycles per FOV (a
    decade per sixth of the pairs), x components uniform in [-1/2, 1/2)."""
    rng = np.random.default_rng(60)
    n = 1 << 20
    mag = 10.0 ** np.repeat(np.arange(6), -(-n // 6))[:n]
    a = (rng.uniform(-1, 1, (3, n)) * mag).astype(np.float32)
    b = rng.uniform(-0.5, 0.5, (3, n)).astype(np.float32)
    return a, b


def run(lib, which, a, b):
    import torch

    t = [dev(v) for v in (*a, *b)]
    s = torch.empty_like(t[0])
    c = torch.empty_like(t[0])
    st = lib.fhd_test_phasor(which, t[0].numel(), *(v.data_ptr() for v in t), s.data_ptr(), c.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return s.cpu().numpy().astype(np.float64), c.cpu().numpy().astype(np.float64)


def exact(a, b):
    """sin, cos of 2 pi a.b in fp64 (the products of float32 values are exact in
    fp64; the argument is reduced in fp64 first)."""
    p = sum(a[i].astype(np.float64) * b[i].astype(np.float64) for i in range(3))
    t = p - np.rint(p)
    return np.sin(2 * math.pi * t), np.cos(2 * math.pi * t)


def chain_bound(a, b):
    """Rounding bound, in cycles, of p = fma(az, bz, fma(ay, by, ax*bx)) in
    float32: each of the three operations rounds its result once."""
    h1 = a[0].astype(np.float64) * b[0]
    h2 = h1 + a[1].astype(np.float64) * b[1]
    p = h2 + a[2].astype(np.float64) * b[2]
    return 1.01 * U * (np.abs(h1) + np.abs(h2) + np.abs(p))


def test_accurate_phasor_any_magnitude(lib, pairs):
    a, b = pairs
    s, c = run(lib, ACCURATE, a, b)
    es, ec = exact(a, b)
    err = np.maximum(np.abs(s - es), np.abs(c - ec))
    # phase within 1.8e-7 cycles (three fractions within 2^-25 each, two sums
    # of values below 1 and 1.5) plus the polynomial's 2.4e-7 (measured on a
    # dense grid; a little slack for arguments between its points)
    bound = 2 * math.pi * 1.8e-7 + 2.6e-7
    print(f"accurate phasor: max |error| {err.max():.3e} (bound {bound:.3e}), rms {np.sqrt(np.mean(err ** 2)):.3e}")
    assert err.max() <= bound
    # and independent of the magnitude: each decade of |k| within the same bound
    n6 = -(-err.size // 6)
    for d in range(6):
        assert err[d * n6:(d + 1) * n6].max() <= bound, d


def test_accurate_polynomial_against_sincospif(lib, pairs):
    a, b = pairs
    s_ref, c_ref = run(lib, SINCOSPIF, a, b)
    s, c = run(lib, ACCURATE_POLY_OF_T, a, b)
    diff = max(np.abs(s - s_ref).max(), np.abs(c - c_ref).max())
    print(f"accurate polynomial vs sincospif on the same t: max |difference| {diff:.3e}")
    assert diff <= 3.5e-7


@pytest.mark.parametrize("which,approx", [(FAST_MUFU, 2.0 ** -21.19 + 2.0e-7), (FAST_POLY, 8.0e-7)])
def test_fast_phasor_reduced(lib, pairs, which, approx):
    """|error| <= 2 pi (the FMA chain's rounding bound) + the sin/cos
    approximation's error on [-pi, pi] (hardware: at most 2^-21.19 for the
    cosine, 2^-21.41 for the sine, plus the rounding of 2 pi t; polynomial:
    its measured 7.6e-7), for |k.x| up to 1e5 cycles."""
    a, b = pairs
    s, c = run(lib, which, a, b)
    es, ec = exact(a, b)
    err = np.maximum(np.abs(s - es), np.abs(c - ec))
    allowed = 2 * math.pi * chain_bound(a, b) + approx
    worst = np.argmax(err / allowed)
    print(f"fast method {which}: worst error/allowed {err[worst] / allowed[worst]:.3f} "
          f"(|p| there {abs(np.dot(a[:, worst].astype(np.float64), b[:, worst])):.1f} cycles)")
    assert np.all(err <= allowed)
