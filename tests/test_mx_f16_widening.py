"""CPU checks of the two number-format facts the MXFP8 tensor-core decode rests on (numpy emulation of
the format arithmetic, not of the kernel):

* a layer's E4M3 codes times 2^(S - 127 + c), c = 134 - Smax, are exact f16 values for every scale
  code S within 22 binades of the layer's largest Smax, and the bound is tight (23 binades lose the
  smallest subnormal code);
* the three-plane f16 split of a batch value, x ~ 2^16 p0 + 2^5 p1 + 2^-6 p2 with each plane the f16
  rounding of what the planes before it left, is within 2^-33 |x| + 2^-31 of x below 2^32.

The codes' values come from the oracle's E4M3 decoder, which tests/test_oracle_mx.py pins to the
format's definition."""
import numpy as np
import pytest

import oracle

CODES = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
VALUES = oracle.e4m3_to_float(CODES)  # f64, exact


def _f16_exact(v: np.ndarray) -> np.ndarray:
    return v.astype(np.float16).astype(np.float64) == v


@pytest.mark.parametrize("smax", [60, 100, 115, 127, 142, 200, 254])
def test_widened_weights_exact_within_22_binades(smax):
    c = 134 - smax
    for s in range(max(0, smax - 22), smax + 1):
        w = VALUES * 2.0 ** (s - 127 + c)
        assert np.all(_f16_exact(w)), (smax, s)
        assert np.abs(w).max() <= 65504.0
        nz = np.abs(w[w != 0])
        assert nz.min() >= 2.0 ** -24


def test_widening_bound_is_tight():
    # 23 binades below the largest scale, the smallest subnormal code (2^-9) lands on 2^-25
    smax = 120
    w = VALUES * 2.0 ** (smax - 23 - 127 + 134 - smax)
    assert not np.all(_f16_exact(w))


def test_power_of_two_factor_is_an_f16():
    # the converters multiply by 2^(S - 127 + c) = 2^(S - Smax + 7), k in [-15, 7]: every such power
    # of two is an f16 (2^-15 as a subnormal)
    for k in range(-15, 8):
        assert _f16_exact(np.array([2.0 ** k]))[0]


def _split3(x: np.ndarray):
    f = np.float32
    x = x.astype(np.float32)
    p0 = (x * f(2.0 ** -16)).astype(np.float16)
    r0 = (x - p0.astype(np.float32) * f(2.0 ** 16)).astype(np.float32)
    p1 = (r0 * f(2.0 ** -5)).astype(np.float16)
    r1 = (r0 - p1.astype(np.float32) * f(2.0 ** 5)).astype(np.float32)
    p2 = (r1 * f(2.0 ** 6)).astype(np.float16)
    return p0, p1, p2


def test_three_plane_split_error_bound():
    rng = np.random.default_rng(5)
    n = 200_000
    x = (rng.standard_normal(n) * 2.0 ** rng.uniform(-40, 31, n)).astype(np.float32)
    x = x[np.abs(x) < 2.0 ** 32]
    x = np.concatenate([x, np.float32([0.0, -0.0, 1.0, -1.0, 2.0 ** -149, 65504.0, 2.0 ** 31, -(2.0 ** 31)])])
    with np.errstate(over="ignore"):
        p0, p1, p2 = _split3(x)
    assert np.isfinite(p0).all() and np.isfinite(p1).all() and np.isfinite(p2).all()
    got = p0.astype(np.float64) * 2.0 ** 16 + p1.astype(np.float64) * 2.0 ** 5 + p2.astype(np.float64) * 2.0 ** -6
    xd = x.astype(np.float64)
    assert np.all(np.abs(got - xd) <= 2.0 ** -33 * np.abs(xd) + 2.0 ** -31)


def test_three_plane_split_overflows_at_2_32():
    with np.errstate(over="ignore"):
        p0, _, _ = _split3(np.float32([2.0 ** 32, -(2.0 ** 33)]))
    assert np.isinf(p0.astype(np.float64)).all()
