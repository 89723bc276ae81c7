"""Pins for the oracle's rounding helpers (CPU only).

Each helper is checked against something other than itself: numpy's and
torch's hardware casts, exact rational arithmetic, and brute force over the
neighbouring grid points.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import numerics


def _samples(rng, n):
    mant = rng.uniform(-2, 2, n)
    exps = rng.integers(-140, 130, n)
    x = np.ldexp(mant, exps)
    return np.concatenate([x, [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24,
                               2.0 ** -25, 3 * 2.0 ** -26, 1e-45, -1e-45, 3.4e38]])


def test_f32_matches_numpy_cast():
    rng = np.random.default_rng(0)
    x = _samples(rng, 200_000)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).astype(np.float64)
    got = numerics.round_to(x, "f32")
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_f16_matches_numpy_cast():
    rng = np.random.default_rng(1)
    x = np.ldexp(rng.uniform(-2, 2, 200_000), rng.integers(-30, 18, 200_000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    got = numerics.round_to(x, "f16")
    assert np.array_equal(got, ref)


def test_bf16_matches_torch_cast_on_fp32_inputs():
    rng = np.random.default_rng(2)
    x = _samples(rng, 200_000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = numerics.round_to(x.astype(np.float64), "bf16")
    assert np.array_equal(got, ref)


def _exact_rne(v, p, emin):
    """Brute force: the two grid neighbours of v in (p, emin), pick the nearer,
    ties to the even significand."""
    v = Fraction(v)
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = emin
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    while e > emin and Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (e - (p - 1))
    lo = (a // q) * q
    hi = lo + q
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / q) % 2 == 0 else hi
    return r if v > 0 else -r


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16"])
def test_brute_force_neighbours(fmt):
    p, emin, _ = numerics.FORMATS[fmt]
    rng = np.random.default_rng(3)
    xs = list(np.ldexp(rng.uniform(-2, 2, 300), rng.integers(emin - 5, 10, 300)))
    # exact ties: midpoints between adjacent grid values
    for k in range(40):
        q = 2.0 ** (int(rng.integers(emin, 5)) - (p - 1))
        xs.append((int(rng.integers(1 << (p - 1), 1 << p)) + 0.5) * q)
    for x in xs:
        assert numerics.round_to(np.array([x]), fmt)[0] == float(_exact_rne(x, p, emin)), (fmt, x)


def test_f32_div_is_correctly_rounded():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(3000).astype(np.float32) * np.float32(3)
    b = np.abs(rng.standard_normal(3000).astype(np.float32)) / np.float32(448)
    got = numerics.f32_div(a, b)
    for ai, bi, gi in zip(a, b, got):
        exact = Fraction(float(ai)) / Fraction(float(bi))
        assert Fraction(float(gi)) == _exact_rne(exact, 24, -126)


def test_ulp():
    assert numerics.ulp(1.0, "bf16") == 2.0 ** -7
    assert numerics.ulp(1.5, "f32") == 2.0 ** -23
    assert numerics.ulp(0.0, "f16") == 2.0 ** -24
    assert numerics.ulp(-3.0, "f16") == 2.0 ** -9
