"""The parity bars for fetched V, checked against the arithmetic that sets them.

The fetch dequantizes V as an fp32 product code x scale and converts it to
the output dtype; the oracle rounds the exact product once.  The two agree
bit for bit when the fp32 product is exact, and may differ by one ulp of a
16-bit output when it is not (the second rounding can cross a midpoint).
"""
import numpy as np
import pytest

from tests.bars import compare_v
from oracle.numerics import round_to


def _products(scale_fmt, n, seed):
    """Exact fp64 products of INT4 codes (+-1..7) and scales of `scale_fmt`."""
    r = np.random.default_rng(seed)
    s = round_to(r.uniform(1e-3, 1.0, n), scale_fmt)
    c = r.integers(1, 8, n) * r.choice([-1.0, 1.0], n)
    return c * s                      # at most 3 + 24 significant bits: exact in fp64


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_int4_f32_scales_round_twice(out):
    p = _products("f32", 400_000, 7)
    once = round_to(p, out)
    twice = round_to(round_to(p, "f32"), out)
    diff = once != twice
    assert diff.any()                 # the fp32 product is not always exact ...
    ok, exact = compare_v(twice, once, "int4", out, "f32")
    assert ok and not exact           # ... and the bar admits the second rounding
    ok16, _ = compare_v(twice, once, "int4", out, "f16")
    assert not ok16                   # the fp16-scale bar would not


@pytest.mark.parametrize("out", ["bf16", "f16", "f32"])
def test_int4_f16_scales_exact_in_f32(out):
    p = _products("f16", 400_000, 8)
    assert np.array_equal(round_to(p, "f32"), p)       # 3 + 11 bits fit in fp32
    once = round_to(p, out)
    ok, exact = compare_v(round_to(round_to(p, "f32"), out), once, "int4", out, "f16")
    assert ok and exact


def test_f32_output_is_one_rounding():
    p = _products("f32", 100_000, 9)
    g = round_to(p, "f32")
    assert compare_v(g, g, "int4", "f32", "f32") == (True, True)
    bumped = np.nextafter(g.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    assert not compare_v(bumped, g, "int4", "f32", "f32")[0]


def test_two_ulps_fail():
    p = _products("f32", 1000, 10)
    e = round_to(p, "bf16")
    g = e + 2.0 * np.abs(e) * 2.0 ** -7          # two bf16 ulps in the binade of e
    assert not compare_v(g, e, "int4", "bf16", "f32")[0]
    assert not compare_v(g, e, "fp8", "bf16")[0]
