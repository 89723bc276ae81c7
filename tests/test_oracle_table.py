"""Pins for the oracle's rotation table, oracle.paged.delta_sincos_table
(CPU only).

The table row of a delta-m holds (cos, sin)(delta-m * theta_i) with the
angle the fp64 product and each entry rounded once to fp32 ["HyperCache -
Distributed KV-cache quantization and relative RoPE reuse", "Core Design",
relative RoPE paragraph: the rotation is done in float32 with an error near
4.7e-7].  Every row is pinned by something other than numpy's cos/sin:

* arbitrary precision: mpmath evaluates cos and sin of the same fp64 angle
  with 200-bit arithmetic and rounds to 24 bits; every entry must be an fp32
  value within 1 fp32 ulp of that (numpy's fp64 routines may differ in the
  last fp64 bit, which moves the fp32 rounding with probability about 2^-29);
* the group law: the rows of delta-1 and delta-2, multiplied as complex
  numbers, give the row of delta-1 + delta-2 to fp32 accuracy; row(-delta)
  is the conjugate of row(delta); row(2) follows from row(1) by the double
  angle formulas; cos^2 + sin^2 = 1;
* the pages' printed error: keys cached in fp32 at position 1024 and turned
  to 8192 with the table's fp32 entries land within 1e-6 of fresh RoPE at
  8192 ("Example output" part B prints 4.77e-7).

``test_pins_reject_planted_mistakes`` plants plausible mistakes in copies of
the function (the angle's sign, an fp32 angle, cos and sin swapped, a shifted
frequency index, entries left unrounded) and checks that the pins catch each.
"""
import numpy as np
import pytest

from oracle import paged, rope
from oracle.numerics import round_to

mpmath = pytest.importorskip("mpmath")

BASES = (1e4, 5e5, 1e6)
D = 128
DELTAS = np.array([0, 1, -1, 2, -2, 7, 512, -512, 4096, 7168, -8192, 65535, 1048579,
                   2 ** 31 - 1, -2 ** 31], dtype=np.int64)


def _to_fp32(v):
    """An mpmath number rounded to 24 significant bits, nearest even."""
    with mpmath.workprec(24):
        return float(+v)


def _exact_row(dm, theta):
    """(cos, sin) of each fp64 angle dm * theta_i, by 200-bit arithmetic."""
    out = np.empty((len(theta), 2))
    with mpmath.workprec(200):
        for i, t in enumerate(theta):
            ang = mpmath.mpf(float(dm) * float(t))       # the fp64 product, as a number
            out[i, 0] = _to_fp32(mpmath.cos(ang))
            out[i, 1] = _to_fp32(mpmath.sin(ang))
    return out


def _fp32_ulp(v):
    return np.spacing(np.abs(np.asarray(v, dtype=np.float32))).astype(np.float64)


# ------------------------------------------------------------------ the pins
def pin_arbitrary_precision(table_fn):
    for base in BASES:
        th = rope.inv_freq(D, base)
        t = np.asarray(table_fn(DELTAS, th), dtype=np.float64)
        if t.shape != (len(DELTAS), D // 2, 2):
            return False
        if not np.array_equal(t.astype(np.float32).astype(np.float64), t):
            return False                                  # every entry is an fp32 value
        for n, dm in enumerate(DELTAS):
            want = _exact_row(dm, th)
            if not np.all(np.abs(t[n] - want) <= _fp32_ulp(want)):
                return False
    return True


def pin_group_law(table_fn):
    rng = np.random.default_rng(11)
    for base in BASES:
        th = rope.inv_freq(D, base)
        d1 = rng.integers(-50000, 50000, 40)
        d2 = rng.integers(-50000, 50000, 40)
        r1, r2, r12 = (np.asarray(table_fn(x, th), dtype=np.float64) for x in (d1, d2, d1 + d2))
        z = (r1[..., 0] + 1j * r1[..., 1]) * (r2[..., 0] + 1j * r2[..., 1])
        # each entry is within half an fp32 ulp (<= 2^-25) of its true value
        if np.max(np.abs(z - (r12[..., 0] + 1j * r12[..., 1]))) > 2.0 ** -22:
            return False
        pm = np.asarray(table_fn(np.array([1, -1, 2, -2, 4096, -4096]), th), dtype=np.float64)
        c1, s1 = pm[0, :, 0], pm[0, :, 1]
        if not (np.array_equal(pm[1, :, 0], c1) and np.array_equal(pm[1, :, 1], -s1)):
            return False                                  # cos is even, sin is odd
        if not (np.array_equal(pm[3], pm[2] * [1, -1]) and np.array_equal(pm[5], pm[4] * [1, -1])):
            return False
        if np.max(np.abs(pm[2, :, 0] - (2 * c1 * c1 - 1))) > 2.0 ** -21:
            return False                                  # cos 2t = 2 cos^2 t - 1
        if np.max(np.abs(pm[2, :, 1] - 2 * s1 * c1)) > 2.0 ** -21:
            return False                                  # sin 2t = 2 sin t cos t
        allr = np.asarray(table_fn(np.concatenate([d1, d2]), th), dtype=np.float64)
        if np.max(np.abs(allr[..., 0] ** 2 + allr[..., 1] ** 2 - 1)) > 2.0 ** -22:
            return False
    return True


def pages_shift_error(table_fn):
    """Max |error| of fp32 keys moved from 1024 to 8192 with the table's row,
    against fresh fp64 RoPE at 8192 (the pages' benchmark, part B)."""
    rng = np.random.default_rng(4)
    th = rope.inv_freq(D, 1e4)
    x = rng.standard_normal((256, 8, D))
    a, b = rope.pair_channels(D, rope.INTERLEAVED)
    k_old = round_to(rope.apply_rope(x, np.full(256, 1024), th, rope.INTERLEAVED), "f32").astype(np.float32)
    row = np.asarray(table_fn(np.array([8192 - 1024]), th), dtype=np.float64)[0].astype(np.float32)
    c, s = row[:, 0], row[:, 1]
    y = np.empty_like(k_old)
    y[..., a] = k_old[..., a] * c - k_old[..., b] * s
    y[..., b] = k_old[..., a] * s + k_old[..., b] * c
    ref = rope.apply_rope(x, np.full(256, 8192), th, rope.INTERLEAVED)
    return float(np.max(np.abs(y.astype(np.float64) - ref)))


def pin_pages_error(table_fn, printed=4.77e-7):
    err = pages_shift_error(table_fn)
    return printed / 8 <= err <= 1e-6


PINS = (pin_arbitrary_precision, pin_group_law, pin_pages_error)


# ------------------------------------------------------------------ tests
def test_table_matches_arbitrary_precision():
    assert pin_arbitrary_precision(paged.delta_sincos_table)


def test_table_group_law():
    assert pin_group_law(paged.delta_sincos_table)


def test_pages_fp32_shift_error(golden):
    """The pages print 4.77e-7 for 1024 -> 8192 in fp32; the oracle's table
    gives an error of the same order and within 1e-6."""
    err = pages_shift_error(paged.delta_sincos_table)
    assert err <= 1e-6
    assert err >= golden["rope_shift_err_1024_to_8192"] / 8
    assert pin_pages_error(paged.delta_sincos_table, golden["rope_shift_err_1024_to_8192"])


def test_zero_row_is_identity():
    t = paged.delta_sincos_table(np.array([0]), rope.inv_freq(D, 1e6))
    assert np.all(t[0, :, 0] == 1.0) and np.all(t[0, :, 1] == 0.0)


# planted mistakes (copies of the function; the oracle itself is untouched)
def _sign_flipped(dm, th):
    ang = -np.asarray(dm, np.float64)[:, None] * th[None, :]
    return np.stack([round_to(np.cos(ang), "f32"), round_to(np.sin(ang), "f32")], -1)


def _fp32_angle(dm, th):
    ang = (np.asarray(dm, np.float32)[:, None] * th.astype(np.float32)[None, :]).astype(np.float64)
    return np.stack([round_to(np.cos(ang), "f32"), round_to(np.sin(ang), "f32")], -1)


def _swapped(dm, th):
    return paged.delta_sincos_table(dm, th)[..., ::-1]


def _shifted_index(dm, th):
    return paged.delta_sincos_table(dm, np.roll(th, 1))


def _unrounded(dm, th):
    ang = np.asarray(dm, np.float64)[:, None] * th[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], -1)


MUTANTS = {"sign": (_sign_flipped, {pin_arbitrary_precision, pin_pages_error}),
           "fp32_angle": (_fp32_angle, {pin_arbitrary_precision, pin_group_law, pin_pages_error}),
           "swapped": (_swapped, {pin_arbitrary_precision, pin_group_law, pin_pages_error}),
           "shifted_index": (_shifted_index, {pin_arbitrary_precision, pin_pages_error}),
           "unrounded": (_unrounded, {pin_arbitrary_precision})}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistakes(name):
    fn, must_fail = MUTANTS[name]
    for pin in must_fail:
        assert not pin(fn), f"{pin.__name__} accepts the planted mistake {name!r}"
