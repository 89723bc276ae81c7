"""Pins for the oracle's RoPE, strip-RoPE and relative rotation (CPU only):
closed forms, the SO(2) identity, composition, inversion, norm preservation,
complex multiplication for d = 2, and the pages' printed fp32 error."""
import numpy as np
import pytest

from oracle import rope
from oracle.numerics import round_to

PAIRINGS = [rope.INTERLEAVED, rope.HALF_SPLIT]


def test_inv_freq_closed_form():
    th = rope.inv_freq(128, 1e6)
    assert th[0] == 1.0
    assert np.allclose(th[1:] / th[:-1], 1e6 ** (-2 / 128), rtol=1e-13)
    assert np.isclose(th[-1], 1e6 ** (-126 / 128), rtol=1e-14)
    assert np.array_equal(rope.inv_freq(2, 1e4), [1.0])


def test_pair_convention():
    """The listing's convention pairs (0,1), (2,3), ...; half-split pairs (i, i+d/2)."""
    a, b = rope.pair_channels(8, rope.INTERLEAVED)
    assert list(a) == [0, 2, 4, 6] and list(b) == [1, 3, 5, 7]
    a, b = rope.pair_channels(8, rope.HALF_SPLIT)
    assert list(a) == [0, 1, 2, 3] and list(b) == [4, 5, 6, 7]


@pytest.mark.parametrize("pairing", PAIRINGS)
def test_unit_vector_closed_form(pairing):
    d, base, m = 16, 1e4, 37
    th = rope.inv_freq(d, base)
    a, b = rope.pair_channels(d, pairing)
    for i in range(d // 2):
        x = np.zeros((1, 1, d))
        x[0, 0, a[i]] = 1.0
        y = rope.apply_rope(x, [m], th, pairing)[0, 0]
        want = np.zeros(d)
        want[a[i]] = np.cos(m * th[i])
        want[b[i]] = np.sin(m * th[i])
        assert np.allclose(y, want, atol=1e-15)


def test_d2_matches_complex_multiplication():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 3, 2))
    pos = rng.integers(-5000, 5000, 50)
    y = rope.apply_rope(x, pos, rope.inv_freq(2, 1e4), rope.INTERLEAVED)
    z = (x[..., 0] + 1j * x[..., 1]) * np.exp(1j * pos.astype(float))[:, None]
    assert np.allclose(y[..., 0], z.real, atol=1e-12) and np.allclose(y[..., 1], z.imag, atol=1e-12)


@pytest.mark.parametrize("pairing", PAIRINGS)
@pytest.mark.parametrize("base", [1e4, 5e5, 1e6])
def test_so2_identity(pairing, base):
    """Rotating keys cached at m_old by delta-m gives RoPE at m_new = m_old + delta-m,
    including negative m_new."""
    rng = np.random.default_rng(1)
    d = 128
    th = rope.inv_freq(d, base)
    x = rng.standard_normal((64, 4, d))
    m_old = rng.integers(0, 40000, 64)
    dm = rng.integers(-50000, 50000, 64)
    lhs = rope.rotate_relative(rope.apply_rope(x, m_old, th, pairing), dm, th, pairing)
    rhs = rope.apply_rope(x, m_old + dm, th, pairing)
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(x)) * 10


@pytest.mark.parametrize("pairing", PAIRINGS)
def test_zero_delta_is_identity(pairing):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 2, 64))
    y = rope.rotate_relative(x, np.zeros(16), rope.inv_freq(64, 1e4), pairing)
    assert np.array_equal(y, x)


@pytest.mark.parametrize("pairing", PAIRINGS)
def test_composition_and_inverse_and_norm(pairing):
    rng = np.random.default_rng(3)
    d = 64
    th = rope.inv_freq(d, 5e5)
    x = rng.standard_normal((32, 2, d))
    d1, d2 = rng.integers(-9000, 9000, 32), rng.integers(-9000, 9000, 32)
    two = rope.rotate_relative(rope.rotate_relative(x, d1, th, pairing), d2, th, pairing)
    one = rope.rotate_relative(x, d1 + d2, th, pairing)
    assert np.max(np.abs(two - one)) < 1e-11
    pos = rng.integers(0, 100000, 32)
    assert np.max(np.abs(rope.strip_rope(rope.apply_rope(x, pos, th, pairing), pos, th, pairing) - x)) < 1e-12
    a, b = rope.pair_channels(d, pairing)
    y = rope.apply_rope(x, pos, th, pairing)
    assert np.allclose(x[..., a] ** 2 + x[..., b] ** 2, y[..., a] ** 2 + y[..., b] ** 2, rtol=1e-12)


def test_pages_fp32_shift_error(golden):
    """Moving fp32 post-RoPE keys from position 1024 to 8192 with an fp32
    rotation lands within 1e-6 of fresh RoPE at 8192; the pages print 4.77e-7."""
    rng = np.random.default_rng(4)
    d, base = 128, 1e4
    th = rope.inv_freq(d, base)
    x = rng.standard_normal((256, 8, d))
    a, b = rope.pair_channels(d, rope.INTERLEAVED)
    k_old = round_to(rope.apply_rope(x, np.full(256, 1024), th, rope.INTERLEAVED), "f32").astype(np.float32)
    ang = 7168 * th
    c = round_to(np.cos(ang), "f32").astype(np.float32)
    s = round_to(np.sin(ang), "f32").astype(np.float32)
    y = np.empty_like(k_old)
    y[..., a] = k_old[..., a] * c - k_old[..., b] * s
    y[..., b] = k_old[..., a] * s + k_old[..., b] * c
    ref = rope.apply_rope(x, np.full(256, 8192), th, rope.INTERLEAVED)
    err = np.max(np.abs(y.astype(np.float64) - ref))
    assert err <= 1e-6
    assert err >= golden["rope_shift_err_1024_to_8192"] / 8     # same order as printed
