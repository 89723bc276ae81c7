"""Pins for the oracle's RoPE, strip-RoPE and relative rotation (CPU only):
closed forms, the SO(2) identity, composition, inversion, norm preservation,
and the 2x2 rotation matrix for d = 2.  The pages' printed fp32 shift error is
pinned through the oracle's rotation table in test_oracle_table.py."""
import numpy as np
import pytest

from oracle import rope

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


def test_d2_matches_rotation_matrix():
    """d = 2 (theta_0 = 1): each token's pair is the 2x2 rotation matrix
    [[cos m, -sin m], [sin m, cos m]] times the column (x0, x1), multiplied
    out by numpy's matmul."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 3, 2))
    pos = rng.integers(-5000, 5000, 50).astype(float)
    y = rope.apply_rope(x, pos, rope.inv_freq(2, 1e4), rope.INTERLEAVED)
    c, s = np.cos(pos), np.sin(pos)
    R = np.stack([np.stack([c, -s], -1), np.stack([s, c], -1)], -2)      # [T, 2, 2]
    want = np.matmul(R[:, None], x[..., None])[..., 0]                  # [T, 3, 2]
    assert np.allclose(y, want, atol=1e-12, rtol=0)
    back = rope.strip_rope(y, pos, rope.inv_freq(2, 1e4), rope.INTERLEAVED)
    assert np.allclose(back, np.matmul(np.swapaxes(R, 1, 2)[:, None], y[..., None])[..., 0],
                       atol=1e-12, rtol=0)


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
