"""Pins for the oracle's token selection (CPU only): the norm against
numpy.linalg.norm and a closed form, the selection against constructed
inputs whose answer is known (including exact ties), and the default k."""
import numpy as np

from oracle import blend


def test_default_k():
    assert blend.default_k(1408) == 212      # ceil(211.2)
    assert blend.default_k(20) == 3
    assert blend.default_k(100) == 15        # 15.0 exactly: no extra token
    assert blend.default_k(1) == 1


def test_drift_is_the_l2_norm():
    r = np.random.default_rng(0)
    a = r.standard_normal((3, 50, 64))
    b = r.standard_normal((3, 50, 64))
    assert np.allclose(blend.drift(a, b), np.linalg.norm(b - a, axis=-1), rtol=1e-14, atol=0)
    # closed form: one non-zero difference per token
    c = np.zeros((1, 8, 16))
    f = c.copy()
    f[0, np.arange(8), np.arange(8)] = np.arange(8) - 3.5
    assert np.array_equal(blend.drift(c, f)[0], np.abs(np.arange(8) - 3.5))


def test_selection_of_constructed_drifts():
    T, D = 40, 32
    r = np.random.default_rng(1)
    base = r.standard_normal((1, T, D))
    mags = r.permutation(T).astype(np.float64) + 1.0          # distinct drifts 1..T
    fresh = base.copy()
    fresh[0, :, 5] += mags
    dr, sel = blend.select(base, fresh, 7)
    want = np.sort(np.argsort(-mags)[:7])
    assert np.array_equal(sel[0], want)
    assert np.allclose(dr[0], mags, rtol=1e-12)


def test_ties_go_to_the_lower_index():
    v = np.array([1.0, 5.0, 3.0, 5.0, 5.0, 0.0, 3.0])
    assert np.array_equal(blend.select_topk(v, 2), [1, 3])
    assert np.array_equal(blend.select_topk(v, 4), [1, 2, 3, 4])
    assert np.array_equal(blend.select_topk(v, 5), [1, 2, 3, 4, 6])
    assert np.array_equal(blend.select_topk(v, 7), np.arange(7))
