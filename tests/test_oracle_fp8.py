"""Pins for the oracle's E4M3 codec (CPU only): the format's definition, brute
force against every finite magnitude, and torch's float8_e4m3fn cast."""
import numpy as np
import torch

from oracle import fp8


def test_decode_table_landmarks():
    t = fp8.e4m3_table()
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9                 # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9             # largest subnormal
    assert t[0x08] == 2.0 ** -6                 # smallest normal
    assert t[0x38] == 1.0                       # exponent field 7 = bias
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = t[np.isfinite(t)]
    assert finite.size == 254
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)             # codes 0x00..0x7E strictly increasing


def test_decode_matches_torch_float8():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_decode(codes), ref)


def _brute(q):
    """Nearest of the 127 finite non-negative magnitudes, ties to even code,
    saturating, sign applied separately."""
    mags = fp8.e4m3_table()[:0x7F]
    a = min(abs(q), 448.0)
    d = np.abs(mags - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
    if np.signbit(q):
        code |= 0x80
    return code


def _test_set():
    mags = fp8.e4m3_table()[:0x7F]
    mids = (mags[:-1] + mags[1:]) / 2
    vals = []
    for m in np.concatenate([mids, mags]):
        m32 = np.float32(m)
        for k in (-2, -1, 0, 1, 2):
            vals.append(float(np.nextafter(m32, np.float32(np.inf * np.sign(k))) if k else m32))
            if abs(k) == 2:
                v = m32
                for _ in range(2):
                    v = np.nextafter(v, np.float32(np.inf * np.sign(k)))
                vals.append(float(v))
    hi = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    f = hi.view(np.float32).astype(np.float64)
    vals += list(f[np.isfinite(f)])
    vals += list(np.linspace(448, 480, 65))
    vals = np.array(vals)
    return np.concatenate([vals, -vals])


def test_encode_brute_force():
    qs = _test_set()
    got = fp8.e4m3_encode(qs)
    want = np.array([_brute(q) for q in qs], dtype=np.uint8)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (qs[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_encode_matches_torch_in_range():
    qs = _test_set()
    qs = qs[np.abs(qs) <= 448].astype(np.float32)
    ref = torch.from_numpy(qs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(qs.astype(np.float64)), ref)


def test_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)
    assert list(fp8.e4m3_encode(np.array([464.0, 480.0, 1e30, np.inf]))) == [0x7E] * 4
    assert list(fp8.e4m3_encode(np.array([-464.0, -1e30]))) == [0xFE] * 2
    # sign is kept through underflow
    assert list(fp8.e4m3_encode(np.array([-0.0, -1e-10, 1e-10, 2.0 ** -10]))) == [0x80, 0x80, 0x00, 0x00]
    assert fp8.e4m3_encode(np.array([3 * 2.0 ** -10]))[0] == 0x02   # tie 1.5 q -> even m=2
