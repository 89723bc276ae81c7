"""Pins for the oracle's CRC-32 (CPU only): the published check value of
CRC-32/ISO-HDLC, the bitwise definition against zlib's implementation, and
properties every CRC of this kind has (continuation, affinity over GF(2),
detection of any single-bit error)."""
import numpy as np

from oracle import crc32 as C


def test_check_value():
    assert C.crc32_bitwise(b"123456789") == 0xCBF43926
    assert C.crc32(b"123456789") == 0xCBF43926
    assert C.crc32_bitwise(b"") == 0 and C.crc32(b"") == 0


def test_bitwise_matches_zlib():
    rng = np.random.default_rng(0)
    for n in list(range(0, 40)) + [255, 256, 513]:
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert C.crc32_bitwise(data) == C.crc32(data), n


def test_continuation_and_affinity():
    rng = np.random.default_rng(1)
    a, b, c = (rng.integers(0, 256, 97, dtype=np.uint8) for _ in range(3))
    assert C.crc32_bitwise((a.tobytes() + b.tobytes())) == C.crc32_bitwise(b.tobytes(), C.crc32_bitwise(a.tobytes()))
    # CRC is affine over GF(2): an odd number of equal-length messages xor-combines
    assert C.crc32_bitwise((a ^ b ^ c).tobytes()) == (C.crc32_bitwise(a.tobytes()) ^ C.crc32_bitwise(b.tobytes())
                                                       ^ C.crc32_bitwise(c.tobytes()))


def test_single_bit_errors_are_detected():
    rng = np.random.default_rng(2)
    msg = rng.integers(0, 256, 64, dtype=np.uint8)
    ref = C.crc32(msg.tobytes())
    for bit in range(64 * 8):
        m = msg.copy()
        m[bit // 8] ^= np.uint8(1 << (bit % 8))
        assert C.crc32(m.tobytes()) != ref


def test_units_are_concatenated_ranges():
    rng = np.random.default_rng(3)
    a = rng.integers(0, 256, 5 * 48, dtype=np.uint8)
    b = rng.integers(0, 256, 5 * 8, dtype=np.uint8)
    got = C.crc32_units(a, 40, 48, 5, b, 6, 8)
    for u in range(5):
        want = C.crc32_bitwise(a[u * 48:u * 48 + 40].tobytes() + b[u * 8:u * 8 + 6].tobytes())
        assert got[u] == want
    assert np.array_equal(C.crc32_units(a, 48, 48, 5), [C.crc32(a[u * 48:(u + 1) * 48]) for u in range(5)])
