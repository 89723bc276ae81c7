"""FP8 E4M3 encode/decode from the format's definition.

ORACLE (test infrastructure only; see the package docstring).

The wire format is named "FP8 (E4M3)" ["HyperCache - Distributed KV-cache
quantization and relative RoPE reuse", "Example output", part B].  The pages do
not define the format; the definition followed here is the OCP 8-bit floating
point specification (OFP8), E4M3 variant:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 is subnormal: value = (m / 8) * 2**-6;
* otherwise value = (1 + m / 8) * 2**(e - 7); the largest finite magnitude is
  S.1111.110 = 448;
* no infinities; S.1111.111 is NaN.

Encoding (what the wire stores) rounds to nearest with ties to the even
mantissa, saturates finite magnitudes above 448 to 448 ("satfinite"), and keeps
the sign bit, so -0 and negative values that round to zero encode as 0x80.
"""
import numpy as np

from .numerics import round_to_precision

E4M3_MAX = 448.0
_P = 4          # significant bits incl. the implicit one
_EMIN = -6      # exponent of the smallest normal, 2**-6
_SUB_Q = 2.0 ** -9   # subnormal quantum (1/8 * 2**-6)


def e4m3_value(code):
    """Value of one E4M3 byte (float; NaN for S.1111.111)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table():
    """All 256 decoded values, indexed by code."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(q):
    """Encode finite values q (float64 holding fp32 values) to E4M3 bytes.

    Round to nearest, ties to even mantissa, saturate to +-448, keep the sign.
    NaN inputs are outside the method's domain (finite keys and values) and
    encode to the NaN byte.
    """
    q = np.asarray(q, dtype=np.float64)
    neg = np.signbit(q)
    a = np.abs(q)
    r = round_to_precision(np.where(np.isfinite(a), a, 0.0), _P, _EMIN)
    r = np.minimum(r, E4M3_MAX)          # saturate (RNE past 448 would give 480)
    r = np.where(np.isinf(a), E4M3_MAX, r)
    sub = r < 2.0 ** _EMIN
    # subnormal or zero: field e = 0, m = r / 2**-9 (0..7)
    m_sub = np.rint(r / _SUB_Q).astype(np.int64)
    # normal: r = (1 + m/8) * 2**E
    _, ex = np.frexp(np.where(sub, 1.0, r))
    E = ex - 1
    m_nrm = np.rint((np.where(sub, 1.0, r) / np.ldexp(1.0, E) - 1.0) * 8.0).astype(np.int64)
    field_e = np.where(sub, 0, E + 7)
    field_m = np.where(sub, m_sub, m_nrm)
    code = (field_e << 3) | field_m
    code = np.where(neg, code | 0x80, code)
    code = np.where(np.isnan(q), 0x7F, code)
    return code.astype(np.uint8)


def e4m3_decode(codes):
    """Decode E4M3 bytes to float64 values (exact)."""
    return e4m3_table()[np.asarray(codes, dtype=np.uint8)]
