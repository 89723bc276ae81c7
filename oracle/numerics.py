"""Round float64 values to narrower binary floating-point formats.

ORACLE (test infrastructure only; see the package docstring).

The method stores keys and values in fp32, fp16 or bf16 and the FP8 wire in
E4M3; every conversion on the path is IEEE round-to-nearest-even.  This module
restates that rounding from its definition (keep p significant bits, ties to
the even neighbour, gradual underflow below the smallest normal) so the rest of
the oracle can hold every value as an exact float64.

Pinned by tests against numpy's float32/float16 casts and torch's bfloat16
cast (library routines) and by brute force over neighbouring grid points.
"""
import numpy as np

# (significant bits p incl. the implicit one, smallest normal exponent emin,
#  largest finite value)
FORMATS = {
    "f32": (24, -126, float(np.finfo(np.float32).max)),
    "f16": (11, -14, 65504.0),
    "bf16": (8, -126, float((2.0 - 2.0 ** -7) * 2.0 ** 127)),
}


def round_to_precision(x, p, emin):
    """Round float64 ``x`` to ``p`` significant bits, ties to even.

    Exponents below ``emin`` keep the quantum ``2**(emin-p+1)`` (gradual
    underflow).  No overflow handling: the caller decides.  Signed zeros,
    infinities and NaNs pass through; a value that underflows to zero keeps
    its sign (that is what round-to-nearest-even does to a tiny negative).
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    m = np.isfinite(x) & (x != 0)
    if np.any(m):
        xm = x[m]
        _, e = np.frexp(xm)              # |xm| in [2**(e-1), 2**e)
        exp = np.maximum(e - 1, emin)     # exponent of the leading bit
        quantum = np.ldexp(1.0, exp - (p - 1))
        # xm / quantum is exact (division by a power of two, no underflow for
        # the formats used here); np.rint rounds half to even.
        out[m] = np.rint(xm / quantum) * quantum
    return out


def round_to(x, fmt):
    """Round float64 ``x`` to format ``fmt`` ('f32', 'f16', 'bf16'), RNE.

    Magnitudes that round above the largest finite value become +-inf, as an
    IEEE conversion does.
    """
    p, emin, fmax = FORMATS[fmt]
    r = round_to_precision(x, p, emin)
    big = np.isfinite(r) & (np.abs(r) > fmax)
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, r), r)
    return r


def ulp(x, fmt):
    """Spacing of format ``fmt`` at magnitude |x| (the quantum of |x|'s binade)."""
    p, emin, _ = FORMATS[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x == 0, 1.0, x))
    exp = np.where(x == 0, emin, np.maximum(e - 1, emin))
    return np.ldexp(1.0, exp - (p - 1))


def f32_div(a, b):
    """IEEE fp32 quotient a/b of fp32 operands (one rounding).

    Computed as the float32 division numpy performs in hardware (correctly
    rounded by IEEE 754).  Division by zero gives +-inf or NaN, as IEEE says.
    """
    a32 = np.asarray(a, dtype=np.float32)
    b32 = np.asarray(b, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        return (a32 / b32).astype(np.float64)
