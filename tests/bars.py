"""The parity bars, numpy only (used by the GPU tests in the test process and
by the oracle worker processes of the full-size checks, which import no
torch).

* fetched K: fp32 output within 2e-6 x the (token, head) row's max |k| of
  the oracle; fp16/bf16 output within 1 ulp of the larger of the two values,
  plus the same 2e-6 x row-max floor (below it the fp32 rotation's own
  rounding decides the last bit);
* fetched V: bit-exact, except where the fp32 dequantized value is itself a
  rounding and the output is fp16/bf16, which rounds it a second time
  (within 1 ulp): FP8-sourced V (either FP8 wire), and INT4 with fp32
  scales (a 3-bit code times a 24-bit scale can need 27 bits).  INT4 with
  fp16 scales needs at most 14 bits, so its products are exact and V is
  bit-exact in every output dtype.
"""
import numpy as np

from oracle.numerics import ulp

SENTINEL = -12288.0            # exact in fp32, fp16 and bf16; never a real output here
K_REL = 2e-6


def compare_k(g, e, fmt):
    """(ok, max |err|, bar at that element) for fetched K rows [..., d]."""
    rowmax = np.max(np.abs(e), axis=-1, keepdims=True)
    bar = K_REL * rowmax
    if fmt != "f32":
        bar = bar + np.maximum(ulp(g, fmt), ulp(e, fmt))
    err = np.abs(g - e)
    bar = np.broadcast_to(bar, err.shape)
    i = np.unravel_index(np.argmax(err - bar), err.shape) if err.size else ()
    return bool(np.all(err <= bar)), float(err.max(initial=0)), float(bar[i]) if err.size else 0.0


def compare_v(g, e, wire, fmt, scale_dtype="f16"):
    """(ok, exact) for fetched V values."""
    exact = bool(np.array_equal(g, e))
    rounded_twice = wire in ("fp8", "fp8_rows") or (wire == "int4" and scale_dtype == "f32")
    if rounded_twice and fmt != "f32":
        return bool(np.all(np.abs(g - e) <= np.maximum(ulp(g, fmt), ulp(e, fmt)))), exact
    return exact, exact
