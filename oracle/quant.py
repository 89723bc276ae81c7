"""Group quantizers: FP8 E4M3 with one scale per group, symmetric INT4 per group.

ORACLE (test infrastructure only; see the package docstring).

The pages say blocks are compressed before they leave L1 and print the two
formats and their ratios: "FP8 (E4M3) Wire Quantization: 1.97x" and
"INT4 (Grouped) L3 Disk: 3.88x" ["HyperCache - Distributed KV-cache
quantization and relative RoPE reuse", "Core Design" compression paragraph and
"Example output", part B].  They do not print the scale rule; the reading
implemented here (one per group, absmax-based, symmetric) is:

FP8:  s = fp32(amax / 448);  q = fp32(x / s);  code = E4M3(q), RNE, satfinite.
INT4: s32 = fp32(amax / 7);  s = fp16_rne(s32) when scales are stored as fp16,
      else s32;  q = fp32(x / s) with the STORED scale;
      code = clamp(round_half_even(q), -7, 7), a 4-bit two's-complement nibble,
      even channel in the low nibble.

Both divisions are single IEEE fp32 divisions.  A group whose scale is zero
(amax = 0, or an fp16 scale that underflows) stores scale 0 and all-zero codes.
Elements outside ``valid`` (the padding rows of a ragged block) are excluded
from amax and get code 0.

Parity unpinned: the pages' FP8 cosine similarity of 0.999979 is not
reproduced by a direct round trip of Gaussian keys (about 0.9997 for E4M3); it
is reported as context only.  The INT4 cosine (0.993258) and both compression
ratios are pinned in the tests.
"""
import numpy as np

from .fp8 import E4M3_MAX, e4m3_encode, e4m3_decode
from .numerics import f32_div, round_to


def _amax(x, valid):
    a = np.abs(np.asarray(x, dtype=np.float64))
    if valid is not None:
        a = np.where(valid, a, 0.0)
    return a.max(axis=-1, keepdims=True)


def fp8_quantize(x, valid=None, scale_dtype="f32"):
    """Quantize groups along the last axis of x (fp32-representable values).

    Returns (codes uint8 with x's shape, scales float64 with shape x.shape[:-1]).
    """
    x = np.asarray(x, dtype=np.float64)
    amax = _amax(x, valid)
    s = f32_div(amax, E4M3_MAX)
    if scale_dtype == "f16":
        s = round_to(s, "f16")
    elif scale_dtype != "f32":
        raise ValueError(scale_dtype)
    q = f32_div(x, s)
    codes = e4m3_encode(np.where(s != 0, q, 0.0))
    codes = np.where(s != 0, codes, 0).astype(np.uint8)
    if valid is not None:
        codes = np.where(valid, codes, 0).astype(np.uint8)
    return codes, s[..., 0]


def fp8_dequantize(codes, scales):
    """Exact products code_value * scale (float64; both factors are exact)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def int4_quantize(x, valid=None, scale_dtype="f16"):
    """Quantize groups along the last axis of x to signed ints in [-7, 7].

    Returns (ints int8 with x's shape, scales float64 with shape x.shape[:-1]).
    """
    x = np.asarray(x, dtype=np.float64)
    amax = _amax(x, valid)
    s = f32_div(amax, 7.0)
    if scale_dtype == "f16":
        s = round_to(s, "f16")
    elif scale_dtype != "f32":
        raise ValueError(scale_dtype)
    q = f32_div(x, s)
    with np.errstate(invalid="ignore"):
        r = np.clip(np.rint(np.where(s != 0, q, 0.0)), -7, 7)
    r = np.where(s != 0, r, 0)
    if valid is not None:
        r = np.where(valid, r, 0)
    return r.astype(np.int8), s[..., 0]


def int4_dequantize(ints, scales):
    return np.asarray(ints, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def int4_pack(ints):
    """Pack ints [..., n] (n even) into bytes [..., n/2]: channel 2k in the low
    nibble, channel 2k+1 in the high nibble, 4-bit two's complement."""
    v = np.asarray(ints, dtype=np.int64) & 0xF
    return (v[..., 0::2] | (v[..., 1::2] << 4)).astype(np.uint8)


def int4_unpack(packed):
    """Inverse of int4_pack: bytes [..., n/2] -> ints int8 [..., n]."""
    b = np.asarray(packed, dtype=np.int64)
    lo, hi = b & 0xF, (b >> 4) & 0xF
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int64)
    out[..., 0::2], out[..., 1::2] = lo, hi
    out = np.where(out >= 8, out - 16, out)
    return out.astype(np.int8)


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
