"""Rotary position embedding, its inverse, and the relative rotation by delta-m.

ORACLE (test infrastructure only; see the package docstring).

Conventions (pages):
* theta_i = base ** (-2 i / d), i = 0 .. d/2-1, and the pair (x_2i, x_2i+1) is
  rotated by the angle m * theta_i:  r1 = x1 cos - x2 sin,  r2 = x1 sin + x2 cos
  ["Module 13: KV handoff", code listing module13.py, rope_cache / apply_rope].
* strip-RoPE is the transposed rotation: r1 = x1 cos + x2 sin,
  r2 = -x1 sin + x2 cos [same listing, strip_rope].
* Reusing a block cached at m_old at the offset m_new rotates every post-RoPE
  key pair by delta-m = m_new - m_old, because R(m_new theta) =
  R(delta-m theta) R(m_old theta) in SO(2) ["HyperCache - Distributed KV-cache
  quantization and relative RoPE reuse", "Core Design", relative RoPE
  paragraph].  Values are not rotated.

Pairing: the listing pairs interleaved channels; "half-split" pairs channel i
with channel i + d/2 (the layout of the Qwen3/Llama checkpoints the workload
shapes are named after).  Both are selectable.

Everything is float64.  Angles are formed as the fp64 product m * theta_i and
cos/sin are numpy's fp64 routines.
"""
import numpy as np

INTERLEAVED = "interleaved"
HALF_SPLIT = "half_split"


def inv_freq(d_head, base):
    """theta_i = base ** (-2 i / d_head) in float64, i = 0 .. d_head/2 - 1."""
    if d_head % 2:
        raise ValueError("d_head must be even")
    i = np.arange(d_head // 2, dtype=np.float64)
    return np.power(np.float64(base), -(2.0 * i) / d_head)


def pair_channels(d_head, pairing):
    """Channel indices (first, second) of the d/2 rotation pairs."""
    h = d_head // 2
    if pairing == INTERLEAVED:
        return np.arange(0, d_head, 2), np.arange(1, d_head, 2)
    if pairing == HALF_SPLIT:
        return np.arange(h), np.arange(h, d_head)
    raise ValueError(f"unknown pairing {pairing!r}")


def _angles(pos, theta):
    """Angle table [T, d/2] = pos[t] * theta[i] (fp64 product)."""
    pos = np.asarray(pos, dtype=np.float64)
    return pos[:, None] * np.asarray(theta, dtype=np.float64)[None, :]


def apply_rope(x, pos, theta, pairing):
    """Rotate every pair of x [T, H, d] by pos[t] * theta_i (RoPE at pos)."""
    x = np.asarray(x, dtype=np.float64)
    a, b = pair_channels(x.shape[-1], pairing)
    ang = _angles(pos, theta)[:, None, :]          # [T, 1, d/2]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., a], x[..., b]
    out = np.empty_like(x)
    out[..., a] = x1 * c - x2 * s
    out[..., b] = x1 * s + x2 * c
    return out


def strip_rope(x, pos, theta, pairing):
    """Undo RoPE at pos: rotate every pair of x [T, H, d] by -pos[t] * theta_i,
    written as the transposed rotation."""
    x = np.asarray(x, dtype=np.float64)
    a, b = pair_channels(x.shape[-1], pairing)
    ang = _angles(pos, theta)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., a], x[..., b]
    out = np.empty_like(x)
    out[..., a] = x1 * c + x2 * s
    out[..., b] = -x1 * s + x2 * c
    return out


def rotate_relative(k, delta_m, theta, pairing):
    """Move post-RoPE keys k [T, H, d] from m_old to m_old + delta_m[t].

    The SO(2) identity turns this into one rotation of each pair by
    delta_m[t] * theta_i; no knowledge of m_old is needed.
    """
    return apply_rope(k, delta_m, theta, pairing)
