"""Rotary position embedding, its inverse, and the relative rotation by delta-m.

ORACLE (test infrastructure only; see the package docstring).

What the pages fix:
* theta_i = base ** (-2 i / d), i = 0 .. d/2-1, and RoPE at position m turns
  the i-th channel pair by the angle m * theta_i, the first channel of the
  pair taking the cosine part ["Module 13: KV handoff", code listing
  module13.py, rope_cache / apply_rope]; strip-RoPE turns it back
  [same listing, strip_rope].
* Each channel pair is a complex coordinate, and RoPE multiplies it by the
  unit phase exp(i m theta_i).  Reusing a block cached at m_old at the
  offset m_new multiplies every post-RoPE key pair by exp(i delta-m theta_i),
  delta-m = m_new - m_old, since phases multiply by adding their angles:
  R(m_new theta) = R(delta-m theta) R(m_old theta) in SO(2) ["HyperCache -
  Distributed KV-cache quantization and relative RoPE reuse", "Core Design",
  relative RoPE paragraph].  Values are not rotated.

This module writes RoPE as that complex product: the pair (x_a, x_b) is the
number x_a + i x_b, the phase is numpy's complex exponential of the fp64
angle m * theta_i, and the product's real and imaginary parts go back to
channels a and b.  strip-RoPE multiplies by the conjugate phase.

Pairing: the listing pairs interleaved channels; "half-split" pairs channel i
with channel i + d/2 (the layout of the Qwen3/Llama checkpoints the workload
shapes are named after).  Both are selectable.

Everything is float64 (complex128).
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


def _phase(pos, theta, sign):
    """Unit phases exp(sign * i * pos[t] * theta_k), shape [T, 1, d/2]; the
    angle is the fp64 product pos[t] * theta_k."""
    ang = np.asarray(pos, dtype=np.float64)[:, None] * np.asarray(theta, dtype=np.float64)[None, :]
    return np.exp(1j * (sign * ang))[:, None, :]


def _turn(x, phase, pairing):
    """Multiply every channel pair of x [T, H, d], read as a complex number,
    by ``phase`` and return the real array of the products."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    first, second = pair_channels(d, pairing)
    z = (x[..., first] + 1j * x[..., second]) * phase
    # real parts belong to the first channels, imaginary parts to the second
    order = np.argsort(np.concatenate([first, second]))
    return np.concatenate([z.real, z.imag], axis=-1)[..., order]


def apply_rope(x, pos, theta, pairing):
    """RoPE at pos: every pair of x [T, H, d] times exp(i pos[t] theta_k)."""
    return _turn(x, _phase(pos, theta, 1.0), pairing)


def strip_rope(x, pos, theta, pairing):
    """Undo RoPE at pos: every pair of x [T, H, d] times exp(-i pos[t] theta_k)."""
    return _turn(x, _phase(pos, theta, -1.0), pairing)


def rotate_relative(k, delta_m, theta, pairing):
    """Move post-RoPE keys k [T, H, d] from m_old to m_old + delta_m[t].

    The phases multiply, so this is one more multiplication of each pair by
    exp(i delta_m[t] theta_k); no knowledge of m_old is needed.
    """
    return apply_rope(k, delta_m, theta, pairing)
