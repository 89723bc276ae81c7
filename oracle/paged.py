"""Evict (gather + encode) and fetch (decode + relative rotate + scatter) over a
paged KV buffer.

ORACLE (test infrastructure only; see the package docstring).

Pages: keys are taken post-RoPE "directly from the engine's PagedAttention
buffer" at m_old and every pair is rotated by delta-m on fetch; blocks are
compressed before leaving L1; the fetched frame is dequantized and rotated "on
the fly" ["HyperCache - Distributed KV-cache quantization and relative RoPE
reuse", "Core Design" relative-RoPE and compression paragraphs, "Example
output" part B, "Live TCP Socket Fetch + On-The-Fly RoPE"].  Blocks hold 16 or
64 tokens ["Core Design", item 1].

The pages give no memory layout; the readings implemented here:

* paged buffer (one for K, one for V): [L, num_slots, B, H, d], token-major
  inside a block;
* block j of a call lives in slot src_slots[j] (encode) or goes to slot
  dst_slots[j] (fetch); one table entry per block, shared by all layers and by
  K and V;
* wire: [L, NB, 2, H, B, d] (kv = 0 is K, 1 is V) of E4M3 bytes with one fp32
  scale per (layer, block, kv, head); INT4 packs [L, NB, 2, H, B, d/2] bytes
  with one scale per (layer, block, kv, head, token, group of g channels);
* the row-scaled FP8 wire ("pages layout"): the same E4M3 bytes with one
  scale per (layer, block, kv, head, token) row of d channels, fp16 by
  default - the granularity whose sizes reproduce the printed FP8 frame
  (133,120 payload bytes for 131,072 fp16 values, 1.97x);
* n_valid[j] tokens of block j are real; the rest are padding: excluded from
  amax, encoded as 0 (INT4 scale 0), never written by fetch;
* one delta-m per block (a block moves as a unit).

Arrays are float64 and hold values exactly representable in the stated
formats.  All functions return new arrays and leave their inputs unchanged.
"""
import numpy as np

from . import quant
from .numerics import round_to
from .rope import rotate_relative


def _valid_rows(n_valid, nb, B):
    nv = np.full(nb, B, dtype=np.int64) if n_valid is None else np.asarray(n_valid, dtype=np.int64)
    return np.arange(B)[None, :] < nv[:, None]            # [NB, B]


def gather_slabs(paged_k, paged_v, src_slots):
    """Wire-ordered copy of the cached blocks: [L, NB, 2, H, B, d]."""
    src = np.asarray(src_slots, dtype=np.int64)
    k = np.asarray(paged_k, dtype=np.float64)[:, src]      # [L, NB, B, H, d]
    v = np.asarray(paged_v, dtype=np.float64)[:, src]
    kv = np.stack([k, v], axis=2)                          # [L, NB, 2, B, H, d]
    return kv.transpose(0, 1, 2, 4, 3, 5).copy()           # [L, NB, 2, H, B, d]


def encode_fp8(paged_k, paged_v, src_slots, n_valid=None):
    """FP8 E4M3 encode, one fp32 scale per (layer, block, kv, head) slab of B x d.

    Returns codes uint8 [L, NB, 2, H, B, d] and scales float64 [L, NB, 2, H].
    """
    slabs = gather_slabs(paged_k, paged_v, src_slots)
    L, NB, _, H, B, d = slabs.shape
    valid = _valid_rows(n_valid, NB, B)[None, :, None, None, :, None]
    valid = np.broadcast_to(valid, slabs.shape)
    flat = slabs.reshape(L, NB, 2, H, B * d)
    codes, scales = quant.fp8_quantize(flat, valid.reshape(flat.shape), "f32")
    return codes.reshape(slabs.shape), scales


def encode_int4(paged_k, paged_v, src_slots, n_valid=None, group=32, scale_dtype="f16"):
    """Grouped INT4 encode, one scale per (layer, block, kv, head, token, group).

    Returns packed codes uint8 [L, NB, 2, H, B, d/2] and scales float64
    [L, NB, 2, H, B, d/group].
    """
    slabs = gather_slabs(paged_k, paged_v, src_slots)
    L, NB, _, H, B, d = slabs.shape
    if d % group:
        raise ValueError("group must divide d_head")
    g = slabs.reshape(L, NB, 2, H, B, d // group, group)
    valid = _valid_rows(n_valid, NB, B)[None, :, None, None, :, None, None]
    valid = np.broadcast_to(valid, g.shape)
    ints, scales = quant.int4_quantize(g, valid, scale_dtype)
    ints = ints.reshape(L, NB, 2, H, B, d)
    return quant.int4_pack(ints), scales


def encode_fp8_rows(paged_k, paged_v, src_slots, n_valid=None, scale_dtype="f16"):
    """FP8 E4M3 encode, one scale per (layer, block, kv, head, token) row of d.

    s = fp32(amax / 448), rounded to fp16 when scale_dtype is "f16"; the codes
    use the stored scale (a scale that overflows fp16 is +inf and gives codes
    of x / inf = +-0).  Padding rows get scale 0 and codes 0.

    Returns codes uint8 [L, NB, 2, H, B, d] and scales float64 [L, NB, 2, H, B].
    """
    slabs = gather_slabs(paged_k, paged_v, src_slots)
    L, NB, _, H, B, d = slabs.shape
    valid = _valid_rows(n_valid, NB, B)[None, :, None, None, :, None]
    valid = np.broadcast_to(valid, slabs.shape)
    with np.errstate(over="ignore"):
        return quant.fp8_quantize(slabs, valid, scale_dtype)


def decode_fp8_rows(codes, scales):
    """[L, NB, 2, H, B, d] exact dequantized values (code * stored row scale;
    a row whose fp16 scale overflowed to +inf decodes to 0 * inf = NaN)."""
    with np.errstate(invalid="ignore"):
        return quant.fp8_dequantize(codes, scales)


def decode_fp8(codes, scales):
    """[L, NB, 2, H, B, d] exact dequantized values."""
    codes = np.asarray(codes)
    L, NB, _, H, B, d = codes.shape
    flat = codes.reshape(L, NB, 2, H, B * d)
    return quant.fp8_dequantize(flat, scales).reshape(codes.shape)


def decode_int4(codes, scales, group=32):
    """[L, NB, 2, H, B, d] exact dequantized values (code * stored scale)."""
    ints = quant.int4_unpack(codes)
    L, NB, _, H, B, d = ints.shape
    g = ints.reshape(L, NB, 2, H, B, d // group, group)
    return quant.int4_dequantize(g, scales).reshape(ints.shape)


def delta_sincos_table(delta_m, theta):
    """[n, d/2, 2] table of (cos, sin)(delta_m[n] * theta_i): fp64 angle and
    fp64 cos/sin, each rounded once to fp32."""
    ang = np.asarray(delta_m, dtype=np.float64)[:, None] * np.asarray(theta, dtype=np.float64)[None, :]
    return np.stack([round_to(np.cos(ang), "f32"), round_to(np.sin(ang), "f32")], axis=-1)


def fetch_rotate_scatter(values, delta_m, theta, pairing, dst_slots, out_k, out_v,
                         out_fmt, n_valid=None):
    """Rotate the K half of ``values`` [L, NB, 2, H, B, d] by delta_m[j] per
    block (exact fp64 angles), leave V as is, round to ``out_fmt`` and write
    the valid token rows of block j to slot dst_slots[j] of copies of
    out_k / out_v [L, num_slots, B, H, d].  Unwritten slots and padding rows
    keep their previous contents.
    """
    vals = np.asarray(values, dtype=np.float64)
    L, NB, _, H, B, d = vals.shape
    dm = np.asarray(delta_m, dtype=np.int64)
    new_k = np.array(out_k, dtype=np.float64, copy=True)
    new_v = np.array(out_v, dtype=np.float64, copy=True)
    dst = np.asarray(dst_slots, dtype=np.int64)
    if len(set(dst.tolist())) != len(dst):
        raise ValueError("destination slots must be distinct")
    nv = np.full(NB, B, dtype=np.int64) if n_valid is None else np.asarray(n_valid, dtype=np.int64)
    for j in range(NB):
        n = int(nv[j])
        k = vals[:, j, 0].transpose(0, 2, 1, 3)            # [L, B, H, d]
        v = vals[:, j, 1].transpose(0, 2, 1, 3)
        for layer in range(L):
            kr = rotate_relative(k[layer, :n], np.full(n, dm[j]), theta, pairing)
            new_k[layer, dst[j], :n] = round_to(kr, out_fmt)
            new_v[layer, dst[j], :n] = round_to(v[layer, :n], out_fmt)
    return new_k, new_v
