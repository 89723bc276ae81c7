"""Byte accounting: KV-cache size and wire-buffer sizes with their scales.

ORACLE (test infrastructure only; see the package docstring).

* KV bytes = 2 * L * H_kv * d_head * n_ctx * b ["Module 13: KV handoff",
  section 1 "Arithmetic", KV-bytes formula; the checklist repeats it as
  144 KiB/token for the 36 x 8 x 128 fp16 shape].
* Compression ratio = source bytes / (code bytes + scale bytes), scales
  counted ["HyperCache - Distributed KV-cache quantization and relative RoPE
  reuse", "Example output", part B: 1.97x FP8, 3.88x INT4].
"""


def kv_bytes(L, H_kv, d_head, n_ctx, b):
    """Bytes of a K+V cache: 2 * L * H_kv * d_head * n_ctx * b (b may be 0.5)."""
    return 2 * L * H_kv * d_head * n_ctx * b


def wire_bytes(n_elems, code_bits, n_scales, scale_bytes):
    """Bytes of an encoded buffer: packed codes plus stored scales."""
    return n_elems * code_bits // 8 + n_scales * scale_bytes


def compression_ratio(n_elems, src_bytes_per_elem, code_bits, n_scales, scale_bytes):
    return (n_elems * src_bytes_per_elem) / wire_bytes(n_elems, code_bits, n_scales, scale_bytes)
