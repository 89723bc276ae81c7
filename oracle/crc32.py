"""CRC-32 of encoded payloads (tamper detection of cached blocks).

ORACLE (test infrastructure only; see the package docstring).

The pages store INT4 blocks on disk "(.hckv + CRC32)" and list CRC32 tamper
detection among their tests ["HyperCache - Distributed KV-cache quantization
and relative RoPE reuse", "Example output" part B and the test-suite
paragraph].  They do not name the CRC variant.  The reading taken is the
common CRC-32 of zlib, PNG and Ethernet (CRC-32/ISO-HDLC): generator
polynomial 0x04C11DB7 processed bit-reflected (0xEDB88320), register
initialised to 0xFFFFFFFF, input and output reflected, result xor 0xFFFFFFFF.
Its published check value is crc32(b"123456789") = 0xCBF43926.

``crc32_bitwise`` is that definition, one bit at a time (small inputs only);
``crc32`` is zlib's implementation of the same function, used as a library
step for large inputs.  A "unit" is the concatenation of one range of a
buffer ``a`` and, optionally, one range of a buffer ``b`` (for example a
block's codes followed by its scales).
"""
import zlib

import numpy as np

POLY_REFLECTED = 0xEDB88320


def crc32_bitwise(data, crc=0):
    """CRC-32 of ``data`` (bytes-like), continuing from a previous result."""
    reg = crc ^ 0xFFFFFFFF
    for byte in bytes(data):
        reg ^= byte
        for _ in range(8):
            reg = (reg >> 1) ^ (POLY_REFLECTED if reg & 1 else 0)
    return reg ^ 0xFFFFFFFF


def crc32(data, crc=0):
    return zlib.crc32(bytes(data), crc) & 0xFFFFFFFF


def crc32_units(a, a_bytes, a_stride, n_units, b=None, b_bytes=0, b_stride=0):
    """CRC-32 of unit u = a[u*a_stride : u*a_stride + a_bytes] followed by
    b[u*b_stride : u*b_stride + b_bytes], for u < n_units (uint32 array)."""
    a = np.frombuffer(np.ascontiguousarray(a).tobytes(), dtype=np.uint8)
    bb = None if b is None else np.frombuffer(np.ascontiguousarray(b).tobytes(), dtype=np.uint8)
    out = np.empty(n_units, dtype=np.uint32)
    for u in range(n_units):
        c = crc32(a[u * a_stride:u * a_stride + a_bytes])
        if bb is not None and b_bytes:
            c = crc32(bb[u * b_stride:u * b_stride + b_bytes], c)
        out[u] = c
    return out
