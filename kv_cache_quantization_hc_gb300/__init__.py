"""GB300 (sm_103a) KV-cache wire codec with relative-RoPE fetch.

* ``hc``     - ctypes binding of libhc.so, the C ABI declared in include/hc.h
               (hc_encode_fp8, hc_encode_int4, hc_build_delta_sincos,
               hc_fetch_rotate_scatter);
* ``build``  - compiles libhc.so in-tree with nvcc for sm_103a;
* ``path``   - the hot path composed from the C-ABI calls on torch-owned
               device buffers (encode, table, fetch; the layer-streamed fetch).

The library is loaded on first use; a missing library raises.
"""
from . import hc  # noqa: F401
