"""ctypes binding of libhc.so: the C-ABI calls under the same names.

Argument marshalling only: every call here converts tensors to device
addresses, fills the descriptor struct, passes the stream and turns a negative
status into an exception.  All work runs in the library's CUDA kernels.  If
libhc.so is missing the first call raises; there is no other code path.
"""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhc.so")

HC_OK, HC_ERR_INVALID_ARG, HC_ERR_UNSUPPORTED, HC_ERR_CUDA = 0, -1, -2, -3
HC_F32, HC_F16, HC_BF16 = 0, 1, 2
HC_PAIR_INTERLEAVED, HC_PAIR_HALF_SPLIT = 0, 1
HC_WIRE_FP8, HC_WIRE_INT4, HC_WIRE_RAW, HC_WIRE_FP8_ROWS = 0, 1, 2, 3
HC_DEVERR_SLOT, HC_DEVERR_DELTA, HC_DEVERR_NVALID = 1, 2, 4

DTYPE_NAMES = {"f32": HC_F32, "f16": HC_F16, "bf16": HC_BF16}
PAIRING_NAMES = {"interleaved": HC_PAIR_INTERLEAVED, "half_split": HC_PAIR_HALF_SPLIT}


class HCError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn} returned {status_string(status)}" + (f" ({detail})" if detail else ""))


class hc_paged_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("d_head", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("slot_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64)]


_LIB = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32


def lib():
    """Load libhc.so once; raise if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`"
                " (the CUDA path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        desc_p = ctypes.POINTER(hc_paged_desc)
        L.hc_encode_fp8.argtypes = [_P, _P, desc_p, _P, _P, _I32, _P, _P, _P, _P]
        L.hc_encode_int4.argtypes = [_P, _P, desc_p, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P]
        L.hc_encode_fp8_rows.argtypes = [_P, _P, desc_p, _P, _P, _I32, _I32, _P, _P, _P, _P]
        L.hc_encode_fp8_crc.argtypes = [_P, _P, desc_p, _P, _P, _I32, _P, _P, _P, _P, _P]
        L.hc_build_delta_sincos.argtypes = [_P, _I32, _I32, ctypes.c_double, _P, _P, _P]
        L.hc_fetch_rotate_scatter.argtypes = [_I32, _P, _P, _I32, _I32, _P, _P, _I32, _I32, _P, _P,
                                              _I32, _P, _P, desc_p, _P, _P]
        _I64 = ctypes.c_int64
        L.hc_crc32.argtypes = [_P, _I64, _I64, _P, _I64, _I64, _I32, _P, _P]
        L.hc_drift_select.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I64, _I64, _I32, _P, _P, _P]
        L.hc_tenant_key.argtypes = [_P, _I32, ctypes.c_char_p, _P]
        L.hc_block_digests.argtypes = [_P, _I64, _I32, _P, _I32, _P, _P]
        for fn in ("hc_encode_fp8", "hc_encode_fp8_crc", "hc_encode_int4", "hc_encode_fp8_rows",
                   "hc_build_delta_sincos",
                   "hc_fetch_rotate_scatter", "hc_crc32", "hc_drift_select", "hc_tenant_key",
                   "hc_block_digests"):
            getattr(L, fn).restype = ctypes.c_int
        L.hc_status_string.argtypes = [_I32]
        L.hc_status_string.restype = ctypes.c_char_p
        L.hc_last_cuda_error.argtypes = []
        L.hc_last_cuda_error.restype = ctypes.c_char_p
        L.hc_version.argtypes = []
        L.hc_version.restype = ctypes.c_int32
        L.hc_selection_size.argtypes = [_I32]
        L.hc_selection_size.restype = ctypes.c_int32
        _LIB = L
    return _LIB


# ------------------------------------------------------------- marshalling
def _ptr(x):
    """Device/host address of a tensor, an int address, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _dptr(x, name):
    """Address of a device buffer: like _ptr, but a torch tensor must live on
    a CUDA device (the kernels dereference these pointers; a host tensor
    would make them fault)."""
    if x is not None and not isinstance(x, int) and not getattr(x, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor (or a device address)")
    return _ptr(x)


def _avail(x):
    """Bytes reachable from a tensor's data pointer (None for a raw address
    or NULL, which are not checked)."""
    if x is None or isinstance(x, int):
        return None
    return x.untyped_storage().nbytes() - x.storage_offset() * x.element_size()


def _need(x, nbytes, name):
    """Refuse a tensor smaller than the bytes the call will address."""
    a = _avail(x)
    if a is not None and a < nbytes:
        raise ValueError(f"{name} holds {a} bytes; the call addresses {nbytes}")


_ES = {HC_F32: 4, HC_F16: 2, HC_BF16: 2}


def _pool_bytes(desc):
    """Bytes a call addresses in a paged pool described by `desc`."""
    last = ((desc.n_layers - 1) * desc.layer_stride + (desc.num_slots - 1) * desc.slot_stride
            + desc.block_size * desc.n_kv_heads * desc.d_head)
    return last * _ES.get(desc.dtype, 1)


def _wire_bytes(desc, n_blocks, wire, group, scale_dtype):
    """(codes bytes, scales bytes) of the wire of a call on pools like `desc`."""
    cs, cdt, ss = wire_shapes(desc.n_layers, n_blocks, desc.n_kv_heads, desc.block_size,
                              desc.d_head, wire, group)
    n = 1
    for v in cs:
        n *= v
    codes = n * (_ES.get(desc.dtype, 1) if cdt == "paged" else 1)
    if ss is None:
        return codes, 0
    m = 1
    for v in ss:
        m *= v
    return codes, m * (4 if wire == HC_WIRE_FP8 or scale_dtype == HC_F32 else 2)


def _sizes_apply(desc, n_blocks, wire, group=32):
    """True for a call the C layer would accept on its descriptor, wire and
    group: only then are buffer sizes checked here, so that a malformed
    call still gets the C layer's own status."""
    return (n_blocks > 0 and desc.dtype in _ES and desc.d_head in (64, 128)
            and desc.block_size in (16, 32, 64, 128) and desc.n_layers >= 1
            and desc.num_slots >= 1 and desc.n_kv_heads >= 1 and desc.slot_stride >= 0
            and desc.layer_stride >= 0
            and wire in (HC_WIRE_FP8, HC_WIRE_INT4, HC_WIRE_RAW, HC_WIRE_FP8_ROWS)
            and (wire != HC_WIRE_INT4 or (group in (32, 64, 128) and group <= desc.d_head)))


def _check_encode(desc, paged_k, paged_v, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  wire, group=32, scale_dtype=HC_F16, crc=None):
    if not _sizes_apply(desc, n_blocks, wire, group):
        return
    pool = _pool_bytes(desc)
    _need(paged_k, pool, "paged_k")
    _need(paged_v, pool, "paged_v")
    _need(src_slots, 4 * n_blocks, "src_slots")
    _need(n_valid, 4 * n_blocks, "n_valid")
    cb, sb = _wire_bytes(desc, n_blocks, wire, group, scale_dtype)
    _need(codes, cb, "codes")
    _need(scales, sb, "scales")
    _need(err_flag, 4, "err_flag")
    _need(crc, 4 * desc.n_layers * n_blocks * 2 * desc.n_kv_heads, "crc")


def _stream(s):
    """cudaStream_t of a torch stream; None means torch's current stream."""
    if isinstance(s, int):
        return s
    import torch
    if s is None:
        s = torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn, status):
    if status != HC_OK:
        detail = lib().hc_last_cuda_error().decode() if status == HC_ERR_CUDA else ""
        raise HCError(fn, status, detail)


def status_string(status):
    return lib().hc_status_string(status).decode()


def hc_version():
    return lib().hc_version()


def paged_desc(pool, dtype=None, n_layers=None, layer_stride=None, slot_stride=None):
    """Descriptor of a pool tensor shaped [L, num_slots, B, H, d] (or
    [num_slots, B, H, d] for one layer).  Strides are taken from the tensor."""
    if pool.dim() == 4:
        pool = pool.unsqueeze(0)
    L, S, B, H, d = pool.shape
    if pool.stride(4) != 1 or pool.stride(3) != d or pool.stride(2) != H * d:
        raise ValueError("each slot must be a contiguous [B, H, d] block")
    if dtype is None:
        dtype = {"torch.float32": HC_F32, "torch.float16": HC_F16,
                 "torch.bfloat16": HC_BF16}[str(pool.dtype)]
    return hc_paged_desc(n_layers if n_layers is not None else L, H, d, B, S, dtype,
                         slot_stride if slot_stride is not None else pool.stride(1),
                         layer_stride if layer_stride is not None else (pool.stride(0) if L > 1 else 0))


# ------------------------------------------------------------- the C-ABI calls
def hc_encode_fp8(paged_k, paged_v, desc, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  stream=None):
    _check_encode(desc, paged_k, paged_v, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  HC_WIRE_FP8)
    _check("hc_encode_fp8", lib().hc_encode_fp8(
        _dptr(paged_k, "paged_k"), _dptr(paged_v, "paged_v"), ctypes.byref(desc),
        _dptr(src_slots, "src_slots"), _dptr(n_valid, "n_valid"), n_blocks, _dptr(codes, "codes"),
        _dptr(scales, "scales"), _dptr(err_flag, "err_flag"), _stream(stream)))


def hc_encode_fp8_crc(paged_k, paged_v, desc, src_slots, n_valid, n_blocks, codes, scales, crc,
                      err_flag, stream=None):
    _check_encode(desc, paged_k, paged_v, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  HC_WIRE_FP8, crc=crc)
    _check("hc_encode_fp8_crc", lib().hc_encode_fp8_crc(
        _dptr(paged_k, "paged_k"), _dptr(paged_v, "paged_v"), ctypes.byref(desc),
        _dptr(src_slots, "src_slots"), _dptr(n_valid, "n_valid"), n_blocks, _dptr(codes, "codes"),
        _dptr(scales, "scales"), _dptr(crc, "crc"), _dptr(err_flag, "err_flag"), _stream(stream)))


def hc_encode_int4(paged_k, paged_v, desc, src_slots, n_valid, n_blocks, group, scale_dtype,
                   codes, scales, err_flag, stream=None):
    _check_encode(desc, paged_k, paged_v, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  HC_WIRE_INT4, group, scale_dtype)
    _check("hc_encode_int4", lib().hc_encode_int4(
        _dptr(paged_k, "paged_k"), _dptr(paged_v, "paged_v"), ctypes.byref(desc),
        _dptr(src_slots, "src_slots"), _dptr(n_valid, "n_valid"), n_blocks, group, scale_dtype,
        _dptr(codes, "codes"), _dptr(scales, "scales"), _dptr(err_flag, "err_flag"),
        _stream(stream)))


def hc_encode_fp8_rows(paged_k, paged_v, desc, src_slots, n_valid, n_blocks, scale_dtype, codes,
                       scales, err_flag, stream=None):
    _check_encode(desc, paged_k, paged_v, src_slots, n_valid, n_blocks, codes, scales, err_flag,
                  HC_WIRE_FP8_ROWS, 32, scale_dtype)
    _check("hc_encode_fp8_rows", lib().hc_encode_fp8_rows(
        _dptr(paged_k, "paged_k"), _dptr(paged_v, "paged_v"), ctypes.byref(desc),
        _dptr(src_slots, "src_slots"), _dptr(n_valid, "n_valid"), n_blocks, scale_dtype,
        _dptr(codes, "codes"), _dptr(scales, "scales"), _dptr(err_flag, "err_flag"),
        _stream(stream)))


def hc_crc32(a, a_bytes, a_stride, b, b_bytes, b_stride, n_units, crc, stream=None):
    if n_units > 0 and a_bytes >= 0 and a_stride >= a_bytes and b_bytes >= 0 and b_stride >= b_bytes:
        _need(a, (n_units - 1) * a_stride + a_bytes, "a")
        if b_bytes:
            _need(b, (n_units - 1) * b_stride + b_bytes, "b")
        _need(crc, 4 * n_units, "crc")
    _check("hc_crc32", lib().hc_crc32(
        _dptr(a, "a"), a_bytes, a_stride, _dptr(b, "b"), b_bytes, b_stride, n_units,
        _dptr(crc, "crc"), _stream(stream)))


def hc_drift_select(h_cached, h_fresh, dtype, n_seq, n_tokens, hidden, token_stride, seq_stride, k,
                    drift, selected, stream=None):
    # k <= 0 asks the library for its default; the size check below needs the
    # k the library will use, which it reports through hc_selection_size
    k_used = hc_selection_size(n_tokens) if k <= 0 else k
    if (n_seq > 0 and n_tokens > 0 and hidden > 0 and dtype in _ES and 0 < k_used <= n_tokens
            and token_stride >= hidden and seq_stride >= n_tokens * token_stride):
        es = _ES[dtype]
        span = ((n_seq - 1) * seq_stride + (n_tokens - 1) * token_stride + hidden) * es
        _need(h_cached, span, "h_cached")
        _need(h_fresh, span, "h_fresh")
        _need(drift, 4 * n_seq * n_tokens, "drift")
        _need(selected, 4 * n_seq * k_used, "selected")
    _check("hc_drift_select", lib().hc_drift_select(
        _dptr(h_cached, "h_cached"), _dptr(h_fresh, "h_fresh"), dtype, n_seq, n_tokens, hidden,
        token_stride, seq_stride, k, _dptr(drift, "drift"), _dptr(selected, "selected"),
        _stream(stream)))


def hc_selection_size(n_tokens):
    return lib().hc_selection_size(n_tokens)


def selection_size(n_tokens):
    """The library's default number of tokens to recompute per sequence
    (hc_selection_size)."""
    return hc_selection_size(int(n_tokens))


def drift_select(h_cached, h_fresh, k=None, drift=None, selected=None, stream=None):
    """hc_drift_select on tensors shaped [n_seq, n_tokens, hidden] (or
    [n_tokens, hidden]); returns (drift [n_seq, n_tokens] f32, selected
    [n_seq, k] int32).  k = None takes the library's default,
    hc_selection_size(n_tokens)."""
    import torch
    if h_cached.dim() == 2:
        h_cached, h_fresh = h_cached.unsqueeze(0), h_fresh.unsqueeze(0)
    if h_cached.shape != h_fresh.shape or h_cached.stride() != h_fresh.stride():
        raise ValueError("h_cached and h_fresh must have the same shape and strides")
    if h_cached.stride(2) != 1:
        raise ValueError("the hidden dimension must be contiguous")
    n_seq, n_tokens, hidden = h_cached.shape
    k = selection_size(n_tokens) if k is None else k
    dev = h_cached.device
    drift = torch.empty((n_seq, n_tokens), dtype=torch.float32, device=dev) if drift is None else drift
    selected = torch.empty((n_seq, k), dtype=torch.int32, device=dev) if selected is None else selected
    dtype = {"torch.float32": HC_F32, "torch.float16": HC_F16, "torch.bfloat16": HC_BF16}[str(h_cached.dtype)]
    hc_drift_select(h_cached, h_fresh, dtype, n_seq, n_tokens, hidden, h_cached.stride(1),
                    h_cached.stride(0), k, drift, selected, stream)
    return drift, selected


def tenant_key(master, tenant=None):
    """hc_tenant_key on host bytes; returns the 32-byte secret."""
    m = bytes(master)
    out = ctypes.create_string_buffer(32)
    _check("hc_tenant_key", lib().hc_tenant_key(
        m, len(m), None if tenant is None else tenant.encode(), out))
    return out.raw


def block_digests(tokens, block_size, key):
    """hc_block_digests on a host int32 sequence; returns (prefix, content)
    as numpy uint8 arrays [n_blocks, 16]."""
    import numpy as np
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    k = bytes(key)
    n_blocks = -(-len(t) // block_size)
    prefix = np.zeros((n_blocks, 16), np.uint8)
    content = np.zeros((n_blocks, 16), np.uint8)
    _check("hc_block_digests", lib().hc_block_digests(
        t.ctypes.data, len(t), block_size, k, len(k), prefix.ctypes.data, content.ctypes.data))
    return prefix, content


def hc_build_delta_sincos(delta_m, n_distinct, d_head, rope_base, inv_freq, table, stream=None):
    if n_distinct > 0 and d_head > 0 and d_head % 2 == 0:
        _need(delta_m, 4 * n_distinct, "delta_m")
        _need(inv_freq, 8 * (d_head // 2), "inv_freq")
        _need(table, 8 * n_distinct * (d_head // 2), "table")
    _check("hc_build_delta_sincos", lib().hc_build_delta_sincos(
        _dptr(delta_m, "delta_m"), n_distinct, d_head, float(rope_base),
        _dptr(inv_freq, "inv_freq"), _dptr(table, "table"), _stream(stream)))


def hc_fetch_rotate_scatter(wire, codes, scales, group, scale_dtype, table, delta_idx, n_distinct,
                            pairing, dst_slots, n_valid, n_blocks, paged_k, paged_v, desc,
                            err_flag, stream=None):
    if _sizes_apply(desc, n_blocks, wire, group) and n_distinct > 0:
        pool = _pool_bytes(desc)
        _need(paged_k, pool, "paged_k")
        _need(paged_v, pool, "paged_v")
        cb, sb = _wire_bytes(desc, n_blocks, wire, group, scale_dtype)
        _need(codes, cb, "codes")
        _need(scales, sb, "scales")
        _need(table, 8 * n_distinct * (desc.d_head // 2), "table")
        for t, nm in ((delta_idx, "delta_idx"), (dst_slots, "dst_slots"), (n_valid, "n_valid")):
            _need(t, 4 * n_blocks, nm)
        _need(err_flag, 4, "err_flag")
    _check("hc_fetch_rotate_scatter", lib().hc_fetch_rotate_scatter(
        wire, _dptr(codes, "codes"), _dptr(scales, "scales"), group, scale_dtype,
        _dptr(table, "table"), _dptr(delta_idx, "delta_idx"), n_distinct, pairing,
        _dptr(dst_slots, "dst_slots"), _dptr(n_valid, "n_valid"), n_blocks,
        _dptr(paged_k, "paged_k"), _dptr(paged_v, "paged_v"), ctypes.byref(desc),
        _dptr(err_flag, "err_flag"), _stream(stream)))


# ------------------------------------------------------------- buffer shapes
def wire_shapes(n_layers, n_blocks, H, B, d, wire, group=32):
    """(codes shape, codes dtype name, scales shape) of a wire buffer, per the
    layouts in include/hc.h.  RAW codes are in the paged dtype."""
    if wire == HC_WIRE_FP8:
        return (n_layers, n_blocks, 2, H, B, d), "u8", (n_layers, n_blocks, 2, H)
    if wire == HC_WIRE_INT4:
        return (n_layers, n_blocks, 2, H, B, d // 2), "u8", (n_layers, n_blocks, 2, H, B, d // group)
    if wire == HC_WIRE_RAW:
        return (n_layers, n_blocks, 2, H, B, d), "paged", None
    if wire == HC_WIRE_FP8_ROWS:
        return (n_layers, n_blocks, 2, H, B, d), "u8", (n_layers, n_blocks, 2, H, B)
    raise ValueError(wire)
