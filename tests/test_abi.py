"""The C-ABI library builds, loads and exports every symbol include/hc.h
declares; host-side validation answers without touching CUDA (CPU only)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "hc.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_0-9]+\s*\*?\s*(hc_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from kv_cache_quantization_hc_gb300 import build, hc
    build.build()
    return hc.lib()


def test_header_declares_the_calls():
    names = _declared_functions()
    for n in ("hc_encode_fp8", "hc_encode_fp8_crc", "hc_encode_int4", "hc_encode_fp8_rows",
              "hc_build_delta_sincos",
              "hc_fetch_rotate_scatter", "hc_crc32", "hc_drift_select", "hc_tenant_key",
              "hc_block_digests", "hc_status_string"):
        assert n in names, names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    from kv_cache_quantization_hc_gb300 import hc
    assert hc.hc_version() == 3
    assert hc.status_string(0) == "HC_OK"
    assert hc.status_string(-1) == "HC_ERR_INVALID_ARG"
    assert hc.status_string(-2) == "HC_ERR_UNSUPPORTED"
    assert hc.status_string(-3) == "HC_ERR_CUDA"
    assert hc.status_string(5) == "HC_UNKNOWN_STATUS"
    assert lib.hc_last_cuda_error() == b""


def test_host_validation_without_cuda(lib):
    """Every check below returns before any CUDA call (fake addresses)."""
    from kv_cache_quantization_hc_gb300 import hc
    A = 1 << 20          # a 16-byte aligned fake address; never dereferenced
    good = hc.hc_paged_desc(1, 8, 128, 16, 4, hc.HC_BF16, 16 * 8 * 128, 0)
    L = lib
    P = ctypes.byref
    # null paged pointer
    assert L.hc_encode_fp8(None, A, P(good), A, None, 1, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    # unsupported d_head / block size / group
    for bad in (hc.hc_paged_desc(1, 8, 96, 16, 4, hc.HC_BF16, 16 * 8 * 96, 0),
                hc.hc_paged_desc(1, 8, 128, 8, 4, hc.HC_BF16, 8 * 8 * 128, 0)):
        assert L.hc_encode_fp8(A, A, P(bad), A, None, 1, A, A, A, None) == hc.HC_ERR_UNSUPPORTED
    assert L.hc_encode_int4(A, A, P(good), A, None, 1, 16, hc.HC_F16, A, A, A, None) == hc.HC_ERR_UNSUPPORTED
    # misaligned codes, negative block count, unknown dtype, too-small slot stride
    assert L.hc_encode_fp8(A, A, P(good), A, None, 1, A + 1, A, A, None) == hc.HC_ERR_INVALID_ARG
    assert L.hc_encode_fp8(A, A, P(good), A, None, -1, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    bad = hc.hc_paged_desc(1, 8, 128, 16, 4, 9, 16 * 8 * 128, 0)
    assert L.hc_encode_fp8(A, A, P(bad), A, None, 1, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    bad = hc.hc_paged_desc(1, 8, 128, 16, 4, hc.HC_BF16, 100, 0)
    assert L.hc_encode_fp8(A, A, P(bad), A, None, 1, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    bad = hc.hc_paged_desc(2, 8, 128, 16, 4, hc.HC_BF16, 16 * 8 * 128, 0)   # 2 layers, stride 0
    assert L.hc_encode_fp8(A, A, P(bad), A, None, 1, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    # fetch: unknown wire / pairing, missing scales, no table rows
    f = L.hc_fetch_rotate_scatter
    assert f(7, A, A, 32, hc.HC_F16, A, A, 1, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    assert f(0, A, A, 32, hc.HC_F16, A, A, 1, 5, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    assert f(0, A, None, 32, hc.HC_F16, A, A, 1, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    assert f(0, A, A, 32, hc.HC_F16, A, A, 0, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    assert f(1, A, A, 256, hc.HC_F16, A, A, 1, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_UNSUPPORTED
    # table: odd d_head, bad base
    t = L.hc_build_delta_sincos
    assert t(A, 1, 127, ctypes.c_double(1e4), None, A, None) == hc.HC_ERR_INVALID_ARG
    assert t(A, 1, 128, ctypes.c_double(0.0), None, A, None) == hc.HC_ERR_INVALID_ARG
    assert t(A, -1, 128, ctypes.c_double(1e4), None, A, None) == hc.HC_ERR_INVALID_ARG
    # zero blocks / rows launch nothing and succeed
    assert L.hc_encode_fp8(A, A, P(good), A, None, 0, A, A, A, None) == hc.HC_OK
    assert f(0, A, A, 32, hc.HC_F16, A, A, 0, 0, A, None, 0, A, A, P(good), A, None) == hc.HC_OK
    assert t(A, 0, 128, ctypes.c_double(1e4), None, A, None) == hc.HC_OK


def test_host_validation_of_rows_and_crc(lib):
    """Row-scaled FP8 and CRC-32 argument checks (fake addresses, no CUDA)."""
    from kv_cache_quantization_hc_gb300 import hc
    A = 1 << 20
    good = hc.hc_paged_desc(1, 8, 128, 16, 4, hc.HC_BF16, 16 * 8 * 128, 0)
    P = ctypes.byref
    r = lib.hc_encode_fp8_rows
    assert r(A, A, P(good), A, None, 1, 7, A, A, A, None) == hc.HC_ERR_INVALID_ARG      # scale dtype
    assert r(A, A, P(good), A, None, 1, hc.HC_F16, A + 8, A, A, None) == hc.HC_ERR_INVALID_ARG  # codes
    assert r(A, A, P(good), A, None, 1, hc.HC_F16, A, A + 1, A, None) == hc.HC_ERR_INVALID_ARG  # scales
    assert r(A, A, P(good), A, None, 0, hc.HC_F16, A, A, A, None) == hc.HC_OK
    f = lib.hc_fetch_rotate_scatter
    assert f(3, A, A, 32, 9, A, A, 1, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    assert f(3, A, A + 2, 32, hc.HC_F32, A, A, 1, 0, A, None, 1, A, A, P(good), A, None) == hc.HC_ERR_INVALID_ARG
    c = lib.hc_crc32
    assert c(A + 4, 64, 64, None, 0, 0, 1, A, None) == hc.HC_ERR_INVALID_ARG          # a alignment
    assert c(A, 64, 72, None, 0, 0, 2, A, None) == hc.HC_ERR_INVALID_ARG              # a stride
    assert c(A, 64, 32, None, 0, 0, 2, A, None) == hc.HC_ERR_INVALID_ARG              # overlap
    assert c(A, 64, 64, None, 8, 8, 1, A, None) == hc.HC_ERR_INVALID_ARG              # b missing
    assert c(A, 64, 64, None, 0, 0, -1, A, None) == hc.HC_ERR_INVALID_ARG
    assert c(A, 64, 64, None, 0, 0, 0, A, None) == hc.HC_OK


def test_host_validation_of_drift_select(lib):
    from kv_cache_quantization_hc_gb300 import hc
    A = 1 << 20
    d = lib.hc_drift_select
    ok = (A, A, hc.HC_BF16, 2, 100, 64, 64, 6400, 15, A, A, None)
    assert d(*ok[:2], 9, *ok[3:]) == hc.HC_ERR_INVALID_ARG                       # dtype
    assert d(A, A, hc.HC_BF16, 2, 100, 60, 64, 6400, 15, A, A, None) == hc.HC_ERR_INVALID_ARG   # hidden % 8
    # k <= 0 takes the default (15 of 100 tokens): valid, so an invalid stride still decides
    assert d(A, A, hc.HC_BF16, 2, 100, 64, 60, 6400, 0, A, A, None) == hc.HC_ERR_INVALID_ARG    # stride
    assert d(A, A, hc.HC_BF16, 2, 100, 64, 64, 6400, 101, A, A, None) == hc.HC_ERR_INVALID_ARG  # k > T
    assert d(A, A, hc.HC_BF16, 2, 100, 64, 60, 6400, 15, A, A, None) == hc.HC_ERR_INVALID_ARG   # stride
    assert d(A, A, hc.HC_BF16, 2, 100, 64, 64, 6000, 15, A, A, None) == hc.HC_ERR_INVALID_ARG   # overlap
    assert d(A + 8, A, hc.HC_BF16, 2, 100, 64, 64, 6400, 15, A, A, None) == hc.HC_ERR_INVALID_ARG
    assert d(A, A, hc.HC_BF16, 0, 100, 64, 64, 6400, 15, A, A, None) == hc.HC_OK


def test_host_validation_of_fused_crc(lib):
    from kv_cache_quantization_hc_gb300 import hc
    A = 1 << 20
    good = hc.hc_paged_desc(1, 8, 128, 16, 4, hc.HC_BF16, 16 * 8 * 128, 0)
    P = ctypes.byref
    e = lib.hc_encode_fp8_crc
    assert e(A, A, P(good), A, None, 1, A, A, None, A, None) == hc.HC_ERR_INVALID_ARG     # no crc
    assert e(A, A, P(good), A, None, 1, A, A, A + 2, A, None) == hc.HC_ERR_INVALID_ARG    # alignment
    assert e(A, A, P(good), A, None, 0, A, A, A, A, None) == hc.HC_OK


def test_host_rejects_grids_past_32_bit_indexing(lib):
    """2^31 or more 16-token sub-slabs in one call would overflow the kernels'
    32-bit sub-slab index: every entry point rejects it before any CUDA call."""
    from kv_cache_quantization_hc_gb300 import hc
    A = 1 << 20
    P = ctypes.byref
    slot = 16 * 8 * 128
    # 2^14 layers x 2^13 blocks x 2 (K, V) x 8 heads x 1 sub-slab = 2^31
    big = hc.hc_paged_desc(1 << 14, 8, 128, 16, 1 << 13, hc.HC_BF16, slot, slot << 13)
    nb = 1 << 13
    assert lib.hc_encode_fp8(A, A, P(big), A, None, nb, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    assert lib.hc_encode_fp8_crc(A, A, P(big), A, None, nb, A, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    assert lib.hc_encode_int4(A, A, P(big), A, None, nb, 32, hc.HC_F16, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    assert lib.hc_encode_fp8_rows(A, A, P(big), A, None, nb, hc.HC_F16, A, A, A, None) == hc.HC_ERR_INVALID_ARG
    f = lib.hc_fetch_rotate_scatter
    assert f(0, A, A, 32, hc.HC_F16, A, A, 1, 0, A, None, nb, A, A, P(big), A, None) == hc.HC_ERR_INVALID_ARG


def test_binding_rejects_host_tensors_for_device_buffers(lib):
    """The kernels dereference every buffer pointer: the binding refuses a
    host tensor before the call instead of letting a kernel fault on it."""
    import torch
    from kv_cache_quantization_hc_gb300 import hc
    good = hc.hc_paged_desc(1, 8, 128, 16, 4, hc.HC_BF16, 16 * 8 * 128, 0)
    host = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(ValueError, match="src_slots"):
        hc.hc_encode_fp8(1 << 20, 1 << 20, good, host, None, 1, 1 << 20, 1 << 20, 1 << 20)
    with pytest.raises(ValueError, match="codes"):
        hc.hc_fetch_rotate_scatter(0, host, 1 << 20, 32, hc.HC_F16, 1 << 20, 1 << 20, 1, 0,
                                   1 << 20, None, 1, 1 << 20, 1 << 20, good, 1 << 20)
    with pytest.raises(ValueError, match="crc"):
        hc.hc_crc32(1 << 20, 64, 64, None, 0, 0, 1, host)
    with pytest.raises(ValueError, match="h_cached"):
        hc.hc_drift_select(host, 1 << 20, hc.HC_BF16, 1, 16, 8, 8, 128, 2, 1 << 20, 1 << 20)
    with pytest.raises(ValueError, match="table"):
        hc.hc_build_delta_sincos(1 << 20, 1, 128, 1e4, None, host)


def test_binding_refuses_buffers_smaller_than_the_call(lib):
    """A buffer smaller than the bytes the call will address is refused
    before the call (checked ahead of the device check, so it runs here).
    A view is measured by the storage behind its data pointer."""
    import torch
    from kv_cache_quantization_hc_gb300 import hc
    L, H, d, B, S, nb = 2, 8, 128, 16, 4, 3
    slot = B * H * d
    desc = hc.hc_paged_desc(L, H, d, B, S, hc.HC_BF16, slot, S * slot)
    pool = torch.zeros(L * S * slot, dtype=torch.bfloat16)
    small = torch.zeros(L * S * slot - 1, dtype=torch.bfloat16)
    tab = torch.zeros(nb, dtype=torch.int32)
    codes = torch.zeros(L * nb * 2 * H * B * d, dtype=torch.uint8)
    scales = torch.zeros(L * nb * 2 * H, dtype=torch.float32)
    err = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="paged_v holds"):
        hc.hc_encode_fp8(pool, small, desc, tab, None, nb, codes, scales, err)
    with pytest.raises(ValueError, match="src_slots holds"):
        hc.hc_encode_fp8(pool, pool, desc, torch.zeros(nb - 1, dtype=torch.int32), None, nb,
                         codes, scales, err)
    with pytest.raises(ValueError, match="codes holds"):
        hc.hc_encode_fp8(pool, pool, desc, tab, None, nb,
                         torch.zeros(codes.numel() - 1, dtype=torch.uint8), scales, err)
    with pytest.raises(ValueError, match="scales holds"):
        hc.hc_encode_int4(pool, pool, desc, tab, None, nb, 32, hc.HC_F16,
                          torch.zeros(codes.numel() // 2, dtype=torch.uint8),
                          torch.zeros(3, dtype=torch.float16), err)
    with pytest.raises(ValueError, match="crc holds"):
        hc.hc_encode_fp8_crc(pool, pool, desc, tab, None, nb, codes, scales,
                             torch.zeros(L * nb * 2 * H - 1, dtype=torch.int32), err)
    with pytest.raises(ValueError, match="table holds"):
        hc.hc_fetch_rotate_scatter(hc.HC_WIRE_FP8, codes, scales, 32, hc.HC_F16,
                                   torch.zeros(64 * 2 - 1, dtype=torch.float32), tab, 1, 0, tab,
                                   None, nb, pool, pool, desc, err)
    with pytest.raises(ValueError, match="a holds"):
        hc.hc_crc32(torch.zeros(100, dtype=torch.uint8), 64, 64, None, 0, 0, 2, err)
    with pytest.raises(ValueError, match="selected holds"):
        h = torch.zeros(2 * 16 * 8, dtype=torch.bfloat16)
        hc.hc_drift_select(h, h, hc.HC_BF16, 2, 16, 8, 8, 128, 3,
                           torch.zeros(32, dtype=torch.float32), torch.zeros(5, dtype=torch.int32))
    # a call whose buffers are large enough gets past the size checks, to the device check
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        hc.hc_encode_fp8(pool, pool, desc, tab, None, nb, codes, scales, err)
