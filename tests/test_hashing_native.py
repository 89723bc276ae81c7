"""The library's host-side block digests (hc_tenant_key, hc_block_digests)
against the oracle and the primitives' published vectors (CPU only: these
calls never touch the GPU)."""
import os
import shutil

import numpy as np
import pytest

from oracle import hashing


@pytest.fixture(scope="module")
def hc():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from kv_cache_quantization_hc_gb300 import build, hc as _hc
    build.build()
    return _hc


def test_tenant_keys_match_the_oracle(hc):
    for master in (b"", b"k", b"master secret", bytes(range(200))):   # > 64 bytes: hashed first
        for tenant in (None, "", "acme", "globex-" + "x" * 300):
            assert hc.tenant_key(master, tenant) == hashing.tenant_key(master, tenant)
    # RFC 4231 test case 2 reaches HMAC-SHA256 through the same code path
    # when the message is the tenant prefix: compare with hmac on that message
    import hashlib
    import hmac
    assert hc.tenant_key(b"Jefe", "x") == hmac.new(b"Jefe", b"hc-tenant:x", hashlib.sha256).digest()


@pytest.mark.parametrize("n_tokens,block", [(0, 16), (1, 16), (16, 16), (31, 16), (1000, 64),
                                            (4096 + 5, 64), (300, 1), (50, 2000)])
def test_block_digests_match_the_oracle(hc, n_tokens, block):
    r = np.random.default_rng(n_tokens + block)
    tokens = r.integers(-2 ** 31, 2 ** 31, n_tokens, dtype=np.int64).astype(np.int32)
    for key in (hashing.tenant_key(b"m", "acme"), bytes([7]), bytes(range(64))):
        p, c = hc.block_digests(tokens, block, key)
        wp, wc = hashing.block_digests(tokens, block, key)
        assert np.array_equal(p, wp) and np.array_equal(c, wc)


def test_host_validation(hc):
    L = hc.lib()
    import ctypes
    buf = ctypes.create_string_buffer(64)
    assert L.hc_block_digests(None, 0, 16, buf, 0, None, None) == hc.HC_ERR_INVALID_ARG      # key_len 0
    assert L.hc_block_digests(None, 0, 16, buf, 65, None, None) == hc.HC_ERR_INVALID_ARG     # key_len > 64
    assert L.hc_block_digests(None, 0, 0, buf, 16, None, None) == hc.HC_ERR_INVALID_ARG      # block 0
    assert L.hc_block_digests(None, 5, 16, buf, 16, None, None) == hc.HC_ERR_INVALID_ARG     # null tokens
    assert L.hc_block_digests(None, 0, 16, buf, 16, None, None) == hc.HC_OK                  # empty
    assert L.hc_tenant_key(None, 3, None, buf) == hc.HC_ERR_INVALID_ARG
    assert L.hc_tenant_key(buf, 4, None, None) == hc.HC_ERR_INVALID_ARG
