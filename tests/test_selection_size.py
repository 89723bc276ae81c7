"""The default number of tokens the drift-ranked selection recomputes,
computed by the library (hc_selection_size, a host function of the C ABI),
against the oracle's, which is written independently (a float ceil of
0.15 * n_tokens): they agree for every sequence length used.  Also checks
that hc_drift_select accepts k <= 0 as "the default" on the host side."""
import ctypes

import pytest

from oracle import blend


@pytest.fixture(scope="module")
def hc():
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_quantization_hc_gb300 import hc
    return hc


def test_library_selection_size_agrees_with_the_oracle(hc):
    L = hc.lib()
    for t in list(range(1, 5000)) + [20480, 131072, 1 << 20, (1 << 31) - 1]:
        assert L.hc_selection_size(t) == blend.default_k(t), t
    assert L.hc_selection_size(100) == 15 and L.hc_selection_size(1408) == 212
    assert L.hc_selection_size(0) == 0 and L.hc_selection_size(-5) == 0
    assert hc.selection_size(2048) == 308


def test_drift_select_default_k_is_validated_on_the_host(hc):
    """k <= 0 passes the k check (the default is 1 <= k <= n_tokens); with a
    null drift pointer the call still fails on the host before any launch."""
    L = hc.lib()
    p = ctypes.c_void_p(1 << 20)
    assert L.hc_drift_select(p, p, hc.HC_BF16, 1, 16, 8, 8, 128, 0, None, p, None) == hc.HC_ERR_INVALID_ARG
    # n_seq = 0 with every argument valid launches nothing and returns HC_OK,
    # for an explicit k and for the default
    for k in (3, 0, -1):
        assert L.hc_drift_select(p, p, hc.HC_BF16, 0, 16, 8, 8, 128, k, p, p, None) == hc.HC_OK
    assert L.hc_drift_select(p, p, hc.HC_BF16, 0, 16, 8, 8, 128, 17, p, p, None) == hc.HC_ERR_INVALID_ARG
