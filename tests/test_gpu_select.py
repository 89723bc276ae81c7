"""GPU parity of the drift-ranked token selection (hc_drift_select) against
the oracle.

Bars: drift within 2e-5 x the oracle value plus 1e-30 (fp32 differences,
squares and sum); the selection has k distinct ascending indices, every
selected token's oracle drift is at least every unselected token's minus
twice that tolerance, and where the oracle's k-th and (k+1)-th drifts differ
by more than that, the set equals the oracle's.  Constructed inputs with one
non-zero difference per token give exact drifts, so exact ties are checked
bit for bit, including the lower-index rule.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import blend

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
REL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check(cached, fresh, k, got_drift, got_sel):
    c = cached.double().cpu().numpy()
    f = fresh.double().cpu().numpy()
    want_drift, want_sel = blend.select(c, f, k)
    gd = got_drift.double().cpu().numpy()
    gs = got_sel.cpu().numpy().astype(np.int64)
    tol = REL * want_drift + 1e-30
    assert np.all(np.abs(gd - want_drift) <= tol), float(np.max(np.abs(gd - want_drift) - tol))
    for s in range(c.shape[0]):
        sel = gs[s]
        assert len(sel) == k and np.all(np.diff(sel) > 0) and sel[0] >= 0 and sel[-1] < c.shape[1]
        chosen = np.zeros(c.shape[1], bool)
        chosen[sel] = True
        dr = want_drift[s]
        if k < len(dr):
            assert dr[chosen].min() >= dr[~chosen].max() - 2 * tol[s].max()
            srt = np.sort(dr)[::-1]
            if srt[k - 1] - srt[k] > 2 * tol[s].max():
                assert np.array_equal(sel, want_sel[s])


@pytest.mark.parametrize("fmt", ["bf16", "f16", "f32"])
def test_random_hidden_states(fmt):
    w = workloads.blend_small()
    cached, fresh = workloads.blend_hidden(w, DEV)
    cached, fresh = cached.to(TDT[fmt]), fresh.to(TDT[fmt])
    from kv_cache_quantization_hc_gb300 import hc
    k = blend.default_k(w.n_tokens)
    d, s = hc.drift_select(cached, fresh, k)
    torch.cuda.synchronize()
    _check(cached, fresh, k, d, s)


@pytest.mark.parametrize("n_tokens,k", [(1, 1), (5, 5), (1000, 1), (2500, 375), (2500, 2500), (3000, 451)])
def test_sizes_and_k(n_tokens, k):
    from kv_cache_quantization_hc_gb300 import hc
    g = torch.Generator(device=DEV)
    g.manual_seed(n_tokens * 31 + k)
    cached = torch.randn((2, n_tokens, 64), generator=g, device=DEV).to(torch.bfloat16)
    fresh = (cached.float() + 0.1 * torch.randn((2, n_tokens, 64), generator=g, device=DEV)
             * torch.rand((2, n_tokens, 1), generator=g, device=DEV)).to(torch.bfloat16)
    d, s = hc.drift_select(cached, fresh, k)
    torch.cuda.synchronize()
    _check(cached, fresh, k, d, s)


def test_exact_ties_and_strides():
    """One non-zero difference per token from a small set of values: exact
    drifts with many ties; rows and sequences strided (padding between)."""
    from kv_cache_quantization_hc_gb300 import hc
    r = np.random.default_rng(3)
    n_seq, T, D, pad_t, pad_s = 3, 700, 64, 16, 48
    vals = np.array([0.5, 1.0, 1.5, 2.0, 3.0])
    buf_c = torch.zeros((n_seq * (T * (D + pad_t) + pad_s)), dtype=torch.float16, device=DEV)
    buf_f = torch.zeros_like(buf_c)
    cached = buf_c.as_strided((n_seq, T, D), (T * (D + pad_t) + pad_s, D + pad_t, 1))
    fresh = buf_f.as_strided((n_seq, T, D), (T * (D + pad_t) + pad_s, D + pad_t, 1))
    base = torch.from_numpy(r.standard_normal((n_seq, T, D))).to(torch.float16).to(DEV)
    cached.copy_(base)
    delta = np.zeros((n_seq, T, D))
    delta[:, np.arange(T), r.integers(0, D, T)] = r.choice(vals, size=(n_seq, T)) * r.choice([-1, 1], size=(n_seq, T))
    fresh.copy_(base + torch.from_numpy(delta).to(torch.float16).to(DEV))
    # the fp16 sums base + delta are exact only where they are representable: use
    # the stored values for the oracle (it reads the same tensors back)
    for k in (1, 37, 140, 699, 700):
        drift = torch.empty((n_seq, T), dtype=torch.float32, device=DEV)
        sel = torch.empty((n_seq, k), dtype=torch.int32, device=DEV)
        hc.hc_drift_select(cached, fresh, hc.HC_F16, n_seq, T, D, D + pad_t, T * (D + pad_t) + pad_s,
                           k, drift, sel)
        torch.cuda.synchronize()
        c = cached.double().cpu().numpy()
        f = fresh.double().cpu().numpy()
        want_d, want_s = blend.select(c, f, k)
        assert np.array_equal(drift.double().cpu().numpy(), want_d.astype(np.float32).astype(np.float64))
        assert np.array_equal(sel.cpu().numpy(), want_s)


def test_full_size_workload_sampled():
    """The benchmark's 64 x 2048 x 4096 bf16 call, checked on three
    sequences re-drawn alone."""
    from kv_cache_quantization_hc_gb300 import hc
    w = workloads.blend_selection()
    cached, fresh = workloads.blend_hidden(w, DEV)
    k = blend.default_k(w.n_tokens)
    d, s = hc.drift_select(cached, fresh, k)
    torch.cuda.synchronize()
    for seq in (0, 31, 63):
        c1, f1 = workloads.blend_hidden(w, DEV, seqs=[seq])
        _check(c1, f1, k, d[seq:seq + 1], s[seq:seq + 1])


def test_default_k_through_the_c_abi():
    """k = 0 through the C ABI selects the library's default share of the
    tokens (hc_selection_size): the oracle's ceil(15%), and the same drift and
    selection as an explicit k of that size."""
    from kv_cache_quantization_hc_gb300 import hc
    w = workloads.blend_small()
    cached, fresh = workloads.blend_hidden(w, DEV)
    k = blend.default_k(w.n_tokens)
    assert hc.lib().hc_selection_size(w.n_tokens) == k
    n_seq, T, D = cached.shape
    drift = torch.empty((n_seq, T), dtype=torch.float32, device=DEV)
    sel = torch.full((n_seq, k), -1, dtype=torch.int32, device=DEV)
    hc.hc_drift_select(cached, fresh, hc.HC_BF16, n_seq, T, D, D, T * D, 0, drift, sel)
    d2, s2 = hc.drift_select(cached, fresh, k)
    torch.cuda.synchronize()
    assert torch.equal(drift, d2) and torch.equal(sel, s2)
    _check(cached, fresh, k, drift, sel)
