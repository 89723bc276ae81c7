"""Host logic of the binding: the number of tokens the drift-ranked
selection recomputes by default."""
from oracle import blend


def test_product_selection_size_agrees_with_the_oracle():
    """The binding's k (exact rational ceil) and the oracle's (float ceil)
    are written independently; they agree for every sequence length used."""
    from kv_cache_quantization_hc_gb300 import hc
    for t in list(range(1, 5000)) + [20480, 131072, 1 << 20]:
        assert hc.selection_size(t) == blend.default_k(t), t
    assert hc.selection_size(100) == 15 and hc.selection_size(1408) == 212
    assert hc.selection_size(7, 0.5) == 4 and hc.selection_size(3, 0.01) == 1
