"""Which tokens to recompute after cached chunks are reordered.

ORACLE (test infrastructure only; see the package docstring).

The page pairs the relative RoPE rotation with selective recomputation: layer
0 K/V depends only on the token embeddings, so the rotated layer-0 KV is
exact, and about 15% of the tokens, those whose layer-0 hidden state moved
furthest, are recomputed through the deeper layers, following CacheBlend
["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
"Core Design", paragraph after the relative-RoPE identity; "Example output"
part A, "RoPE Shift + 15% CacheBlend"].

Reading taken (the page gives no formula):

* drift_t = || h_fresh[t] - h_cached[t] ||_2 over the hidden dimension, where
  h_cached is the layer-0 output hidden state kept with the cache and h_fresh
  the one recomputed in the new context;
* k = ceil(0.15 * n_tokens) by default (the caller may pass any k);
* the k tokens with the largest drift are selected, ties going to the lower
  token index; the result is their indices in ascending order.

The recompute itself needs a model and is not part of this path.
"""
import math

import numpy as np


def default_k(n_tokens, fraction=0.15):
    return max(1, math.ceil(fraction * n_tokens - 1e-12))


def drift(h_cached, h_fresh):
    """[..., T] float64 L2 norms of h_fresh - h_cached over the last axis."""
    d = np.asarray(h_fresh, dtype=np.float64) - np.asarray(h_cached, dtype=np.float64)
    return np.sqrt(np.sum(d * d, axis=-1))


def select_topk(drift_values, k):
    """Ascending indices of the k largest values of a 1-D array; among equal
    values the lower index wins."""
    v = np.asarray(drift_values, dtype=np.float64)
    order = sorted(range(len(v)), key=lambda t: (-v[t], t))
    return np.array(sorted(order[:k]), dtype=np.int64)


def select(h_cached, h_fresh, k):
    """Per sequence: (drift [n_seq, T], selected [n_seq, k]) for inputs
    shaped [n_seq, T, hidden]."""
    dr = drift(h_cached, h_fresh)
    sel = np.stack([select_topk(dr[s], k) for s in range(dr.shape[0])])
    return dr, sel
