"""Plain float64 CPU oracle for the KV-cache wire codec and relative-RoPE fetch.

TEST INFRASTRUCTURE ONLY.  This package is a slow, obviously correct
restatement of what the method computes, written from the pages' text:

* "HyperCache - Distributed KV-cache quantization and relative RoPE reuse"
  (the relative RoPE rotation on fetch, FP8 E4M3 wire quantization, grouped
  INT4, and the example benchmark output), and
* "Module 13: KV handoff" (the KV-bytes formula, the RoPE / strip-RoPE
  convention in its numpy listing).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
legs may import it.  It shares no code with the CUDA path and imports nothing
from it; the CUDA path never imports this package.

Every function states the passage it follows.  Every function is pinned by a
``-m "not gpu"`` test against something other than itself (a value the pages
print, a closed form, a library routine, or brute force); the one measurement
the oracle cannot reproduce (the FP8 cosine similarity of 0.999979) is marked
"parity unpinned" in ``quant.py``.
"""

from . import numerics, rope, fp8, quant, paged, kvbytes  # noqa: F401
