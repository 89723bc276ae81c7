"""Seeded synthetic inputs for the five workloads.

This module draws random numbers and builds block tables; it holds none of
the method's arithmetic (no RoPE, no quantization, no rounding rules).  It is
the one piece both the oracle side (tests, CPU baseline) and the CUDA side
(tests, benchmark) use.

Workloads (all shapes from the pages' named models; no weights involved):

* ``tiny``         1 layer, 2 KV heads, d 64, 4 blocks x 16 tokens, fp32,
                   interleaved pairs, RoPE base 1e4, m_old = 16 j + t,
                   delta-m ~ U{-48..1024}, 16-slot pools, seed 0.
* ``gqa_reorder``  4 layers, 8 heads, d 128, bf16, chunks [Sys 256, DocB 512,
                   DocA 512, Q 128] reordered to [Sys, DocA, DocB, Q],
                   4 outlier channels x8 per (layer, kv, head), base 5e5,
                   half-split pairs, block 16, seed 1.
* ``qwen3_8b``     36 layers, 8 heads, d 128, 32768 tokens, fp16 ~N(0, 0.5^2),
                   block 16, delta-m = +4096, shuffled block tables, base 1e6,
                   bf16 destination, seed 2.
* ``llama3_70b``   80 layers, 8 heads, d 128, 65536 tokens, block 64, K/V
                   Student-t(5) x 0.3 in bf16, 1024 RAG chunks of 64 tokens
                   shuffled (delta-m = 64 (pi(c) - c)), base 5e5, seed 3.
* ``ragged``       36 layers, 8 heads, d 128, 64 requests with lengths
                   log-uniform in [200, 25000], block 16 or 64 per request,
                   delta-m ~ U{-8192..8192} per block, bf16 ~N(0,1) with 3 of
                   128 channels (2 %) x10 per (layer, kv, head), base 1e6,
                   seed 4.

The small workloads (tiny, gqa_reorder) are drawn on the host in float64 as
PRE-RoPE keys and values plus positions; the caller makes the cached
(post-RoPE) tensor.  The large ones are drawn on the device directly as the
cached tensor (post-RoPE keys of an isotropic draw are again isotropic, so the
draw has the stated distribution), one layer at a time where memory requires.
"""
from dataclasses import dataclass, field
import math

import numpy as np

INTERLEAVED = "interleaved"
HALF_SPLIT = "half_split"


@dataclass
class Blocks:
    """Per-block tables of one call (one block size)."""
    B: int
    src_slots: np.ndarray          # int32 [NB]
    dst_slots: np.ndarray          # int32 [NB]
    n_valid: np.ndarray            # int32 [NB]
    delta_m: np.ndarray            # int64 [NB]
    num_src_slots: int
    num_dst_slots: int

    @property
    def nb(self):
        return len(self.src_slots)

    def distinct(self):
        """(distinct delta-m values int32 [n], delta_idx int32 [NB])."""
        vals, idx = np.unique(self.delta_m, return_inverse=True)
        return vals.astype(np.int32), idx.astype(np.int32)

    def tokens(self):
        return int(self.n_valid.sum())


@dataclass
class Workload:
    name: str
    L: int
    H: int
    d: int
    src_dtype: str                 # 'f32' | 'f16' | 'bf16'
    out_dtype: str
    rope_base: float
    pairing: str
    blocks: list                   # list[Blocks], one per block size
    seed: int
    extra: dict = field(default_factory=dict)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- host draws
@dataclass
class HostDraw:
    """Pre-RoPE K/V for every block of one Blocks entry, plus m_old per token."""
    k_pre: np.ndarray              # float64 [L, NB, B, H, d]
    v: np.ndarray                  # float64 [L, NB, B, H, d]
    m_old: np.ndarray              # int64 [NB, B]
    filler_src: np.ndarray         # float64 [L, num_src_slots, B, H, d] (unused slots' contents)


def tiny(seed=0):
    r = _rng(seed)
    L, H, d, B, NB, S = 1, 2, 64, 16, 4, 16
    src = r.permutation(S)[:NB].astype(np.int32)
    dst = r.permutation(S)[:NB].astype(np.int32)
    dm = r.integers(-48, 1024, size=NB, endpoint=True).astype(np.int64)
    blk = Blocks(B, src, dst, np.full(NB, B, np.int32), dm, S, S)
    w = Workload("tiny", L, H, d, "f32", "f32", 1e4, INTERLEAVED, [blk], seed)
    k = r.standard_normal((L, NB, B, H, d))
    v = r.standard_normal((L, NB, B, H, d))
    filler = r.standard_normal((L, S, B, H, d))
    m_old = (B * np.arange(NB))[:, None] + np.arange(B)[None, :]
    return w, [HostDraw(k, v, m_old, filler)]


def gqa_reorder(seed=1):
    """Chunks [Sys 256, DocB 512, DocA 512, Q 128] cached in that order, reused
    in the order [Sys, DocA, DocB, Q]: DocB moves by +512, DocA by -512."""
    r = _rng(seed)
    L, H, d, B = 4, 8, 128, 16
    chunks = [("Sys", 256), ("DocB", 512), ("DocA", 512), ("Q", 128)]
    new_order = ["Sys", "DocA", "DocB", "Q"]
    old_start, pos = {}, 0
    for name, n in chunks:
        old_start[name] = pos
        pos += n
    T = pos
    new_start, pos = {}, 0
    for name in new_order:
        new_start[name] = pos
        pos += dict(chunks)[name]
    NB = T // B
    dm = np.zeros(NB, np.int64)
    new_block = np.zeros(NB, np.int64)
    for name, n in chunks:
        for b in range(n // B):
            j = old_start[name] // B + b
            dm[j] = new_start[name] - old_start[name]
            new_block[j] = new_start[name] // B + b
    S = NB + 8
    src = r.permutation(S)[:NB].astype(np.int32)
    dperm = r.permutation(S)
    dst = dperm[new_block].astype(np.int32)
    blk = Blocks(B, src, dst, np.full(NB, B, np.int32), dm, S, S)
    w = Workload("gqa_reorder", L, H, d, "bf16", "bf16", 5e5, HALF_SPLIT, [blk], seed,
                 extra={"chunks": chunks, "new_order": new_order})
    k = r.standard_normal((L, NB, B, H, d))
    v = r.standard_normal((L, NB, B, H, d))
    # 4 outlier channels per (layer, kv, head), scaled x8 (applied pre-RoPE)
    for arr in (k, v):
        for layer in range(L):
            for h in range(H):
                ch = r.choice(d, size=4, replace=False)
                arr[layer, :, :, h, ch] *= 8.0
    filler = r.standard_normal((L, S, B, H, d))
    m_old = (B * np.arange(NB))[:, None] + np.arange(B)[None, :]
    return w, [HostDraw(k, v, m_old, filler)]


# ---------------------------------------------------------------- large shapes
def qwen3_8b(seed=2):
    r = _rng(seed)
    L, H, d, B, T = 36, 8, 128, 16, 32768
    NB = T // B
    src = r.permutation(NB).astype(np.int32)
    dst = r.permutation(NB).astype(np.int32)
    dm = np.full(NB, 4096, np.int64)
    blk = Blocks(B, src, dst, np.full(NB, B, np.int32), dm, NB, NB)
    return Workload("qwen3_8b", L, H, d, "f16", "bf16", 1e6, HALF_SPLIT, [blk], seed,
                    extra={"dist": ("normal", 0.5)})


def llama3_70b(seed=3):
    r = _rng(seed)
    L, H, d, B, T = 80, 8, 128, 64, 65536
    NB = T // B                                   # 1024 chunks of one block each
    pi = r.permutation(NB)                        # chunk c is reused at position pi[c]
    dm = (B * (pi - np.arange(NB))).astype(np.int64)
    src = r.permutation(NB).astype(np.int32)
    dperm = r.permutation(NB)
    dst = dperm[pi].astype(np.int32)
    blk = Blocks(B, src, dst, np.full(NB, B, np.int32), dm, NB, NB)
    return Workload("llama3_70b", L, H, d, "bf16", "bf16", 5e5, HALF_SPLIT, [blk], seed,
                    extra={"dist": ("student_t", 5.0, 0.3)})


def ragged(seed=4, n_requests=64):
    r = _rng(seed)
    L, H, d = 36, 8, 128
    lengths = np.rint(np.exp(r.uniform(math.log(200), math.log(25000), n_requests))).astype(np.int64)
    bsz = np.where(r.random(n_requests) < 0.5, 16, 64)
    blocks = []
    for B in (16, 64):
        nv = []
        for n, b in zip(lengths, bsz):
            if b != B:
                continue
            full, tail = divmod(int(n), B)
            nv += [B] * full + ([tail] if tail else [])
        NB = len(nv)
        src = r.permutation(NB).astype(np.int32)
        dst = r.permutation(NB).astype(np.int32)
        dm = r.integers(-8192, 8192, size=NB, endpoint=True).astype(np.int64)
        blocks.append(Blocks(B, src, dst, np.asarray(nv, np.int32), dm, NB, NB))
    return Workload("ragged", L, H, d, "bf16", "bf16", 1e6, HALF_SPLIT, blocks, seed,
                    extra={"lengths": lengths, "block_size": bsz,
                           "dist": ("normal_outliers", 1.0, 3, 10.0)})


WORKLOADS = {"tiny": tiny, "gqa_reorder": gqa_reorder, "qwen3_8b": qwen3_8b,
             "llama3_70b": llama3_70b, "ragged": ragged}


# ---------------------------------------------------------------- device draws
_TORCH_DTYPE = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def torch_dtype(name):
    import torch
    return getattr(torch, _TORCH_DTYPE[name])


def device_pool(w, blk, layers, kv, device, seed_offset=0):
    """Draw the cached pool [len(layers), num_src_slots, B, H, d] on the device.

    ``layers`` is a range of layer indices; each (layer, kv) gets its own
    generator seed so that any layer can be re-drawn alone.
    """
    import torch
    dt = torch_dtype(w.src_dtype)
    out = torch.empty((len(layers), blk.num_src_slots, blk.B, w.H, w.d), dtype=dt, device=device)
    dist = w.extra.get("dist", ("normal", 1.0))
    for i, layer in enumerate(layers):
        g = torch.Generator(device=device)
        g.manual_seed(w.seed * 1_000_003 + layer * 2 + kv + 7919 * (seed_offset + blk.B))
        shape = out.shape[1:]
        if dist[0] == "normal":
            x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * dist[1]
        elif dist[0] == "student_t":
            nu, sc = dist[1], dist[2]
            z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            # chi-square(nu) as a sum of nu squared normals (nu is an integer here)
            chi = torch.zeros(shape, device=device, dtype=torch.float32)
            for _ in range(int(nu)):
                chi += torch.randn(shape, generator=g, device=device, dtype=torch.float32) ** 2
            x = z / torch.sqrt(chi / nu) * sc
        elif dist[0] == "normal_outliers":
            sigma, n_out, factor = dist[1], dist[2], dist[3]
            x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma
            mult = torch.ones(w.H, w.d, device=device)
            for h in range(w.H):
                ch = torch.randperm(w.d, generator=g, device=device)[:n_out]
                mult[h, ch] = factor
            x *= mult
        else:
            raise ValueError(dist)
        out[i] = x.to(dt)
    return out


# ------------------------------------------------------------------ token selection
@dataclass
class BlendWorkload:
    """Layer-0 hidden states before (cached) and after (fresh) a reorder, for
    the drift-ranked token selection: n_seq sequences of n_tokens rows of
    `hidden` values.  cached ~ N(0, 1); fresh = cached + delta with
    delta_t ~ N(0, sigma_t^2), sigma_t = 0.05 * exp(N(0, 1)) per token (a
    heavy-tailed spread of drifts, so the top 15% is a real selection)."""
    name: str
    n_seq: int
    n_tokens: int
    hidden: int
    dtype: str
    seed: int
    fraction: float = 0.15


def blend_selection(seed=5):
    """64 sequences x 2048 tokens x hidden 4096 (the Qwen3-8B hidden size), bf16."""
    return BlendWorkload("blend_selection", 64, 2048, 4096, "bf16", seed)


def blend_small(seed=6):
    return BlendWorkload("blend_small", 3, 1408, 256, "bf16", seed)


def blend_hidden(w, device, seqs=None):
    """(cached, fresh) [len(seqs), n_tokens, hidden] drawn on `device`; each
    sequence has its own generator seed, so any sequence can be re-drawn."""
    import torch
    seqs = range(w.n_seq) if seqs is None else seqs
    dt = torch_dtype(w.dtype)
    cached = torch.empty((len(seqs), w.n_tokens, w.hidden), dtype=dt, device=device)
    fresh = torch.empty_like(cached)
    for i, s in enumerate(seqs):
        g = torch.Generator(device=device)
        g.manual_seed(w.seed * 1_000_003 + s)
        c = torch.randn((w.n_tokens, w.hidden), generator=g, device=device, dtype=torch.float32)
        sigma = 0.05 * torch.exp(torch.randn((w.n_tokens, 1), generator=g, device=device))
        d = torch.randn((w.n_tokens, w.hidden), generator=g, device=device, dtype=torch.float32) * sigma
        cached[i] = c.to(dt)
        fresh[i] = (c + d).to(dt)
    return cached, fresh
