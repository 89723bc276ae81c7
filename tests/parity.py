"""Parity machinery shared by the GPU tests and the smoke check.

A ``Case`` is a set of host inputs (float64 arrays holding values exact in the
source dtype).  ``run_case`` feeds the same inputs to the oracle and, through
the C ABI, to the CUDA path, and compares:

* wire codes and scales: bit-exact;
* rotation table: within 1 fp32 ulp (both sides round fp64 cos/sin once);
* fetched K: fp32 output within 2e-6 x the row's max |k|; fp16/bf16 output
  within 1 ulp of the larger of the two values, plus the same 2e-6 x row-max
  floor (below it the fp32 rotation's own rounding decides the last bit);
* fetched V: bit-exact, except where the fp32 dequantized value is rounded
  a second time to fp16/bf16 (FP8-sourced V, and INT4 with fp32 scales;
  within 1 ulp);
* every element the fetch must not touch keeps its sentinel, bit for bit.
"""
from dataclasses import dataclass

import numpy as np
import torch

import workloads
from oracle import paged, rope
from oracle.numerics import round_to, ulp
from tests.bars import K_REL, SENTINEL, compare_k, compare_v  # noqa: F401

_TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Case:
    name: str
    L: int
    H: int
    d: int
    B: int
    src_fmt: str
    out_fmt: str
    pairing: str
    rope_base: float
    src_k: np.ndarray             # [L, S_src, B, H, d]
    src_v: np.ndarray
    src_slots: np.ndarray
    dst_slots: np.ndarray
    n_valid: np.ndarray
    delta_m: np.ndarray
    num_dst_slots: int


def case_from_workload(name):
    """Small workload: cache post-RoPE keys at m_old (oracle RoPE), round to
    the source dtype, and place block j at slot src_slots[j]; the other slots
    hold unrelated draws that the encode must never read."""
    w, draws = workloads.WORKLOADS[name]()
    blk, dr = w.blocks[0], draws[0]
    th = rope.inv_freq(w.d, w.rope_base)
    src_k = round_to(dr.filler_src, w.src_dtype)
    src_v = round_to(dr.filler_src[:, ::-1].copy(), w.src_dtype)
    for j in range(blk.nb):
        for layer in range(w.L):
            k_old = rope.apply_rope(dr.k_pre[layer, j], dr.m_old[j], th, w.pairing)
            src_k[layer, blk.src_slots[j]] = round_to(k_old, w.src_dtype)
            src_v[layer, blk.src_slots[j]] = round_to(dr.v[layer, j], w.src_dtype)
    return Case(name, w.L, w.H, w.d, blk.B, w.src_dtype, w.out_dtype, w.pairing, w.rope_base,
                src_k, src_v, blk.src_slots, blk.dst_slots, blk.n_valid, blk.delta_m,
                blk.num_dst_slots)


def random_case(seed, L=2, H=3, d=128, B=16, nb=5, src_fmt="bf16", out_fmt="bf16",
                pairing="half_split", ragged=False, rope_base=1e4, scale=1.0, extra_slots=3):
    r = np.random.default_rng(seed)
    S = nb + extra_slots
    src_k = round_to(r.standard_normal((L, S, B, H, d)) * scale, src_fmt)
    src_v = round_to(r.standard_normal((L, S, B, H, d)) * scale, src_fmt)
    nv = r.integers(1, B, size=nb, endpoint=True) if ragged else np.full(nb, B)
    return Case(f"random{seed}", L, H, d, B, src_fmt, out_fmt, pairing, rope_base, src_k, src_v,
                r.permutation(S)[:nb].astype(np.int32), r.permutation(S)[:nb].astype(np.int32),
                nv.astype(np.int32), r.integers(-20000, 20000, size=nb).astype(np.int64), S)


# ------------------------------------------------------------------ oracle side
def oracle_run(c, wire, group=32, scale_dtype="f16"):
    th = rope.inv_freq(c.d, c.rope_base)
    out = {}
    if wire == "fp8":
        codes, scales = paged.encode_fp8(c.src_k, c.src_v, c.src_slots, c.n_valid)
        vals = paged.decode_fp8(codes, scales)
    elif wire == "int4":
        codes, scales = paged.encode_int4(c.src_k, c.src_v, c.src_slots, c.n_valid, group, scale_dtype)
        vals = paged.decode_int4(codes, scales, group)
    elif wire == "fp8_rows":
        codes, scales = paged.encode_fp8_rows(c.src_k, c.src_v, c.src_slots, c.n_valid, scale_dtype)
        vals = paged.decode_fp8_rows(codes, scales)
    else:
        codes, scales = None, None
        vals = paged.gather_slabs(c.src_k, c.src_v, c.src_slots)
    out["codes"], out["scales"] = codes, scales
    dm_vals, _ = np.unique(c.delta_m, return_inverse=True)
    out["table"] = paged.delta_sincos_table(dm_vals, th)
    sent = np.full((c.L, c.num_dst_slots, c.B, c.H, c.d), SENTINEL)
    out["k"], out["v"] = paged.fetch_rotate_scatter(vals, c.delta_m, th, c.pairing, c.dst_slots,
                                                    sent, sent, c.out_fmt, n_valid=c.n_valid)
    return out


# ------------------------------------------------------------------ CUDA side
def gpu_run(c, wire, group=32, scale_dtype="f16", device="cuda"):
    from kv_cache_quantization_hc_gb300 import path as kvpath

    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p = kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots),
                      src_slots=c.src_slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                      delta_m_distinct=dm_vals, delta_idx=dm_idx, wire=wire, pairing=c.pairing,
                      rope_base=c.rope_base, paged_dtype=c.out_fmt, group=group,
                      scale_dtype=scale_dtype, device=device)
    src_k = torch.as_tensor(c.src_k, device=device).to(_TORCH[c.src_fmt])
    src_v = torch.as_tensor(c.src_v, device=device).to(_TORCH[c.src_fmt])
    dst_shape = (c.L, c.num_dst_slots, c.B, c.H, c.d)
    dst_k = torch.full(dst_shape, SENTINEL, dtype=_TORCH[c.out_fmt], device=device)
    dst_v = torch.full(dst_shape, SENTINEL, dtype=_TORCH[c.out_fmt], device=device)
    if wire == "raw":
        # the unquantized wire holds the cached blocks in wire order, in the paged dtype
        sl = torch.as_tensor(np.asarray(c.src_slots, np.int64), device=device)
        kv = torch.stack([src_k[:, sl], src_v[:, sl]], dim=2)          # [L, NB, 2, B, H, d]
        p.codes.copy_(kv.permute(0, 1, 2, 4, 3, 5).to(p.codes.dtype))
    else:
        p.encode(src_k, src_v)
    p.build_table()
    p.fetch(dst_k, dst_v)
    torch.cuda.synchronize(device)
    to64 = lambda t: None if t is None else t.double().cpu().numpy()
    return {"codes": None if wire == "raw" else p.codes.cpu().numpy(),
            "scales": to64(p.scales) if wire != "raw" else None,
            "table": to64(p.table)[:len(dm_vals)], "k": to64(dst_k), "v": to64(dst_v),
            "err": p.error_bits()}


# ------------------------------------------------------------------ comparison
def written_mask(c):
    m = np.zeros((c.L, c.num_dst_slots, c.B), bool)
    for j, s in enumerate(c.dst_slots):
        m[:, s, :c.n_valid[j]] = True
    return m


def compare_outputs(c, wire, gout, oout, scale_dtype="f16"):
    rep = {}
    m = written_mask(c)
    for name in ("k", "v"):
        untouched_ok = np.array_equal(gout[name][~m], oout[name][~m])
        rep[f"{name}_untouched_ok"] = bool(untouched_ok)
    ok_k, kerr, kbar = compare_k(gout["k"][m], oout["k"][m], c.out_fmt)
    rep.update(k_ok=ok_k, k_max_err=kerr, k_bar=kbar)
    rep["v_ok"], rep["v_exact"] = compare_v(gout["v"][m], oout["v"][m], wire, c.out_fmt, scale_dtype)
    return rep


def run_case(c, wire, group=32, scale_dtype="f16", device="cuda"):
    o = oracle_run(c, wire, group, scale_dtype)
    g = gpu_run(c, wire, group, scale_dtype, device)
    rep = {"err": g["err"]}
    if wire != "raw":
        rep["codes_exact"] = bool(np.array_equal(g["codes"], o["codes"]))
        rep["scales_exact"] = bool(np.array_equal(g["scales"], o["scales"]))
        if not rep["codes_exact"]:
            bad = np.argwhere(g["codes"] != o["codes"])
            rep["codes_mismatch"] = int(len(bad))
            i = tuple(bad[0])
            rep["first_code_mismatch"] = (i, int(g["codes"][i]), int(o["codes"][i]))
    t_ulp = ulp(o["table"], "f32")
    rep["table_ok"] = bool(np.all(np.abs(g["table"] - o["table"]) <= t_ulp))
    rep["table_exact"] = bool(np.array_equal(g["table"], o["table"]))
    rep.update(compare_outputs(c, wire, g, o, scale_dtype))
    rep["ok"] = (rep["err"] == 0 and rep.get("codes_exact", True) and rep.get("scales_exact", True)
                 and rep["table_ok"] and rep["k_ok"] and rep["v_ok"]
                 and rep["k_untouched_ok"] and rep["v_untouched_ok"])
    return rep


def run_small_case(name, wire, device="cuda", **kw):
    return run_case(case_from_workload(name), wire, device=device, **kw)
