"""The full-size parity checker (tests/full_parity.py) on the CPU: a chunk
whose "GPU" outputs are the oracle's own passes, and each kind of fault the
checker exists to catch is caught - a wrong code byte, a wrong scale, blocks
placed in each other's slots, a stray write into a padding row, a V value
off by more than the bar.  The worker pool runs two spawned processes."""
import numpy as np
import pytest

from oracle import paged, rope
from oracle.numerics import round_to
from tests import full_parity as fp


def _bits(a):
    return (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _chunk(wire, seed=0, n=4, B=16, H=2, d=64):
    r = np.random.default_rng(seed)
    k = round_to(r.standard_normal((1, n, B, H, d)), "bf16")
    v = round_to(r.standard_normal((1, n, B, H, d)), "bf16")
    nv = np.array([B, 5, B, 1][:n])
    dm = r.integers(-9000, 9000, n)
    ids = np.arange(n)
    if wire == "fp8":
        oc, osc = paged.encode_fp8(k, v, ids, nv)
        vals = paged.decode_fp8(oc, osc)
        sc = osc.astype(np.float32)
    else:
        oc, osc = paged.encode_int4(k, v, ids, nv, 32, "f16")
        vals = paged.decode_int4(oc, osc, 32)
        sc = osc.astype(np.float16)
    th = rope.inv_freq(d, 1e6)
    sent = np.full((1, n, B, H, d), fp.SENTINEL)
    ek, ev = paged.fetch_rotate_scatter(vals, dm, th, "half_split", ids, sent, sent, "bf16", n_valid=nv)
    return dict(label=("host", 0, n), wire=wire, src_fmt="bf16", out_fmt="bf16",
                src_k=_bits(k), src_v=_bits(v), codes=oc, scales=sc,
                dst_k=_bits(ek), dst_v=_bits(ev), n_valid=nv, delta_m=dm, d=d, rope_base=1e6,
                pairing="half_split", group=32, scale_dtype="f16")


@pytest.mark.parametrize("wire", ["fp8", "int4"])
def test_checker_accepts_the_oracle_and_rejects_faults(wire):
    t = _chunk(wire)
    assert fp.check_chunk(t)["ok"]

    bad = dict(t, codes=t["codes"].copy())
    bad["codes"][0, 2, 1, 0, 3, 7] ^= 0x01
    r = fp.check_chunk(bad)
    assert not r["ok"] and not r["codes_ok"] and r["codes_bad"] == 1

    bad = dict(t, scales=t["scales"].copy())
    bad["scales"].flat[5] = np.nextafter(bad["scales"].flat[5], np.inf, dtype=bad["scales"].dtype)
    assert not fp.check_chunk(bad)["scales_ok"]

    swapped = dict(t, dst_k=t["dst_k"][:, [2, 1, 0, 3]].copy())    # blocks 0 and 2 placed in each other's slots
    r = fp.check_chunk(swapped)
    assert not r["ok"] and not r["k_ok"]

    stray = dict(t, dst_v=t["dst_v"].copy())
    stray["dst_v"][0, 1, 9, 0, 0] = _bits(np.array(1.0))            # block 1 holds 5 valid rows
    r = fp.check_chunk(stray)
    assert not r["ok"] and not r["padding_ok"] and r["v_ok"]

    off = dict(t, dst_v=t["dst_v"].copy())
    off["dst_v"][0, 0, 0, 0, 0] += 2                                # 2 bf16 ulps
    assert not fp.check_chunk(off)["v_ok"]


def test_pool_runs_chunks_in_spawned_processes():
    with fp.OraclePool(procs=2, window=2) as pool:
        for s in range(5):
            pool.submit(_chunk("fp8", seed=s))
        res = pool.results()
        assert len(res) == 5 and all(r["ok"] for r in res)
        bad = _chunk("int4", seed=9)
        bad["codes"] = bad["codes"].copy()
        bad["codes"][0, 0, 0, 0, 0, 0] ^= 0x10
        pool.submit(bad)
        s = fp.summarize(pool.results())
        assert s["chunks"] == 1 and len(s["failed"]) == 1
