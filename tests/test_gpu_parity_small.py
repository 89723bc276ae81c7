"""GPU parity on the small workloads and a sweep of shapes, through the C ABI.

Bars (tests/parity.py): codes/scales bit-exact; K within 2e-6 x row max
(fp32) or 1 ulp (+ that floor) for fp16/bf16; V bit-exact (1 ulp for FP8, and
INT4 with fp32 scales, into 16-bit outputs); untouched destination bytes
unchanged.
"""
import zlib

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _assert_ok(rep):
    assert rep["ok"], rep


@pytest.mark.parametrize("wire", ["fp8", "int4", "raw", "fp8_rows"])
def test_tiny(wire):
    _assert_ok(parity.run_small_case("tiny", wire))


@pytest.mark.parametrize("wire,scale_dtype", [("fp8", "f16"), ("int4", "f16"), ("int4", "f32"),
                                              ("raw", "f16"), ("fp8_rows", "f16"),
                                              ("fp8_rows", "f32")])
def test_gqa_reorder(wire, scale_dtype):
    rep = parity.run_small_case("gqa_reorder", wire, scale_dtype=scale_dtype)
    _assert_ok(rep)


SWEEP = [
    # d, B, src, out, pairing, ragged, wire, group, scale
    (128, 16, "bf16", "bf16", "half_split", False, "fp8", 32, "f16"),
    (128, 32, "f16", "f16", "interleaved", True, "fp8", 32, "f16"),
    (128, 64, "bf16", "bf16", "half_split", True, "fp8", 32, "f16"),
    (128, 128, "f32", "f32", "interleaved", True, "fp8", 32, "f16"),
    (64, 16, "f16", "f32", "half_split", True, "fp8", 32, "f16"),
    (64, 64, "f32", "bf16", "interleaved", False, "fp8", 32, "f16"),
    (128, 16, "bf16", "bf16", "half_split", True, "int4", 32, "f16"),
    (128, 64, "f16", "f32", "interleaved", True, "int4", 64, "f32"),
    (128, 32, "f32", "f16", "half_split", False, "int4", 128, "f16"),
    (64, 128, "bf16", "bf16", "interleaved", True, "int4", 64, "f16"),
    (64, 16, "f32", "f32", "half_split", True, "int4", 32, "f32"),
    (128, 64, "bf16", "f32", "half_split", True, "raw", 32, "f16"),
    (64, 32, "f16", "f16", "interleaved", True, "raw", 32, "f16"),
    (128, 16, "bf16", "bf16", "half_split", True, "fp8_rows", 32, "f16"),
    (128, 64, "f16", "f16", "interleaved", True, "fp8_rows", 32, "f32"),
    (64, 32, "bf16", "f32", "half_split", False, "fp8_rows", 32, "f16"),
    (64, 128, "f16", "bf16", "interleaved", True, "fp8_rows", 32, "f16"),
    (128, 32, "f32", "f32", "half_split", True, "fp8_rows", 32, "f16"),
    (64, 16, "f32", "bf16", "interleaved", True, "fp8_rows", 32, "f32"),
]


@pytest.mark.parametrize("d,B,src,out,pairing,ragged,wire,group,scale", SWEEP)
def test_shape_sweep(d, B, src, out, pairing, ragged, wire, group, scale):
    seed = zlib.crc32(repr((d, B, src, out, pairing, ragged, wire, group, scale)).encode())
    c = parity.random_case(seed, L=2, H=3, d=d, B=B, nb=7, src_fmt=src, out_fmt=out,
                           pairing=pairing, ragged=ragged)
    if wire == "raw":
        c.src_fmt = out
        c.src_k, c.src_v = parity.round_to(c.src_k, out), parity.round_to(c.src_v, out)
    _assert_ok(parity.run_case(c, wire, group=group, scale_dtype=scale))


# ---------------------------------------------------------------- adversarial values
def _midpoint_case(seed, wire):
    """Slabs whose quotients x/s land within a few fp32 ulps of every E4M3
    rounding midpoint (FP8) or half-integer (INT4), with a non-trivial scale."""
    from oracle import fp8
    r = np.random.default_rng(seed)
    c = parity.random_case(seed, L=1, H=2, d=128, B=16, nb=4, src_fmt="f32", out_fmt="f32")
    mags = fp8.e4m3_table()[:0x7E]                   # every finite magnitude below 448
    if wire in ("fp8", "fp8_rows"):
        targets, amax_q = np.concatenate([(mags[:-1] + mags[1:]) / 2, mags]), 448.0
    else:
        targets, amax_q = np.arange(-13, 14) / 2.0, 7.0
    n = c.B * c.d
    for slot in c.src_slots:
        for pool in (c.src_k, c.src_v):
            for h in range(c.H):
                s_target = np.float32(np.exp(r.uniform(-6, 6)))
                x = (r.choice(targets, size=n) * r.choice([-1.0, 1.0], size=n)).astype(np.float32)
                x = x * s_target
                walk = r.integers(-3, 4, size=n)     # move up to 3 fp32 ulps either way
                for _ in range(3):
                    step = np.sign(walk)
                    toward = np.where(step > 0, np.float32(np.inf), np.float32(-np.inf))
                    x = np.where(walk != 0, np.nextafter(x, toward), x)
                    walk = walk - step
                x[0] = np.float32(amax_q) * s_target   # pins the slab / group / row amax
                if wire == "int4":
                    x.reshape(c.B, c.d // 32, 32)[:, :, 0] = np.float32(amax_q) * s_target
                if wire == "fp8_rows":
                    x.reshape(c.B, c.d)[:, 0] = np.float32(amax_q) * s_target
                pool[0, slot, :, h, :] = x.astype(np.float64).reshape(c.B, c.d)
    return c


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
@pytest.mark.parametrize("seed", [11, 12])
def test_midpoint_adversarial(wire, seed):
    c = _midpoint_case(seed, wire)
    _assert_ok(parity.run_case(c, wire, scale_dtype="f32"))


def test_zero_slab_signed_zero_and_tiny():
    c = parity.random_case(21, L=1, H=2, d=64, B=16, nb=3, src_fmt="f32", out_fmt="f32")
    s0 = c.src_slots[0]
    c.src_k[0, s0] = 0.0                       # all-zero slab: scale 0, codes 0
    c.src_v[0, s0] = -0.0
    s1 = c.src_slots[1]
    c.src_k[0, s1, :, :, :8] = -0.0            # -0 next to non-zeros: 0x80
    c.src_k[0, s1, :, :, 8:16] = -1e-30        # underflows to -0: 0x80
    for wire in ("fp8", "int4", "fp8_rows"):
        _assert_ok(parity.run_case(c, wire))


@pytest.mark.parametrize("fmt,big", [("f16", 65504.0), ("bf16", 3.0e38), ("f32", 3.0e38)])
def test_large_magnitudes(fmt, big):
    c = parity.random_case(31, L=1, H=1, d=128, B=16, nb=2, src_fmt=fmt, out_fmt="f32", scale=1.0)
    c.src_k[0, c.src_slots[0], 3, 0, 5] = parity.round_to(np.array(big), fmt)
    c.src_v[0, c.src_slots[1], 0, 0, 0] = parity.round_to(np.array(-big), fmt)
    _assert_ok(parity.run_case(c, "fp8"))
    _assert_ok(parity.run_case(c, "int4", scale_dtype="f32"))
    _assert_ok(parity.run_case(c, "fp8_rows", scale_dtype="f32"))


@pytest.mark.parametrize("fmt", ["bf16", "f32"])
def test_fp8_rows_scale_overflow_encode(fmt):
    """A row whose fp16 scale overflows (amax above 65504 * 448) stores +inf
    and the codes of x / inf = +-0; compared on the encode side (the decode of
    such a row is 0 * inf = NaN on both sides)."""
    c = parity.random_case(33, L=1, H=2, d=128, B=16, nb=2, src_fmt=fmt, out_fmt="f32")
    c.src_k[0, c.src_slots[0], 4, 1, 9] = parity.round_to(np.array(3.0e38), fmt)
    c.src_v[0, c.src_slots[1], 0, 0, 0] = parity.round_to(np.array(-4.0e7), fmt)
    o = parity.oracle_run(c, "fp8_rows", scale_dtype="f16")
    g = parity.gpu_run(c, "fp8_rows", scale_dtype="f16")
    assert np.isinf(o["scales"]).sum() == 2
    assert g["err"] == 0
    assert np.array_equal(g["codes"], o["codes"])
    assert np.array_equal(g["scales"], o["scales"])


# ---------------------------------------------------------------- extreme shapes
@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows", "raw"])
def test_many_heads_one_block(wire):
    """32 KV heads, 128-token blocks, a single block whose n_valid is 1: a
    unit of 8 sub-slabs is one head's slab, and all but one row is padding."""
    c = parity.random_case(71, L=1, H=32, d=64, B=128, nb=1, src_fmt="bf16", out_fmt="bf16",
                           pairing="interleaved")
    c.n_valid = np.array([1], dtype=np.int32)
    if wire == "raw":
        c.src_k, c.src_v = parity.round_to(c.src_k, "bf16"), parity.round_to(c.src_v, "bf16")
    _assert_ok(parity.run_case(c, wire))


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
def test_one_head_many_blocks(wire):
    """One KV head: a unit of 8 sub-slabs spans four blocks (two slabs each),
    with ragged tails and a mix of delta-m values."""
    c = parity.random_case(72, L=3, H=1, d=128, B=16, nb=53, src_fmt="f16", out_fmt="f16",
                           pairing="half_split", ragged=True, extra_slots=11)
    _assert_ok(parity.run_case(c, wire))


# ---------------------------------------------------------------- error paths
def _tiny_path(wire="fp8", **over):
    from kv_cache_quantization_hc_gb300 import path as kvpath
    c = parity.random_case(41, L=1, H=2, d=64, B=16, nb=4, src_fmt="f32", out_fmt="f32")
    args = dict(n_layers=1, H=2, d=64, B=16, n_blocks=4, src_slots=c.src_slots,
                dst_slots=c.dst_slots, n_valid=c.n_valid, delta_m_distinct=np.array([0, 5]),
                delta_idx=np.array([0, 1, 0, 1]), wire=wire, pairing="interleaved",
                rope_base=1e4, paged_dtype="f32")
    args.update(over)
    p = kvpath.KVPath(**args)
    src_k = torch.as_tensor(c.src_k, device="cuda").float()
    src_v = torch.as_tensor(c.src_v, device="cuda").float()
    return c, p, src_k, src_v


@pytest.mark.parametrize("bad,bit", [("slot", 1), ("nvalid", 4)])
def test_device_error_flag_encode_skips_block(bad, bit):
    c, p, k, v = _tiny_path()
    if bad == "slot":
        p.src_slots[2] = c.num_dst_slots + 100
    else:
        p.n_valid = torch.as_tensor(np.array([16, 16, 0, 16], np.int32), device="cuda")
    p.codes.fill_(0xAB)
    p.encode(k, v)
    torch.cuda.synchronize()
    assert p.error_bits() == bit
    codes = p.codes.cpu().numpy()
    assert np.all(codes[:, 2] == 0xAB)               # the bad block was skipped
    from oracle import paged
    want, _ = paged.encode_fp8(c.src_k, c.src_v, c.src_slots[[0, 1, 3]])
    assert np.array_equal(codes[:, [0, 1, 3]], want)


@pytest.mark.parametrize("wire", ["fp8", "int4"])
@pytest.mark.parametrize("bad,bit", [("slot", 1), ("delta", 2), ("nvalid", 4)])
def test_device_error_flag_fetch_skips_block(bad, bit, wire):
    """A bad destination slot, delta-m index or n_valid flags its bit and skips
    the block's K and V; every other block is written.  The INT4 fetch takes K
    and V of a sub-slab in one warp, so both are checked there too."""
    c, p, k, v = _tiny_path(wire)
    p.encode(k, v)
    p.build_table()
    if bad == "slot":
        p.dst_slots[1] = -1
    elif bad == "delta":
        p.delta_idx[1] = 2
    else:
        p.n_valid = torch.as_tensor(np.array([16, 17, 16, 16], np.int32), device="cuda")
    dk = torch.full((1, c.num_dst_slots, 16, 2, 64), parity.SENTINEL, device="cuda")
    dv = dk.clone()
    p.fetch(dk, dv)
    torch.cuda.synchronize()
    assert p.error_bits() == bit
    good = {int(c.dst_slots[j]) for j in (0, 2, 3)}
    for slot in range(c.num_dst_slots):   # the bad block's slot and unused slots keep the sentinel
        for t in (dk, dv):
            if slot in good:
                assert not torch.any(t[0, slot] == parity.SENTINEL)
            else:
                assert torch.all(t[0, slot] == parity.SENTINEL)


def test_empty_call_is_a_no_op():
    from kv_cache_quantization_hc_gb300 import hc
    c, p, k, v = _tiny_path()
    p.codes.fill_(7)
    hc.hc_encode_fp8(k, v, hc.paged_desc(k), p.src_slots, None, 0, p.codes, p.scales, p.err)
    hc.hc_fetch_rotate_scatter(hc.HC_WIRE_FP8, p.codes, p.scales, 32, hc.HC_F16, p.table, p.delta_idx,
                               0, 0, p.dst_slots, None, 0, k, v, hc.paged_desc(k), p.err)
    hc.hc_build_delta_sincos(p.delta_m, 0, 64, 1e4, None, p.table)
    torch.cuda.synchronize()
    assert p.error_bits() == 0 and torch.all(p.codes == 7)


def test_host_argument_errors():
    from kv_cache_quantization_hc_gb300 import hc
    c, p, k, v = _tiny_path()
    desc = hc.paged_desc(k)

    def status(fn, *a):
        try:
            fn(*a)
            return 0
        except hc.HCError as e:
            return e.status

    enc = lambda **o: status(hc.hc_encode_fp8, o.get("k", k), v, o.get("desc", desc), p.src_slots,
                             None, o.get("nb", 4), o.get("codes", p.codes), p.scales, p.err)
    assert enc(k=None) == hc.HC_ERR_INVALID_ARG
    assert enc(nb=-1) == hc.HC_ERR_INVALID_ARG
    assert enc(codes=p.codes.data_ptr() + 1) == hc.HC_ERR_INVALID_ARG
    bad = hc.hc_paged_desc(1, 2, 96, 16, desc.num_slots, hc.HC_F32, desc.slot_stride, 0)
    assert enc(desc=bad) == hc.HC_ERR_UNSUPPORTED
    bad = hc.hc_paged_desc(1, 2, 64, 24, desc.num_slots, hc.HC_F32, desc.slot_stride, 0)
    assert enc(desc=bad) == hc.HC_ERR_UNSUPPORTED
    bad = hc.hc_paged_desc(1, 2, 64, 16, desc.num_slots, 7, desc.slot_stride, 0)
    assert enc(desc=bad) == hc.HC_ERR_INVALID_ARG
    bad = hc.hc_paged_desc(1, 2, 64, 16, desc.num_slots, hc.HC_F32, 100, 0)
    assert enc(desc=bad) == hc.HC_ERR_INVALID_ARG
    assert status(hc.hc_encode_int4, k, v, desc, p.src_slots, None, 4, 48, hc.HC_F16, p.codes,
                  p.scales, p.err) == hc.HC_ERR_UNSUPPORTED
    assert status(hc.hc_encode_int4, k, v, desc, p.src_slots, None, 4, 128, hc.HC_F16, p.codes,
                  p.scales, p.err) == hc.HC_ERR_UNSUPPORTED          # group > d_head
    assert status(hc.hc_fetch_rotate_scatter, 9, p.codes, p.scales, 32, hc.HC_F16, p.table,
                  p.delta_idx, 2, 0, p.dst_slots, None, 4, k, v, desc, p.err) == hc.HC_ERR_INVALID_ARG
    assert status(hc.hc_fetch_rotate_scatter, hc.HC_WIRE_FP8, p.codes, p.scales, 32, hc.HC_F16,
                  p.table, p.delta_idx, 0, 0, p.dst_slots, None, 4, k, v, desc,
                  p.err) == hc.HC_ERR_INVALID_ARG                     # n_distinct 0
    assert status(hc.hc_build_delta_sincos, p.delta_m, 2, 63, 1e4, None, p.table) == hc.HC_ERR_INVALID_ARG
    assert status(hc.hc_build_delta_sincos, p.delta_m, 2, 64, -1.0, None, p.table) == hc.HC_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert p.error_bits() == 0


def test_table_with_inv_freq_override():
    from kv_cache_quantization_hc_gb300 import hc
    from oracle import paged
    th = np.linspace(1.0, 1e-4, 64)
    dm = np.array([-8192, -1, 0, 3, 4096, 65535], np.int32)
    t = torch.zeros((6, 64, 2), device="cuda")
    hc.hc_build_delta_sincos(torch.as_tensor(dm, device="cuda"), 6, 128, 0.0,
                             torch.as_tensor(th, device="cuda"), t)
    want = paged.delta_sincos_table(dm, th)
    got = t.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= parity.ulp(want, "f32"))


def _tie_case(fmt, seed):
    """Slabs whose amax sweeps the format's mantissas and whose elements sweep
    all mantissas over several binades: with 16-bit values many quotients
    x/s land exactly on E4M3 midpoints (e.g. x = 3/4 amax -> 336)."""
    from oracle.numerics import FORMATS
    p_bits = FORMATS[fmt][0] - 1
    r = np.random.default_rng(seed)
    H, d, B = 1, 128, 16
    mant = np.arange(1 << p_bits)
    amax_m = mant if fmt == "bf16" else r.choice(mant, 128, replace=False)
    nb = len(amax_m)
    c = parity.random_case(seed, L=1, H=H, d=d, B=B, nb=nb, src_fmt=fmt, out_fmt="f32", extra_slots=0)
    for j, m in enumerate(amax_m):
        amax = (1.0 + m / (1 << p_bits)) * 2.0 ** int(r.integers(-3, 4))
        xs_m = r.choice(mant, B * d)
        xs = (1.0 + xs_m / (1 << p_bits)) * amax / 2.0 ** r.integers(0, 9, B * d)
        xs = parity.round_to(np.minimum(xs, amax) * r.choice([-1.0, 1.0], B * d), fmt)
        xs[0] = amax
        for pool in (c.src_k, c.src_v):
            pool[0, c.src_slots[j], :, 0, :] = xs.reshape(B, d)
    return c


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_exact_ties_16bit(fmt):
    c = _tie_case(fmt, 51)
    _assert_ok(parity.run_case(c, "fp8"))
    _assert_ok(parity.run_case(c, "int4", scale_dtype="f16"))
    _assert_ok(parity.run_case(c, "int4", scale_dtype="f32"))
    _assert_ok(parity.run_case(c, "fp8_rows", scale_dtype="f16"))
    _assert_ok(parity.run_case(c, "fp8_rows", scale_dtype="f32"))


@pytest.mark.parametrize("wire", ["fp8", "raw"])
@pytest.mark.parametrize("pairing", ["half_split", "interleaved"])
def test_extreme_delta_m(wire, pairing):
    """Delta-m at the ends of its int32 range: the table's fp64 angles reach
    2^31 rad (large-argument reduction in both the kernel's sincos and the
    oracle's), and the rotated keys still meet the bars."""
    c = parity.random_case(4242, L=1, H=2, d=128, B=16, nb=7, src_fmt="f32", out_fmt="f32",
                           pairing=pairing)
    c.delta_m = np.array([0, 1, -1, 1 << 30, -(1 << 30), (1 << 31) - 1, -(1 << 31)], np.int64)
    _assert_ok(parity.run_case(c, wire))


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
def test_shared_source_slots_and_single_rows(wire):
    """Several blocks gathered from the same source slot (only destinations
    must be distinct), every block valid for a single row: the amax, the
    scale and the codes come from that row alone."""
    c = parity.random_case(515, L=2, H=3, d=128, B=16, nb=6, src_fmt="bf16", out_fmt="bf16",
                           pairing="half_split")
    c.src_slots = np.array([2, 2, 5, 2, 5, 0], np.int32)
    c.n_valid = np.ones(6, np.int32)
    _assert_ok(parity.run_case(c, wire))
