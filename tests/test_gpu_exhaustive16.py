"""Every 16-bit input pair through the library's encode kernels.

For fp16 and for bf16 sources, each positive finite value `a` is used as a
group's (INT4) or slab's (FP8) absolute maximum, together with every value x
with |x| <= a (both signs): about 1.0e9 (x, amax) pairs per format.  The codes
and scales the C-ABI kernels write are compared, bit for bit, with IEEE fp32
arithmetic done by torch on the GPU:

  FP8:  s = fp32(a / 448),  code = float8_e4m3fn(fp32(x / s))  (RNE; |q| stays
        below 464, so the cast needs no saturation); per slab, and per row
        with fp16 or fp32 scales
  INT4: s = fp16(fp32(a / 7)), code = round_half_even(fp32(x / s)) in [-7, 7]
        (an fp16 scale that overflows to +inf gives x / s = 0)

Every division is tensor by tensor: torch turns a division by a Python
scalar into a multiplication by its reciprocal, which is not the IEEE
quotient (it misses fp16 ties such as amax / 7 = 6.5 * 2^-24).

This covers the kernels' division-free quotient paths for 16-bit sources (the
residual-corrected quotient, for FP8 and for INT4) and the IEEE-division
paths they hand tiny or overflowing scales to, on the whole 16-bit input
domain.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _magnitudes(fmt):
    """All non-negative finite values of the format, ascending (float32)."""
    bits = torch.arange(0, 0x8000, dtype=torch.int32, device=DEV).to(torch.int16)
    v = bits.view(TDT[fmt]).float()
    v = v[torch.isfinite(v)]
    return torch.sort(v).values


def _pairs(mags, ia0, ia1, per):
    """Groups of `per` elements for amax indices [ia0, ia1): element 0 is the
    amax, the others run through +mags[0..ia], then -mags[0..ia]."""
    dev = mags.device
    ia = torch.arange(ia0, ia1, device=dev, dtype=torch.int64)
    n_signed = 2 * (ia + 1)
    n_groups = (n_signed + per - 2) // (per - 1)
    gi = torch.repeat_interleave(torch.arange(len(ia), device=dev), n_groups)
    start = torch.cumsum(n_groups, 0) - n_groups
    first = (torch.arange(len(gi), device=dev) - start[gi]) * (per - 1)
    pos = first[:, None] + torch.arange(per - 1, device=dev)[None, :]
    pos = torch.minimum(pos, n_signed[gi][:, None] - 1)
    iag = ia[gi][:, None]
    mag = mags[torch.where(pos <= iag, pos, pos - iag - 1)]
    val = torch.where(pos <= iag, mag, -mag)
    amax = mags[ia[gi]][:, None]
    return torch.cat([amax, val], dim=1)                      # [groups, per] float32


def _chunks(n, step):
    for a in range(1, n, step):
        yield a, min(n, a + step)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_int4_all_pairs(fmt):
    from kv_cache_quantization_hc_gb300 import hc
    mags = _magnitudes(fmt)
    B, H, d, g = 16, 8, 128, 32
    per_slot = B * H * d // g                                  # groups per slot
    checked = 0
    for ia0, ia1 in _chunks(len(mags), 1024):
        grp = _pairs(mags, ia0, ia1, g)
        ng = grp.shape[0]
        nslots = (ng + per_slot - 1) // per_slot
        flat = torch.zeros((nslots * per_slot, g), device=DEV)
        flat[:ng] = grp
        src = flat.to(TDT[fmt]).reshape(1, nslots, B, H, d)
        assert torch.equal(src.float().reshape(-1, g)[:ng], grp)  # exactly representable
        codes = torch.empty((1, nslots, 2, H, B, d // 2), dtype=torch.uint8, device=DEV)
        scales = torch.empty((1, nslots, 2, H, B, d // g), dtype=torch.float16, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        slots = torch.arange(nslots, dtype=torch.int32, device=DEV)
        hc.hc_encode_int4(src, src, hc.paged_desc(src), slots, None, nslots, g, hc.HC_F16,
                          codes, scales, err)
        # reference, in the source's [slot, t, h, group] order
        x = src.float().reshape(nslots, B, H, d // g, g)
        am = x.abs().amax(-1, keepdim=True)
        s = (am / torch.full_like(am, 7.0)).half().float()   # tensor / tensor: IEEE division
        q = torch.where(s > 0, x / s, torch.zeros_like(x))
        want = torch.round(q).clamp(-7, 7).to(torch.int8)
        got_c = codes[0, :, 0].permute(0, 2, 1, 3).reshape(nslots, B, H, d // 2)
        lo = (got_c & 0xF).to(torch.int8)
        hi = (got_c >> 4).to(torch.int8)
        got = torch.stack([lo, hi], -1).reshape(nslots, B, H, d // g, g)
        got = torch.where(got >= 8, got - 16, got)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        bad = (got != want).reshape(-1, g)[:ng].any(-1)
        assert not bool(bad.any()), (fmt, int(bad.sum()))
        got_s = scales[0, :, 0].permute(0, 2, 1, 3).reshape(nslots, B, H, d // g)
        assert torch.equal(got_s.float(), s[..., 0])
        checked += ng * (g - 1)
    assert checked > 1.0e9


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_fp8_all_pairs(fmt):
    from kv_cache_quantization_hc_gb300 import hc
    mags = _magnitudes(fmt)
    B, H, d = 16, 8, 128
    slab = B * d
    checked = 0
    for ia0, ia1 in _chunks(len(mags), 2048):
        grp = _pairs(mags, ia0, ia1, slab)                      # one slab per group
        ns = grp.shape[0]
        nslots = (ns + H - 1) // H
        flat = torch.zeros((nslots * H, slab), device=DEV)
        flat[:ns] = grp
        del grp
        # slab (slot, h) holds the rows t of head h: paged [slot, t, h, c]
        src = flat.reshape(nslots, H, B, d).permute(0, 2, 1, 3).contiguous().to(TDT[fmt])
        src = src.reshape(1, nslots, B, H, d)
        codes = torch.empty((1, nslots, 2, H, B, d), dtype=torch.uint8, device=DEV)
        scales = torch.empty((1, nslots, 2, H), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        slots = torch.arange(nslots, dtype=torch.int32, device=DEV)
        hc.hc_encode_fp8(src, src, hc.paged_desc(src), slots, None, nslots, codes, scales, err)
        x = flat.to(TDT[fmt]).float().reshape(nslots, H, slab)
        am = x.abs().amax(-1, keepdim=True)
        s = am / torch.full_like(am, 448.0)                   # tensor / tensor: IEEE division
        q = torch.where(s > 0, x / s, torch.zeros_like(x))
        want = q.to(torch.float8_e4m3fn).view(torch.uint8)
        want = torch.where(s > 0, want, torch.zeros_like(want))
        got = codes[0, :, 0].reshape(nslots, H, slab)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        bad = (got != want).reshape(-1, slab)[:ns].any(-1)
        assert not bool(bad.any()), (fmt, int(bad.sum()))
        assert torch.equal(scales[0, :, 0], s[..., 0])
        checked += ns * (slab - 1)
    assert checked > 1.0e9


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("scale", ["f16", "f32"])
def test_fp8_rows_all_pairs(fmt, scale):
    """Row-scaled FP8: each (token, head) row of 128 channels holds one amax
    and 127 values x with |x| <= amax.  Reference: s32 = fp32(a / 448), s =
    fp16(s32) or s32, code = float8_e4m3fn(clamp(fp32(x / s), +-448)): an
    fp16-subnormal scale can be well below a / 448, and torch's cast turns
    values past 448 into NaN, so the reference saturates first (clamping, then
    rounding, is the satfinite rounding).  A scale of 0 gives codes 0, a scale
    that overflows fp16 (+inf) gives the codes of x / inf = +-0."""
    from kv_cache_quantization_hc_gb300 import hc
    mags = _magnitudes(fmt)
    B, H, d = 16, 8, 128
    per_slot = B * H
    checked = 0
    for ia0, ia1 in _chunks(len(mags), 2048):
        grp = _pairs(mags, ia0, ia1, d)                         # one row per group
        nr = grp.shape[0]
        nslots = (nr + per_slot - 1) // per_slot
        flat = torch.zeros((nslots * per_slot, d), device=DEV)
        flat[:nr] = grp
        del grp
        src = flat.to(TDT[fmt]).reshape(1, nslots, B, H, d)     # row (slot, t, h)
        codes = torch.empty((1, nslots, 2, H, B, d), dtype=torch.uint8, device=DEV)
        sdt = torch.float16 if scale == "f16" else torch.float32
        scales = torch.empty((1, nslots, 2, H, B), dtype=sdt, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        slots = torch.arange(nslots, dtype=torch.int32, device=DEV)
        hc.hc_encode_fp8_rows(src, src, hc.paged_desc(src), slots, None, nslots,
                              hc.HC_F16 if scale == "f16" else hc.HC_F32, codes, scales, err)
        x = src.float().reshape(nslots, B, H, d)
        am = x.abs().amax(-1, keepdim=True)
        s = am / torch.full_like(am, 448.0)                   # tensor / tensor: IEEE division
        if scale == "f16":
            s = s.half().float()
        q = torch.where(s > 0, x / s, torch.zeros_like(x)).clamp(-448.0, 448.0)
        want = q.to(torch.float8_e4m3fn).view(torch.uint8)
        want = torch.where(s > 0, want, torch.zeros_like(want))
        got = codes[0, :, 0].permute(0, 2, 1, 3)                # [slot, t, h, d]
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        bad = (got != want).reshape(-1, d)[:nr].any(-1)
        assert not bool(bad.any()), (fmt, scale, int(bad.sum()))
        got_s = scales[0, :, 0].permute(0, 2, 1).float()        # [slot, t, h]
        assert torch.equal(got_s, s[..., 0])
        checked += nr * (d - 1)
    assert checked > 1.0e9
