"""Pins for the oracle's group quantizers and byte accounting (CPU only).

Pinned to: the compression ratios and byte counts the pages print, the INT4
cosine the pages print, the scale rules' closed forms, brute force for the
INT4 rounding, and numpy's rint.
"""
import numpy as np
import pytest

from oracle import quant, kvbytes, fp8
from oracle.numerics import round_to


def _fp16_normal(n, seed):
    return round_to(np.random.default_rng(seed).standard_normal(n), "f16")


# --- pages' "Example output", part B ---------------------------------------
def test_pages_compression_ratios_from_buffer_sizes(golden):
    """A 131072-element fp16 tensor with one fp16 scale per 128 elements
    reproduces the printed 1.97x (FP8) and 3.88x (INT4), and payloads just
    under the printed frame / file sizes."""
    x = _fp16_normal(131072, 0).reshape(-1, 128)
    c8, s8 = quant.fp8_quantize(x, scale_dtype="f16")
    c4, s4 = quant.int4_quantize(x, scale_dtype="f16")
    fp8_bytes = c8.size + s8.size * 2
    int4_bytes = quant.int4_pack(c4).size + s4.size * 2
    src = x.size * 2
    assert fp8_bytes == 133120 and int4_bytes == 67584
    assert round(src / fp8_bytes, 2) == golden["fp8_compression_ratio"]
    assert round(src / int4_bytes, 2) == golden["int4_compression_ratio"]
    # the printed frame and file carry a small header/CRC on top of the payload
    assert 0 < golden["fp8_tcp_frame_bytes"] - fp8_bytes < 128
    assert 0 < golden["int4_bytes_on_disk"] - int4_bytes < 128
    assert kvbytes.wire_bytes(x.size, 8, s8.size, 2) == fp8_bytes
    assert kvbytes.wire_bytes(x.size, 4, s4.size, 2) == int4_bytes


def test_pages_int4_cosine(golden):
    """INT4 g128 round trip of N(0,1) fp16 data lands on the printed 0.993258
    (the exact draw is not stated: agreement to 3e-4 across seeds)."""
    for seed in range(3):
        x = _fp16_normal(131072, seed).reshape(-1, 128)
        q, s = quant.int4_quantize(x, scale_dtype="f16")
        cos = quant.cosine(x, quant.int4_dequantize(q, s))
        assert abs(cos - golden["int4_cosine"]) < 3e-4, cos


def test_workload_layout_ratios():
    """The workloads' own layouts give different ratios than the pages'."""
    r16 = kvbytes.compression_ratio(16 * 128, 2, 8, 1, 4)
    r64 = kvbytes.compression_ratio(64 * 128, 2, 8, 1, 4)
    r4 = kvbytes.compression_ratio(32, 2, 4, 1, 2)
    assert abs(r16 - 1.99610) < 1e-5 and abs(r64 - 1.99902) < 1e-5 and abs(r4 - 3.55556) < 1e-5


# --- scale rules --------------------------------------------------------------
@pytest.mark.parametrize("scale_dtype", ["f32", "f16"])
def test_fp8_amax_element_codes_to_448(scale_dtype):
    rng = np.random.default_rng(5)
    x = round_to(rng.standard_normal((500, 256)) * np.exp(rng.uniform(-8, 8, (500, 1))), "f32")
    codes, s = quant.fp8_quantize(x, scale_dtype=scale_dtype)
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(500), i]
    assert np.all((top & 0x7F) == 0x7E)
    assert np.array_equal(top >> 7, np.signbit(x[np.arange(500), i]).astype(np.uint8))
    if scale_dtype == "f32":
        assert np.array_equal(s, round_to(np.abs(x).max(1) / 448.0, "f32"))


@pytest.mark.parametrize("scale_dtype", ["f32", "f16"])
def test_int4_amax_element_codes_to_7(scale_dtype):
    rng = np.random.default_rng(6)
    x = round_to(rng.standard_normal((500, 32)) * np.exp(rng.uniform(-5, 5, (500, 1))), "bf16")
    q, s = quant.int4_quantize(x, scale_dtype=scale_dtype)
    i = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(q[np.arange(500), i]) == 7)
    want = round_to(np.abs(x).max(1) / 7.0, "f32")
    if scale_dtype == "f16":
        want = round_to(want, "f16")
    assert np.array_equal(s, want)


def test_zero_group_and_padding():
    x = np.zeros((3, 32))
    x[1, 5] = -0.0
    c8, s8 = quant.fp8_quantize(x)
    q4, s4 = quant.int4_quantize(x)
    assert np.all(c8 == 0) and np.all(s8 == 0) and np.all(q4 == 0) and np.all(s4 == 0)
    # padding excluded from amax and zeroed
    y = np.ones((1, 8))
    y[0, 6:] = 1e6
    valid = np.arange(8)[None, :] < 6
    c, s = quant.fp8_quantize(y, valid)
    assert s[0] == round_to(1.0 / 448, "f32") and np.all(c[0, 6:] == 0) and np.all(c[0, :6] == 0x7E)


# --- INT4 rounding ------------------------------------------------------------
def test_int4_rounding_brute_force():
    """q at every half integer in [-6.5, 6.5] and its fp32 neighbours."""
    s = 1.0
    qs = []
    for k in range(-13, 14):
        h = np.float32(k / 2)
        qs += [float(np.nextafter(h, np.float32(-9))), float(h), float(np.nextafter(h, np.float32(9)))]
    qs = np.array(qs)
    x = np.concatenate([qs, [7.0]])          # 7.0 pins amax/7 = 1
    q, sc = quant.int4_quantize(x[None, :], scale_dtype="f32")
    assert sc[0] == s
    for v, got in zip(qs, q[0, :-1]):
        lo = np.floor(v)
        frac = v - lo
        want = lo if frac < 0.5 else lo + 1 if frac > 0.5 else (lo if lo % 2 == 0 else lo + 1)
        assert got == want, (v, got, want)
    # clamping: a subnormal fp16 scale rounded down pushes amax/s to 9.8 -> 7
    x = np.array([[9.8 * 2.0 ** -24, 2.0 ** -24]])
    x = round_to(x, "f32")
    q, s16 = quant.int4_quantize(x, scale_dtype="f16")
    assert s16[0] == 2.0 ** -24 and list(q[0]) == [7, 1]


def test_int4_pack_order_and_round_trip():
    assert quant.int4_pack(np.array([1, -1]))[0] == 0xF1
    assert quant.int4_pack(np.array([-7, 7]))[0] == 0x79
    r = np.random.default_rng(7).integers(-7, 8, (64, 128))
    assert np.array_equal(quant.int4_unpack(quant.int4_pack(r)), r)


def test_dequant_error_bounds():
    rng = np.random.default_rng(8)
    x = round_to(rng.standard_normal((200, 2048)), "f32")
    c, s = quant.fp8_quantize(x)
    err = np.abs(quant.fp8_dequantize(c, s) - x)
    # half an E4M3 step: 2**-4 relative in the normal range, 2**-10 * s below it
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6))
    q, s4 = quant.int4_quantize(x.reshape(-1, 32))
    err4 = np.abs(quant.int4_dequantize(q, s4) - x.reshape(-1, 32))
    assert np.all(err4 <= s4[:, None] * (0.5 + 1e-3) + np.abs(x.reshape(-1, 32)).max(1, keepdims=True) * 2 ** -10)


def test_e4m3_grid_values_round_trip_through_scale():
    """Values already on the E4M3 grid times a power-of-two scale encode exactly."""
    mags = fp8.e4m3_table()[:0x7F]
    x = np.concatenate([mags, -mags[1:]])[None, :] * 2.0 ** -3
    c, s = quant.fp8_quantize(x)
    assert s[0] == 2.0 ** -3
    assert np.array_equal(quant.fp8_dequantize(c, s), x)
