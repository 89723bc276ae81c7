"""Pins for the oracle's paged gather/encode and fetch/scatter (CPU only):
placement by the inverse permutation, sentinel preservation, K/V identity,
padding rows, the SO(2) end-to-end property, and the pages' KV-bytes formula."""
import numpy as np
import pytest

import workloads
from oracle import paged, rope, kvbytes, quant, fp8
from oracle.numerics import round_to


def _tagged_pool(L, S, B, H, d, kv):
    """pool[l, s, t, h, c] = unique code of (l, s, t, h, c, kv)."""
    l, s, t, h, c = np.meshgrid(np.arange(L), np.arange(S), np.arange(B), np.arange(H), np.arange(d),
                                indexing="ij")
    return ((((l * S + s) * B + t) * H + h) * d + c) * 2.0 + kv


def test_gather_placement_is_inverse_permutation():
    L, S, B, H, d = 2, 10, 4, 3, 8
    pk, pv = _tagged_pool(L, S, B, H, d, 0), _tagged_pool(L, S, B, H, d, 1)
    src = np.array([7, 2, 9, 0], dtype=np.int32)
    w = paged.gather_slabs(pk, pv, src)
    assert w.shape == (L, 4, 2, H, B, d)
    for layer in range(L):
        for j, s in enumerate(src):
            for kv, pool in ((0, pk), (1, pv)):
                for h in range(H):
                    assert np.array_equal(w[layer, j, kv, h], pool[layer, s, :, h, :])
    assert np.all(w[:, :, 0] % 2 == 0) and np.all(w[:, :, 1] % 2 == 1)


def test_scatter_placement_sentinels_and_padding():
    L, S, B, H, d, NB = 2, 9, 4, 2, 8, 3
    rng = np.random.default_rng(0)
    vals = rng.standard_normal((L, NB, 2, H, B, d))
    dst = np.array([5, 0, 7])
    nv = np.array([4, 1, 3])
    sentinel = np.full((L, S, B, H, d), -777.0)
    th = rope.inv_freq(d, 1e4)
    k, v = paged.fetch_rotate_scatter(vals, np.zeros(NB), th, rope.INTERLEAVED, dst, sentinel, sentinel,
                                      "f32", n_valid=nv)
    touched = np.zeros((L, S, B), bool)
    for j in range(NB):
        touched[:, dst[j], :nv[j]] = True
        for layer in range(L):
            want_k = round_to(vals[layer, j, 0].transpose(1, 0, 2)[:nv[j]], "f32")
            want_v = round_to(vals[layer, j, 1].transpose(1, 0, 2)[:nv[j]], "f32")
            assert np.array_equal(k[layer, dst[j], :nv[j]], want_k)     # delta-m = 0: identity
            assert np.array_equal(v[layer, dst[j], :nv[j]], want_v)
    assert np.all(k[~touched] == -777.0) and np.all(v[~touched] == -777.0)
    with pytest.raises(ValueError):
        paged.fetch_rotate_scatter(vals, np.zeros(NB), th, rope.INTERLEAVED, [1, 1, 2], sentinel, sentinel, "f32")


@pytest.mark.parametrize("make", [workloads.tiny, workloads.gqa_reorder])
def test_end_to_end_reuse_matches_fresh_rope(make):
    """Cache post-RoPE keys at m_old, fetch them with delta-m (no quantization):
    the keys equal fresh RoPE at m_new; values are untouched."""
    w, draws = make()
    blk, dr = w.blocks[0], draws[0]
    th = rope.inv_freq(w.d, w.rope_base)
    L, NB, B, H, d = dr.k_pre.shape
    k_old = np.stack([np.stack([rope.apply_rope(dr.k_pre[layer, j], dr.m_old[j], th, w.pairing)
                                for j in range(NB)]) for layer in range(L)])
    vals = np.stack([k_old, dr.v], axis=2).transpose(0, 1, 2, 4, 3, 5)    # [L, NB, 2, H, B, d]
    zero = np.zeros((L, blk.num_dst_slots, B, H, d))
    k, v = paged.fetch_rotate_scatter(vals, blk.delta_m, th, w.pairing, blk.dst_slots, zero, zero, "f32")
    for j in range(NB):
        m_new = dr.m_old[j] + blk.delta_m[j]
        for layer in range(L):
            fresh = rope.apply_rope(dr.k_pre[layer, j], m_new, th, w.pairing)
            assert np.max(np.abs(k[layer, blk.dst_slots[j]] - fresh)) < 1e-5 * np.max(np.abs(fresh))
            assert np.array_equal(v[layer, blk.dst_slots[j]], round_to(dr.v[layer, j], "f32"))


def test_encode_fp8_slab_rules():
    L, S, B, H, d = 1, 6, 16, 2, 64
    rng = np.random.default_rng(1)
    pk = round_to(rng.standard_normal((L, S, B, H, d)), "bf16")
    pv = round_to(-np.abs(rng.standard_normal((L, S, B, H, d))) * 3, "bf16")
    src = np.array([4, 1])
    nv = np.array([16, 5])
    pk[0, 1, 5:, 0, 0] = 1e4              # padding rows of block 1 must not count
    codes, scales = paged.encode_fp8(pk, pv, src, nv)
    assert codes.shape == (L, 2, 2, H, B, d) and scales.shape == (L, 2, 2, H)
    for j, s in enumerate(src):
        for kv, pool in ((0, pk), (1, pv)):
            for h in range(H):
                slab = pool[0, s, :nv[j], h, :]
                assert scales[0, j, kv, h] == round_to(np.abs(slab).max() / 448.0, "f32")
                assert np.all(codes[0, j, kv, h, nv[j]:] == 0)
    # V pool is all negative: every valid code carries its sign bit
    assert np.all(codes[0, 0, 1] & 0x80) and np.all(codes[0, 1, 1, :, :5] & 0x80)


def test_encode_int4_group_rules():
    L, S, B, H, d = 1, 3, 16, 2, 128
    rng = np.random.default_rng(2)
    pk = round_to(rng.standard_normal((L, S, B, H, d)), "bf16")
    pv = round_to(rng.standard_normal((L, S, B, H, d)), "bf16")
    codes, scales = paged.encode_int4(pk, pv, [2, 0], [16, 9], group=32)
    assert codes.shape == (L, 2, 2, H, B, 64) and scales.shape == (L, 2, 2, H, B, 4)
    assert np.all(scales[0, 1, :, :, 9:] == 0) and np.all(codes[0, 1, :, :, 9:] == 0)
    ints = quant.int4_unpack(codes).reshape(L, 2, 2, H, B, 4, 32)
    valid = np.abs(ints[0, 0]).max(-1)
    assert np.all(valid == 7)
    dec = paged.decode_int4(codes, scales, 32)
    assert np.max(np.abs(dec[0, 0, 0, 1] - pk[0, 2, :, 1, :])) <= scales[0, 0, 0, 1].max() * 0.5 * (1 + 1e-3)


def test_decode_fp8_is_exact_product():
    codes = np.arange(256, dtype=np.uint8).reshape(1, 1, 2, 1, 1, 128)
    codes[..., 0x7F % 128] = 0
    s = np.array([0.37, 11.0]).reshape(1, 1, 2, 1) / 448
    s = round_to(s, "f32")
    dec = paged.decode_fp8(codes, s)
    assert np.array_equal(dec[:, :, 0], fp8.e4m3_decode(codes[:, :, 0]) * s[0, 0, 0, 0])
    assert np.array_equal(dec[:, :, 1], fp8.e4m3_decode(codes[:, :, 1]) * s[0, 0, 1, 0])


def test_delta_table_rounding():
    th = rope.inv_freq(128, 1e6)
    t = paged.delta_sincos_table(np.array([0, 4096, -8192]), th)
    assert t.shape == (3, 64, 2)
    assert np.all(t[0, :, 0] == 1.0) and np.all(t[0, :, 1] == 0.0)
    assert np.array_equal(t[1, :, 0], np.cos(4096 * th).astype(np.float32).astype(np.float64))
    assert np.array_equal(t[2, :, 1], np.sin(-8192 * th).astype(np.float32).astype(np.float64))


# --- KV bytes (Module 13, section 1 and checklist) ------------------------------
def test_kv_bytes_pins(golden):
    per_tok = kvbytes.kv_bytes(36, 8, 128, 1, 2)
    assert per_tok == 147456 == golden["qwen3_8b_kib_per_token_fp16"] * 1024
    assert kvbytes.kv_bytes(36, 8, 128, 1, 1) == golden["qwen3_8b_kib_per_token_int8"] * 1024
    assert kvbytes.kv_bytes(36, 8, 128, 1, 0.5) == golden["qwen3_8b_kib_per_token_int4"] * 1024
    assert kvbytes.kv_bytes(36, 8, 128, 32768, 2) == golden["qwen3_8b_32k_fp16_gib"] * 2 ** 30
    assert kvbytes.kv_bytes(36, 8, 128, 25000, 2) == golden["qwen3_8b_25k_fp16_bytes"]
    assert round(kvbytes.kv_bytes(36, 8, 128, 25000, 2) / 2 ** 30, 2) == golden["qwen3_8b_25k_fp16_gib"]
    assert round(kvbytes.kv_bytes(36, 8, 128, 25000, 1) / 2 ** 30, 2) == golden["qwen3_8b_25k_int8_gib"]
    llama = kvbytes.kv_bytes(80, 8, 128, 65536, 1)
    assert llama == 10737418240
    assert round(llama / 2 ** 30) == golden["llama3_70b_64k_fp8_gb_approx"]


# --- row-scaled FP8 (the pages' frame layout) ------------------------------------
def test_encode_fp8_rows_reproduces_the_printed_frame_payload(golden):
    """One 64-token block of 8 heads x 128 channels, K and V, is 131,072 fp16
    values: with one fp16 scale per (token, head) row its FP8 payload is the
    133,120 bytes under the printed 133,188-byte frame (1.97x)."""
    rng = np.random.default_rng(7)
    L, S, B, H, d = 1, 2, 64, 8, 128
    pk = round_to(rng.standard_normal((L, S, B, H, d)), "f16")
    pv = round_to(rng.standard_normal((L, S, B, H, d)), "f16")
    codes, scales = paged.encode_fp8_rows(pk, pv, [1])
    assert codes.shape == (1, 1, 2, H, B, d) and scales.shape == (1, 1, 2, H, B)
    payload = codes.size + scales.size * 2
    assert payload == 133120 and 0 < golden["fp8_tcp_frame_bytes"] - payload < 128
    assert round(2 * pk[0, 1].size * 2 / payload, 2) == golden["fp8_compression_ratio"]
    # same codes as the group quantizer applied to each gathered row
    rows = np.stack([pk[0, 1], pv[0, 1]]).transpose(0, 2, 1, 3)       # [2, H, B, d]
    c2, s2 = quant.fp8_quantize(rows, scale_dtype="f16")
    assert np.array_equal(codes[0, 0], c2) and np.array_equal(scales[0, 0], s2)


def test_encode_fp8_rows_rules():
    rng = np.random.default_rng(8)
    L, S, B, H, d = 2, 4, 16, 2, 64
    pk = round_to(rng.standard_normal((L, S, B, H, d)) * 3, "bf16")
    pv = round_to(rng.standard_normal((L, S, B, H, d)), "bf16")
    pk[1, 2, 3, 1, :] = 0.0
    pk[1, 2, 3, 1, 5] = -0.0
    pk[0, 3, 0, 0, 7] = 3.0e38                      # fp16 scale overflows to +inf
    codes, s = paged.encode_fp8_rows(pk, pv, [2, 3], n_valid=[16, 9])
    assert np.all(s[:, 1, :, :, 9:] == 0) and np.all(codes[:, 1, :, :, 9:] == 0)   # padding rows
    assert s[1, 0, 0, 1, 3] == 0 and np.all(codes[1, 0, 0, 1, 3] == 0)             # zero row (-0 -> 0)
    assert np.isinf(s[0, 1, 0, 0, 0])
    row = pk[0, 3, 0, 0]
    assert np.array_equal(codes[0, 1, 0, 0, 0], np.where(np.signbit(row), 0x80, 0).astype(np.uint8))
    # elsewhere: the amax element codes to +-448, scales are fp16(fp32(amax/448))
    sl = pk[0, 2, :, 1, :]
    want = round_to(round_to(np.abs(sl).max(-1) / 448.0, "f32"), "f16")
    assert np.array_equal(s[0, 0, 0, 1], want)
    i = np.argmax(np.abs(sl), axis=-1)
    assert np.all((codes[0, 0, 0, 1][np.arange(B), i] & 0x7F) == 0x7E)
    dec = paged.decode_fp8_rows(codes, s)
    ok = np.isfinite(s)[..., None] & (s[..., None] > 0)
    err = np.abs(dec - paged.gather_slabs(pk, pv, [2, 3]))
    valid = np.ones_like(err, bool)
    valid[:, 1, :, :, 9:] = False
    assert np.all(err[ok & valid] <= (np.abs(paged.gather_slabs(pk, pv, [2, 3])) * 2.0 ** -4 + 2.0 ** -9 * np.broadcast_to(s[..., None], err.shape))[ok & valid])
