"""GPU parity of the CRC-32 kernel (hc_crc32) against the oracle's CRC-32,
on random units of many sizes (many small units, one warp each; and a few
units of up to 64 MiB, which the library cuts into chunks across warps) and
on encoded wire buffers, plus tamper detection: changing one byte of a unit
changes that unit's CRC only."""
import numpy as np
import pytest
import torch

from oracle import crc32 as ocrc
from tests import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


# a_bytes, a_stride, b_bytes, b_stride, n_units
SHAPES = [(0, 0, 0, 0, 3), (0, 16, 5, 7, 4), (1, 16, 0, 0, 5), (15, 16, 3, 3, 2),
          (16, 32, 0, 0, 9), (4095, 4096, 1, 1, 3), (4096, 4096, 64, 64, 17),
          (4096 + 48, 4160, 13, 20, 6), (32768, 32768, 64, 64, 40), (65536 + 16, 65552, 0, 0, 3),
          (131072, 131072, 2048, 2048, 2), (0, 0, 32, 48, 4), (4096, 4096, 4800, 4800, 5),
          (4096, 4096, 4800, 4808, 3),
          # few, large units: each unit is cut into chunks across warps
          (262144 + 3, 262160, 0, 0, 1), (1 << 20, 1 << 20, 0, 0, 5), (4 << 20, 4 << 20, 4096, 4096, 2),
          (8 * 2 ** 20 + 4100, 8 * 2 ** 20 + 4112, 77, 80, 3), (64 * 2 ** 20 + 5, 64 * 2 ** 20 + 16, 13, 13, 1)]


@pytest.mark.parametrize("a_bytes,a_stride,b_bytes,b_stride,n", SHAPES)
def test_crc32_units(a_bytes, a_stride, b_bytes, b_stride, n):
    from kv_cache_quantization_hc_gb300 import hc
    r = np.random.default_rng(a_bytes * 7 + n)
    a = r.integers(0, 256, max(a_stride * n, 16), dtype=np.uint8)
    b = r.integers(0, 256, max(b_stride * n, b_bytes, 1), dtype=np.uint8)
    da, db = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    out = torch.zeros(n, dtype=torch.int32, device=DEV)
    hc.hc_crc32(da, a_bytes, a_stride, db if b_bytes else None, b_bytes, b_stride, n, out)
    torch.cuda.synchronize()
    want = ocrc.crc32_units(a, a_bytes, a_stride, n, b if b_bytes else None, b_bytes, b_stride)
    assert np.array_equal(_u32(out), want)


@pytest.mark.parametrize("offset", [0, 4, 8, 16])
def test_crc32_second_segment_alignment(offset):
    """b as whole 16-byte words is read word by word when it starts on a
    16-byte boundary, byte by byte otherwise; both give the oracle's CRC."""
    from kv_cache_quantization_hc_gb300 import hc
    r = np.random.default_rng(offset)
    n, a_bytes, b_bytes = 7, 2048, 4096 + 64
    a = r.integers(0, 256, a_bytes * n, dtype=np.uint8)
    b = r.integers(0, 256, b_bytes * n + offset, dtype=np.uint8)
    da, db = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    out = torch.zeros(n, dtype=torch.int32, device=DEV)
    hc.hc_crc32(da, a_bytes, a_bytes, db[offset:], b_bytes, b_bytes, n, out)
    torch.cuda.synchronize()
    want = ocrc.crc32_units(a, a_bytes, a_bytes, n, b[offset:], b_bytes, b_bytes)
    assert np.array_equal(_u32(out), want)


def test_crc32_check_value():
    from kv_cache_quantization_hc_gb300 import hc
    msg = torch.tensor(list(b"123456789") + [0] * 7, dtype=torch.uint8, device=DEV)
    out = torch.zeros(1, dtype=torch.int32, device=DEV)
    hc.hc_crc32(msg, 9, 16, None, 0, 0, 1, out)
    assert _u32(out)[0] == 0xCBF43926


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
def test_crc32_of_the_wire_and_tamper_detection(wire):
    """Per (layer, block): CRC of its codes followed by its scales, on the GPU
    wire, equals the oracle's CRC of the oracle's wire (the two wires are
    bit-identical); one flipped byte changes exactly one unit's CRC."""
    from kv_cache_quantization_hc_gb300 import path as kvpath
    c = parity.random_case(61, L=3, H=4, d=128, B=16, nb=5, src_fmt="bf16", out_fmt="bf16",
                           ragged=True)
    o = parity.oracle_run(c, wire, scale_dtype="f16")
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p = kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots),
                      src_slots=c.src_slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                      delta_m_distinct=dm_vals, delta_idx=dm_idx, wire=wire, pairing=c.pairing,
                      rope_base=c.rope_base, paged_dtype=c.out_fmt, scale_dtype="f16")
    src_k = torch.as_tensor(c.src_k, device=DEV).to(torch.bfloat16)
    src_v = torch.as_tensor(c.src_v, device=DEV).to(torch.bfloat16)
    p.encode(src_k, src_v)
    got = _u32(p.crc32())
    codes = o["codes"]
    sdt = np.float32 if wire == "fp8" else np.float16
    scales = o["scales"].astype(sdt)
    L, NB = c.L, len(c.src_slots)
    a = codes.reshape(L * NB, -1)
    bb = scales.reshape(L * NB, -1).view(np.uint8)
    want = ocrc.crc32_units(a, a.shape[1], a.shape[1], L * NB, bb, bb.shape[1], bb.shape[1])
    assert np.array_equal(got, want)
    # tamper: flip one byte of unit (layer 1, block 3)
    u = 1 * NB + 3
    flat = p.codes.view(-1)
    i = u * a.shape[1] + 777
    flat[i] = flat[i] ^ 0x10
    got2 = _u32(p.crc32())
    changed = np.nonzero(got2 != got)[0]
    assert changed.tolist() == [u]


FUSED = [  # d, B, src dtype, ragged, H
    (128, 16, "bf16", True, 8), (128, 16, "f16", False, 3), (64, 16, "bf16", True, 2),
    (128, 64, "bf16", True, 4), (64, 32, "f16", True, 3), (128, 128, "bf16", False, 2),
    (128, 16, "f32", True, 3), (64, 64, "f32", False, 2)]


@pytest.mark.parametrize("d,B,src,ragged,H", FUSED)
def test_fused_slab_crc_matches_the_oracle(d, B, src, ragged, H):
    """hc_encode_fp8_crc: every slab's CRC (its codes, then its fp32 scale)
    equals the oracle's CRC of the oracle's wire for that slab."""
    from kv_cache_quantization_hc_gb300 import path as kvpath
    c = parity.random_case(81 + B + d, L=3, H=H, d=d, B=B, nb=9, src_fmt=src, out_fmt="bf16",
                           ragged=ragged)
    o = parity.oracle_run(c, "fp8")
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p = kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots),
                      src_slots=c.src_slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                      delta_m_distinct=dm_vals, delta_idx=dm_idx, wire="fp8", pairing=c.pairing,
                      rope_base=c.rope_base, paged_dtype="bf16")
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[src]
    src_k = torch.as_tensor(c.src_k, device=DEV).to(tdt)
    src_v = torch.as_tensor(c.src_v, device=DEV).to(tdt)
    crc = torch.zeros((c.L, len(c.src_slots), 2, c.H), dtype=torch.int32, device=DEV)
    p.encode(src_k, src_v, crc=crc)
    torch.cuda.synchronize()
    assert p.error_bits() == 0
    assert np.array_equal(p.codes.cpu().numpy(), o["codes"])
    n = crc.numel()
    codes = o["codes"].reshape(n, -1)
    scales = o["scales"].astype(np.float32).reshape(n, 1).view(np.uint8)
    want = ocrc.crc32_units(codes, codes.shape[1], codes.shape[1], n, scales, 4, 4)
    assert np.array_equal(_u32(crc).reshape(-1), want)


@pytest.mark.parametrize("src", ["bf16", "f32"])
def test_fused_slab_crc_of_a_skipped_block(src):
    """A block with a bad source slot is flagged and skipped: its wire bytes
    stay as they were.  For 16-bit sources its CRC entries are not written;
    for fp32 sources (encode, then the CRC kernel over every slab) they are
    the CRC of the wire bytes as they stand.  Every other slab's CRC equals
    the oracle's."""
    from kv_cache_quantization_hc_gb300 import hc, path as kvpath
    c = parity.random_case(97, L=2, H=3, d=128, B=16, nb=5, src_fmt=src, out_fmt="bf16")
    o = parity.oracle_run(c, "fp8")
    bad = 2
    slots = c.src_slots.copy()
    slots[bad] = c.src_k.shape[1] + 5                  # outside [0, num_slots)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p = kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(slots),
                      src_slots=slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                      delta_m_distinct=dm_vals, delta_idx=dm_idx, wire="fp8", pairing=c.pairing,
                      rope_base=c.rope_base, paged_dtype="bf16")
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[src]
    src_k = torch.as_tensor(c.src_k, device=DEV).to(tdt)
    src_v = torch.as_tensor(c.src_v, device=DEV).to(tdt)
    p.codes.fill_(0xEE)
    p.scales.fill_(3.0)
    crc = torch.full((c.L, len(slots), 2, c.H), 0x5A5A5A5A, dtype=torch.int32, device=DEV)
    p.encode(src_k, src_v, crc=crc)
    torch.cuda.synchronize()
    assert p.error_bits() == hc.HC_DEVERR_SLOT
    codes = p.codes.cpu().numpy()
    assert np.all(codes[:, bad] == 0xEE) and torch.all(p.scales[:, bad] == 3.0)
    keep = [j for j in range(len(slots)) if j != bad]
    assert np.array_equal(codes[:, keep], o["codes"][:, keep])
    got = _u32(crc)
    n_slab = c.B * c.d
    want = ocrc.crc32_units(o["codes"].reshape(-1, n_slab), n_slab, n_slab, got.size,
                            o["scales"].astype(np.float32).reshape(-1, 1).view(np.uint8), 4, 4)
    want = want.reshape(got.shape)
    assert np.array_equal(got[:, keep], want[:, keep])
    if src == "f32":
        stale = ocrc.crc32_units(codes[:, bad].reshape(-1, n_slab), n_slab, n_slab, c.L * 2 * c.H,
                                 np.full((c.L * 2 * c.H, 1), 3.0, np.float32).view(np.uint8), 4, 4)
        assert np.array_equal(got[:, bad].reshape(-1), stale)
    else:
        assert np.all(got[:, bad] == 0x5A5A5A5A)
