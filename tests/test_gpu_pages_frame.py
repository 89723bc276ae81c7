"""The pages' frame through the CUDA path: one 64-token block of 8 heads x
128 channels, K and V (131,072 fp16 values), encoded with one fp16 scale per
token-head row (FP8) or per 128-channel group (INT4) gives the printed
payloads of 133,120 and 67,584 bytes (1.97x and 3.88x); the codes and scales
are the oracle's, the block round-trips through the fetch within the bars,
and the GPU CRC-32 of the stored block equals zlib's over the same bytes.
[HyperCache page, "Example output" part B: FP8 TCP frame, INT4 grouped disk
block with CRC32.]"""
import zlib

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu

CASES = {"fp8_rows": (133120, 1.97), "int4": (67584, 3.88)}


@pytest.mark.parametrize("wire", sorted(CASES))
def test_pages_frame_payload_parity_and_crc(wire):
    from kv_cache_quantization_hc_gb300 import path as kvpath
    import __graft_entry__
    __graft_entry__.build()
    payload_want, ratio_want = CASES[wire]
    c = parity.random_case(131, L=1, H=8, d=128, B=64, nb=1, src_fmt="f16", out_fmt="bf16",
                           pairing="half_split", extra_slots=1)
    rep = parity.run_case(c, wire, group=128, scale_dtype="f16")
    assert rep["ok"], rep

    dev = torch.device("cuda", 0)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p = kvpath.KVPath(n_layers=1, H=8, d=128, B=64, n_blocks=1, src_slots=c.src_slots,
                      dst_slots=c.dst_slots, n_valid=None, delta_m_distinct=dm_vals,
                      delta_idx=dm_idx, wire=wire, pairing=c.pairing, rope_base=c.rope_base,
                      paged_dtype="bf16", group=128, scale_dtype="f16", device=dev)
    sk = torch.as_tensor(c.src_k, device=dev).to(torch.float16)
    sv = torch.as_tensor(c.src_v, device=dev).to(torch.float16)
    p.encode(sk, sv)
    crc = p.crc32()
    torch.cuda.synchronize(dev)
    assert p.error_bits() == 0
    codes = p.codes.cpu().numpy()
    scales = p.scales.cpu().numpy()
    assert scales.dtype == np.float16
    payload = codes.nbytes + scales.nbytes
    assert payload == payload_want
    assert round(2 * 64 * 8 * 128 * 2 / payload, 2) == ratio_want
    want = parity.oracle_run(c, wire, group=128, scale_dtype="f16")
    assert np.array_equal(codes, want["codes"])
    assert np.array_equal(scales.astype(np.float64), want["scales"])
    stored = codes.tobytes() + scales.tobytes()
    assert int(crc.cpu().numpy().view(np.uint32)[0]) == zlib.crc32(stored)
