"""GPU parity at the workloads' full sizes, in the launch configurations the
benchmark uses, checked against the oracle on EVERY block of the checked
layers (tests/full_parity.py: the oracle runs in spawned worker processes on
chunks of blocks), plus properties that hold at any size.

* qwen3_8b: one encode call over 36 layers x 2048 blocks, one table call, one
  fetch call - exactly the benchmark's step - for both FP8 wires; all 36
  layers, all 2048 blocks each, are compared with the oracle.
* llama3_70b: 80 layers fetched one layer per call on a side stream into a
  bf16 paged cache, after per-layer encodes on the main stream; every block
  of all 80 layers is compared with the oracle.
* ragged: 36 layers, block sizes 16 and 64 in separate calls, ragged tails;
  INT4 (g32, fp16 scales): every block (both block sizes, every padding row)
  of every third layer and the last (13 of 36 layers) is compared with the
  oracle, and placement is checked on all 36; FP8: the first, a middle and
  the last layer.  With HC_PARITY_ALL_LAYERS=1, every block of all 36 layers
  is compared for both wires (about four more minutes).
"""
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import paged, rope
from tests import full_parity, parity

pytestmark = pytest.mark.gpu
CHUNK_TOKENS = 4096            # tokens of one layer per oracle task


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def pool():
    with full_parity.OraclePool() as p:
        yield p


def _nan_pool(shape, dtype, device):
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def _host(t):
    """A tensor's values in their stored form (bf16 as uint16 bit patterns)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def submit_layer(pool, w, blk, wire, label, src_k, src_v, codes, scales, dst_k, dst_v,
                 group=32, scale_dtype="f16"):
    """Queue every block of one layer for the oracle, in chunks.

    src_k, src_v: [num_src_slots, B, H, d] the layer's cached pool;
    codes, scales: the layer's wire [NB, 2, H, ...]; dst_k, dst_v:
    [num_dst_slots, B, H, d] the layer's destination pool after the fetch.
    """
    dev = src_k.device
    src = torch.as_tensor(blk.src_slots.astype(np.int64), device=dev)
    dst = torch.as_tensor(blk.dst_slots.astype(np.int64), device=dev)
    step = max(1, CHUNK_TOKENS // blk.B)
    for a in range(0, blk.nb, step):
        b = min(blk.nb, a + step)
        pool.submit(dict(
            label=(label, a, b), wire=wire, src_fmt=w.src_dtype, out_fmt=w.out_dtype,
            src_k=_host(src_k[src[a:b]])[None], src_v=_host(src_v[src[a:b]])[None],
            codes=_host(codes[a:b])[None], scales=_host(scales[a:b])[None],
            dst_k=_host(dst_k[dst[a:b]])[None], dst_v=_host(dst_v[dst[a:b]])[None],
            n_valid=blk.n_valid[a:b].copy(), delta_m=blk.delta_m[a:b].copy(), d=w.d,
            rope_base=w.rope_base, pairing=w.pairing, group=group, scale_dtype=scale_dtype))


def assert_all_ok(pool, want_blocks):
    s = full_parity.summarize(pool.results())
    assert not s["failed"], s["failed"]
    assert s["blocks"] == want_blocks, (s["blocks"], want_blocks)
    return s


@pytest.mark.parametrize("codec", ["fp8", "fp8_rows"])
def test_qwen3_8b_benchmark_step(codec, pool):
    import bench
    dev = torch.device("cuda", 0)
    w = workloads.qwen3_8b()
    blk = w.blocks[0]
    p, src_k, src_v, dst_k, dst_v = bench.setup_device(w, blk, dev, codec)
    dst_k.fill_(float("nan"))
    dst_v.fill_(float("nan"))
    p.encode(src_k, src_v)
    p.build_table()
    p.fetch(dst_k, dst_v)
    torch.cuda.synchronize()
    assert p.error_bits() == 0
    # every slot of the shuffled destination table is written, nothing is NaN
    assert not torch.isnan(dst_k).any() and not torch.isnan(dst_v).any()
    assert torch.all(p.scales > 0)
    # the single table row: (cos, sin)(4096 theta_i)
    th = rope.inv_freq(w.d, w.rope_base)
    want = paged.delta_sincos_table(np.array([4096]), th)
    assert np.all(np.abs(p.table.double().cpu().numpy() - want) <= parity.ulp(want, "f32"))
    # the oracle on every block of every layer
    for layer in range(w.L):
        submit_layer(pool, w, blk, codec, f"qwen3_8b/{codec}/L{layer}", src_k[layer], src_v[layer],
                     p.codes[layer], p.scales[layer], dst_k[layer], dst_v[layer])
    assert_all_ok(pool, w.L * blk.nb)


def test_llama3_70b_layer_streamed(pool):
    dev = torch.device("cuda", 0)
    from kv_cache_quantization_hc_gb300 import path as kvpath
    w = workloads.llama3_70b()
    blk = w.blocks[0]
    p = kvpath.from_blocks(w, blk, "fp8", device=dev)
    shape = (w.L, blk.num_dst_slots, blk.B, w.H, w.d)
    dst_k = _nan_pool(shape, torch.bfloat16, dev)
    dst_v = _nan_pool(shape, torch.bfloat16, dev)
    side = torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream(dev)
    p.build_table(stream=main)
    for layer in range(w.L):
        k = workloads.device_pool(w, blk, range(layer, layer + 1), 0, dev)
        v = workloads.device_pool(w, blk, range(layer, layer + 1), 1, dev)
        p.encode(k, v, stream=main, codes=p.codes[layer:layer + 1], scales=p.scales[layer:layer + 1])
        ev = torch.cuda.Event()
        ev.record(main)
        side.wait_event(ev)
        p.fetch(dst_k[layer], dst_v[layer], stream=side, codes=p.codes[layer:layer + 1],
                scales=p.scales[layer:layer + 1])
    torch.cuda.synchronize()
    assert p.error_bits() == 0
    assert not torch.isnan(dst_k).any() and not torch.isnan(dst_v).any()
    # distinct delta-m values: one table row each, shared by all 80 layers
    assert p.n_distinct == len(np.unique(blk.delta_m)) <= 1024
    layers = range(w.L)
    for layer in layers:
        k = workloads.device_pool(w, blk, range(layer, layer + 1), 0, dev)[0]
        v = workloads.device_pool(w, blk, range(layer, layer + 1), 1, dev)[0]
        submit_layer(pool, w, blk, "fp8", f"llama3_70b/L{layer}", k, v, p.codes[layer],
                     p.scales[layer], dst_k[layer], dst_v[layer])
    assert_all_ok(pool, len(layers) * blk.nb)


@pytest.mark.parametrize("wire", ["int4", "fp8"])
def test_ragged_sweep(wire, pool):
    dev = torch.device("cuda", 0)
    from kv_cache_quantization_hc_gb300 import path as kvpath
    w = workloads.ragged()
    if os.environ.get("HC_PARITY_ALL_LAYERS") == "1":    # every block of every layer
        all_layers = check_layers = range(w.L)
    elif wire == "int4":
        all_layers = range(w.L)
        check_layers = set(range(0, w.L, 3)) | {w.L - 1}
    else:
        all_layers = check_layers = [0, w.L // 2, w.L - 1]
    want = 0
    for bi, blk in enumerate(w.blocks):
        p = kvpath.from_blocks(w, blk, wire, device=dev, n_layers=1, scale_dtype="f16")
        p.build_table()
        shape = (1, blk.num_dst_slots, blk.B, w.H, w.d)
        for layer in all_layers:
            k = workloads.device_pool(w, blk, range(layer, layer + 1), 0, dev)
            v = workloads.device_pool(w, blk, range(layer, layer + 1), 1, dev)
            dk = torch.full(shape, parity.SENTINEL, dtype=torch.bfloat16, device=dev)
            dv = torch.full(shape, parity.SENTINEL, dtype=torch.bfloat16, device=dev)
            p.encode(k, v)
            p.fetch(dk, dv)
            torch.cuda.synchronize()
            assert p.error_bits() == 0
            # padding rows of tail blocks are never written; valid rows always are
            written = torch.zeros((blk.num_dst_slots, blk.B), dtype=torch.bool, device=dev)
            nv = torch.as_tensor(blk.n_valid, device=dev)
            rows = torch.arange(blk.B, device=dev)[None, :] < nv[:, None]
            written[torch.as_tensor(blk.dst_slots.astype(np.int64), device=dev)] = rows
            untouched = (dk[0] == parity.SENTINEL).all(-1).all(-1)
            assert torch.equal(untouched, ~written)
            if layer in check_layers:
                submit_layer(pool, w, blk, wire, f"ragged/{wire}/B{blk.B}/L{layer}", k[0], v[0],
                             p.codes[0], p.scales[0], dk[0], dv[0])
                want += blk.nb
    assert_all_ok(pool, want)
