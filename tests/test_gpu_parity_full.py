"""GPU parity at the workloads' full sizes, in the launch configurations the
benchmark uses, checked against the oracle on sampled blocks (all of their
layers, or sampled layers) and by properties that hold at any size.

* qwen3_8b: one encode call over 36 layers x 2048 blocks, one table call, one
  fetch call - exactly the benchmark's step.
* llama3_70b: 80 layers fetched one layer per call on a side stream into a
  bf16 paged cache, after per-layer encodes on the main stream.
* ragged: 36 layers, block sizes 16 and 64 in separate calls, ragged tails,
  INT4 (g32, fp16 scales) and FP8.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import paged, rope
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _nan_pool(shape, dtype, device):
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def _check_blocks(w, blk, js, layers, src_k_host, src_v_host, codes, scales, dst_k, dst_v,
                  wire, group=32, scale_dtype="f16"):
    """Oracle on blocks js (src arrays [len(layers), len(js), B, H, d] on the
    host) against the GPU's wire and destination slots."""
    n = len(js)
    nv = blk.n_valid[js]
    if wire == "fp8":
        ocodes, oscales = paged.encode_fp8(src_k_host, src_v_host, np.arange(n), nv)
        vals = paged.decode_fp8(ocodes, oscales)
    elif wire == "fp8_rows":
        ocodes, oscales = paged.encode_fp8_rows(src_k_host, src_v_host, np.arange(n), nv, scale_dtype)
        vals = paged.decode_fp8_rows(ocodes, oscales)
    else:
        ocodes, oscales = paged.encode_int4(src_k_host, src_v_host, np.arange(n), nv, group, scale_dtype)
        vals = paged.decode_int4(ocodes, oscales, group)
    assert np.array_equal(codes, ocodes), "wire codes differ"
    assert np.array_equal(scales, oscales), "wire scales differ"
    th = rope.inv_freq(w.d, w.rope_base)
    sent = np.full((len(layers), n, blk.B, w.H, w.d), parity.SENTINEL)
    ek, ev = paged.fetch_rotate_scatter(vals, blk.delta_m[js], th, w.pairing, np.arange(n), sent, sent,
                                        w.out_dtype, n_valid=nv)
    m = np.zeros((len(layers), n, blk.B), bool)
    for i in range(n):
        m[:, i, :nv[i]] = True
    ok_k, kerr, kbar = parity.compare_k(dst_k[m], ek[m], w.out_dtype)
    assert ok_k, (kerr, kbar)
    gv, evv = dst_v[m], ev[m]
    if wire in ("fp8", "fp8_rows") and w.out_dtype != "f32":
        assert np.all(np.abs(gv - evv) <= np.maximum(parity.ulp(gv, w.out_dtype), parity.ulp(evv, w.out_dtype)))
    else:
        assert np.array_equal(gv, evv)
    return m


@pytest.mark.parametrize("codec", ["fp8", "fp8_rows"])
def test_qwen3_8b_benchmark_step(codec):
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
    # oracle on sampled blocks, all 36 layers
    r = np.random.default_rng(0)
    js = np.unique(np.concatenate([[0, blk.nb - 1], r.choice(blk.nb, 12, replace=False)]))
    sl = torch.as_tensor(blk.src_slots[js].astype(np.int64), device=dev)
    dl = torch.as_tensor(blk.dst_slots[js].astype(np.int64), device=dev)
    host = lambda t: t.double().cpu().numpy()
    _check_blocks(w, blk, js, range(w.L), host(src_k[:, sl]), host(src_v[:, sl]),
                  p.codes[:, js].cpu().numpy(), host(p.scales[:, js]), host(dst_k[:, dl]),
                  host(dst_v[:, dl]), codec)


def test_llama3_70b_layer_streamed():
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
    r = np.random.default_rng(1)
    js = np.unique(np.concatenate([[0, blk.nb - 1], r.choice(blk.nb, 6, replace=False)]))
    layers = [0, 41, 79]
    sl = torch.as_tensor(blk.src_slots[js].astype(np.int64), device=dev)
    dl = torch.as_tensor(blk.dst_slots[js].astype(np.int64), device=dev)
    host = lambda t: t.double().cpu().numpy()
    sk = np.concatenate([host(workloads.device_pool(w, blk, range(l, l + 1), 0, dev)[:, sl]) for l in layers])
    sv = np.concatenate([host(workloads.device_pool(w, blk, range(l, l + 1), 1, dev)[:, sl]) for l in layers])
    li = torch.as_tensor(layers, device=dev)
    _check_blocks(w, blk, js, layers, sk, sv, p.codes[li][:, js].cpu().numpy(),
                  host(p.scales[li][:, js]), host(dst_k[li][:, dl]), host(dst_v[li][:, dl]), "fp8")


@pytest.mark.parametrize("wire", ["int4", "fp8"])
def test_ragged_sweep(wire):
    dev = torch.device("cuda", 0)
    from kv_cache_quantization_hc_gb300 import path as kvpath
    w = workloads.ragged()
    check_layers = [0, 17, 35]
    all_layers = range(w.L) if wire == "int4" else check_layers
    for bi, blk in enumerate(w.blocks):
        p = kvpath.from_blocks(w, blk, wire, device=dev, n_layers=1, scale_dtype="f16")
        p.build_table()
        r = np.random.default_rng(10 + bi)
        tails = np.flatnonzero(blk.n_valid < blk.B)
        js = np.unique(np.concatenate([[0, blk.nb - 1], tails[:6], r.choice(blk.nb, 6, replace=False)]))
        sl = torch.as_tensor(blk.src_slots[js].astype(np.int64), device=dev)
        dl = torch.as_tensor(blk.dst_slots[js].astype(np.int64), device=dev)
        host = lambda t: t.double().cpu().numpy()
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
                _check_blocks(w, blk, js, [layer], host(k[:, sl]), host(v[:, sl]),
                              p.codes[:, js].cpu().numpy(), host(p.scales[:, js]),
                              host(dk[:, dl]), host(dv[:, dl]), wire)
