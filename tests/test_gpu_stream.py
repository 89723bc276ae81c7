"""Layer-streamed pass with host buffers (LayerStream) against the oracle:
per-layer uploads, C-ABI encode + fetch on a compute stream and downloads on
a third stream give the same results as the oracle, and unwritten
destination slots keep their host contents."""
import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
def test_layer_stream_matches_oracle(wire):
    from kv_cache_quantization_hc_gb300.path import KVPath
    from kv_cache_quantization_hc_gb300.stream import LayerStream
    c = parity.case_from_workload("gqa_reorder")
    o = parity.oracle_run(c, wire)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p1 = KVPath(n_layers=1, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots), src_slots=c.src_slots,
                dst_slots=c.dst_slots, n_valid=c.n_valid, delta_m_distinct=dm_vals, delta_idx=dm_idx,
                wire=wire, pairing=c.pairing, rope_base=c.rope_base, paged_dtype=c.out_fmt,
                device="cuda")
    bf = torch.bfloat16
    ls = LayerStream(p1, c.src_k.shape[1:], bf, (c.num_dst_slots, c.B, c.H, c.d), bf, "cuda", ring=2)
    h_src_k = torch.from_numpy(c.src_k).to(bf).pin_memory()
    h_src_v = torch.from_numpy(c.src_v).to(bf).pin_memory()
    shape = (c.L, c.num_dst_slots, c.B, c.H, c.d)
    h_dst_k = torch.full(shape, parity.SENTINEL, dtype=bf).pin_memory()
    h_dst_v = torch.full(shape, parity.SENTINEL, dtype=bf).pin_memory()
    h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    for _ in range(2):          # a second pass reuses every ring slot
        ls.run(h_src_k, h_src_v, h_dst_k, h_dst_v, h_err)
    torch.cuda.synchronize()
    assert int(h_err.item()) == 0
    g = {"k": h_dst_k.double().numpy(), "v": h_dst_v.double().numpy()}
    rep = parity.compare_outputs(c, wire, g, o)
    assert rep["k_ok"] and rep["v_ok"] and rep["k_untouched_ok"] and rep["v_untouched_ok"], rep


@pytest.mark.parametrize("wire", ["fp8", "int4"])
def test_layer_stream_passes_back_to_back_with_table_uploads(wire):
    """Several passes streamed with no join between them, each uploading the
    block tables from host memory first: the device tables start out wrong,
    so the result is right only if every pass's uploads precede its computes."""
    from kv_cache_quantization_hc_gb300.path import KVPath
    from kv_cache_quantization_hc_gb300.stream import LayerStream
    c = parity.case_from_workload("gqa_reorder")
    o = parity.oracle_run(c, wire)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    p1 = KVPath(n_layers=1, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots), src_slots=c.src_slots,
                dst_slots=c.dst_slots, n_valid=c.n_valid, delta_m_distinct=dm_vals, delta_idx=dm_idx,
                wire=wire, pairing=c.pairing, rope_base=c.rope_base, paged_dtype=c.out_fmt,
                device="cuda")
    tables = [p1.src_slots, p1.dst_slots, p1.delta_m, p1.delta_idx]
    h_tables = [t.cpu().pin_memory() for t in tables]
    for t in tables:
        t.zero_()                       # wrong until run() uploads the host copies
    bf = torch.bfloat16
    ls = LayerStream(p1, c.src_k.shape[1:], bf, (c.num_dst_slots, c.B, c.H, c.d), bf, "cuda", ring=3)
    h_src_k = torch.from_numpy(c.src_k).to(bf).pin_memory()
    h_src_v = torch.from_numpy(c.src_v).to(bf).pin_memory()
    shape = (c.L, c.num_dst_slots, c.B, c.H, c.d)
    h_dst_k = torch.full(shape, parity.SENTINEL, dtype=bf).pin_memory()
    h_dst_v = torch.full(shape, parity.SENTINEL, dtype=bf).pin_memory()
    h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    ls.run(h_src_k, h_src_v, h_dst_k, h_dst_v, h_err, passes=3, tables=list(zip(tables, h_tables)))
    torch.cuda.synchronize()
    assert int(h_err.item()) == 0
    g = {"k": h_dst_k.double().numpy(), "v": h_dst_v.double().numpy()}
    rep = parity.compare_outputs(c, wire, g, o)
    assert rep["k_ok"] and rep["v_ok"] and rep["k_untouched_ok"] and rep["v_untouched_ok"], rep
