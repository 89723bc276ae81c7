"""KVPath.step (table on a side stream) and KVPath.capture (a CUDA graph of
the step): both give the eager encode -> table -> fetch results bit for bit,
and those match the oracle."""
import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wire", ["fp8", "int4", "fp8_rows"])
def test_step_and_graph_match_eager_and_oracle(wire):
    from kv_cache_quantization_hc_gb300 import path as kvpath
    import __graft_entry__
    __graft_entry__.build()
    c = parity.random_case(77, L=2, H=4, d=128, B=16, nb=37, src_fmt="bf16", out_fmt="bf16",
                           pairing="half_split", ragged=True)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    dev = torch.device("cuda", 0)
    p = kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots),
                      src_slots=c.src_slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                      delta_m_distinct=dm_vals, delta_idx=dm_idx, wire=wire, pairing=c.pairing,
                      rope_base=c.rope_base, paged_dtype=c.out_fmt, device=dev)
    sk = torch.as_tensor(c.src_k, device=dev).to(torch.bfloat16)
    sv = torch.as_tensor(c.src_v, device=dev).to(torch.bfloat16)
    shape = (c.L, c.num_dst_slots, c.B, c.H, c.d)
    outs = []
    for mode in ("eager", "step", "graph"):
        dk = torch.full(shape, parity.SENTINEL, dtype=torch.bfloat16, device=dev)
        dv = torch.full_like(dk, parity.SENTINEL)
        p.codes.zero_()
        p.table.zero_()
        if mode == "eager":
            p.encode(sk, sv)
            p.build_table()
            p.fetch(dk, dv)
        elif mode == "step":
            p.step(sk, sv, dk, dv)
        else:
            g = p.capture(sk, sv, dk, dv)
            p.codes.zero_()
            dk.fill_(parity.SENTINEL)
            dv.fill_(parity.SENTINEL)
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize(dev)
        assert p.error_bits() == 0
        outs.append((p.codes.cpu().clone(), dk.cpu().clone(), dv.cpu().clone()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)
    want = parity.oracle_run(c, wire)
    got = {"k": outs[2][1].double().numpy(), "v": outs[2][2].double().numpy()}
    rep = parity.compare_outputs(c, wire, got, want)
    assert np.array_equal(outs[2][0].numpy(), want["codes"])
    assert rep["k_ok"] and rep["v_ok"] and rep["k_untouched_ok"] and rep["v_untouched_ok"], rep
