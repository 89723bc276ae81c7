"""The library keeps no global state and its calls are thread-safe: two host
threads, each driving its own KVPath on its own stream, run whole passes at
the same time, and every output equals the same pass run alone (and the
oracle)."""
import threading

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


def _path(c, wire, dev):
    from kv_cache_quantization_hc_gb300 import path as kvpath
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    return kvpath.KVPath(n_layers=c.L, H=c.H, d=c.d, B=c.B, n_blocks=len(c.src_slots),
                         src_slots=c.src_slots, dst_slots=c.dst_slots, n_valid=c.n_valid,
                         delta_m_distinct=dm_vals, delta_idx=dm_idx, wire=wire, pairing=c.pairing,
                         rope_base=c.rope_base, paged_dtype=c.out_fmt, device=dev)


def test_two_threads_two_streams():
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    jobs = []
    for seed, wire, pairing in ((301, "fp8", "half_split"), (302, "int4", "interleaved")):
        c = parity.random_case(seed, L=3, H=4, d=128, B=16, nb=61, src_fmt="bf16", out_fmt="bf16",
                               pairing=pairing, ragged=True)
        sk = torch.as_tensor(c.src_k, device=dev).to(torch.bfloat16)
        sv = torch.as_tensor(c.src_v, device=dev).to(torch.bfloat16)
        shape = (c.L, c.num_dst_slots, c.B, c.H, c.d)
        jobs.append(dict(c=c, wire=wire, p=_path(c, wire, dev), sk=sk, sv=sv, stream=torch.cuda.Stream(dev),
                         dk=torch.full(shape, parity.SENTINEL, dtype=torch.bfloat16, device=dev),
                         dv=torch.full(shape, parity.SENTINEL, dtype=torch.bfloat16, device=dev)))
    # each pass alone
    alone = []
    for j in jobs:
        j["p"].step(j["sk"], j["sv"], j["dk"], j["dv"])
        torch.cuda.synchronize(dev)
        alone.append((j["p"].codes.cpu().clone(), j["dk"].cpu().clone(), j["dv"].cpu().clone()))
        j["dk"].fill_(parity.SENTINEL)
        j["dv"].fill_(parity.SENTINEL)
        j["p"].codes.zero_()
    torch.cuda.synchronize(dev)

    errors = []
    start = threading.Barrier(len(jobs))

    def run(j):
        try:
            torch.cuda.set_device(dev)
            start.wait(timeout=60)
            for _ in range(20):
                j["p"].step(j["sk"], j["sv"], j["dk"], j["dv"], stream=j["stream"])
            j["stream"].synchronize()
        except Exception as e:       # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert not any(t.is_alive() for t in threads)
    torch.cuda.synchronize(dev)
    for j, (codes, dk, dv) in zip(jobs, alone):
        assert j["p"].error_bits() == 0
        assert torch.equal(j["p"].codes.cpu(), codes)
        assert torch.equal(j["dk"].cpu(), dk) and torch.equal(j["dv"].cpu(), dv)
        want = parity.oracle_run(j["c"], j["wire"])
        rep = parity.compare_outputs(j["c"], j["wire"], {"k": dk.double().numpy(), "v": dv.double().numpy()}, want)
        assert rep["k_ok"] and rep["v_ok"] and rep["k_untouched_ok"] and rep["v_untouched_ok"], rep
