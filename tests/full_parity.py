"""Full-size parity: the oracle over every block of a workload's layers,
against the CUDA path's wire and destination rows.

The GPU tests run a workload in the benchmark's launch configuration, then
cut each checked layer into chunks of blocks.  For every chunk they copy to
the host the cached source rows of its blocks, the wire bytes and scales the
encode wrote for them, and the rows the fetch wrote at their destination
slots.  ``check_chunk`` re-encodes the source with the oracle, compares
codes and scales bit for bit, runs the oracle's fetch (decode, exact fp64
rotation, rounding) and compares K and V with the bars of tests/bars.py;
padding rows of ragged blocks must still hold the sentinel.  Reading each
block's output at its own destination slot checks placement as well.

The chunks go to worker processes started with the "spawn" method (never
forked after the test process has used CUDA); they import numpy and the
oracle only.  ``OraclePool`` keeps a bounded number of chunks in flight, so
host memory stays bounded whatever the workload's size.
"""
import os
import time
from concurrent.futures import FIRST_COMPLETED, ProcessPoolExecutor, wait

import numpy as np

from oracle import paged, rope
from tests.bars import SENTINEL, compare_k, compare_v

THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def to_f64(a, fmt):
    """float64 copy of stored values: bf16 arrives as its uint16 bit
    patterns, f16/f32 as numpy floats (both widen exactly)."""
    a = np.asarray(a)
    if fmt == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def check_chunk(t):
    """Oracle on one chunk (one layer, n blocks) against the GPU's output.

    t["src_k"], t["src_v"]: [1, n, B, H, d] cached rows of the blocks, in
    t["src_fmt"]; t["codes"], t["scales"]: the wire the GPU wrote for them;
    t["dst_k"], t["dst_v"]: [1, n, B, H, d] the rows at their destination
    slots after the fetch (t["out_fmt"]); t["n_valid"], t["delta_m"]: [n].
    """
    t0 = time.perf_counter()
    k = to_f64(t["src_k"], t["src_fmt"])
    v = to_f64(t["src_v"], t["src_fmt"])
    _, n, B, H, d = k.shape
    nv = np.asarray(t["n_valid"], np.int64)
    ids = np.arange(n)
    wire = t["wire"]
    if wire == "fp8":
        oc, osc = paged.encode_fp8(k, v, ids, nv)
        vals = paged.decode_fp8(oc, osc)
    elif wire == "fp8_rows":
        oc, osc = paged.encode_fp8_rows(k, v, ids, nv, t["scale_dtype"])
        vals = paged.decode_fp8_rows(oc, osc)
    elif wire == "int4":
        oc, osc = paged.encode_int4(k, v, ids, nv, t["group"], t["scale_dtype"])
        vals = paged.decode_int4(oc, osc, t["group"])
    else:
        raise ValueError(wire)
    res = {"label": t["label"], "blocks": int(n), "tokens": int(nv.sum())}
    gc = np.asarray(t["codes"])
    res["codes_ok"] = bool(gc.shape == oc.shape and np.array_equal(gc, oc))
    if not res["codes_ok"] and gc.shape == oc.shape:
        bad = np.argwhere(gc != oc)
        i = tuple(bad[0])
        res["codes_bad"] = int(len(bad))
        res["first_code_bad"] = ([int(x) for x in i], int(gc[i]), int(oc[i]))
    gs = np.asarray(t["scales"]).astype(np.float64)
    res["scales_ok"] = bool(gs.shape == osc.shape and np.array_equal(gs, osc))
    th = rope.inv_freq(d, t["rope_base"])
    sent = np.full((1, n, B, H, d), SENTINEL)
    ek, ev = paged.fetch_rotate_scatter(vals, t["delta_m"], th, t["pairing"], ids, sent, sent,
                                        t["out_fmt"], n_valid=nv)
    gk = to_f64(t["dst_k"], t["out_fmt"])
    gv = to_f64(t["dst_v"], t["out_fmt"])
    m = np.zeros((1, n, B), bool)
    m[0] = np.arange(B)[None, :] < nv[:, None]
    res["k_ok"], res["k_max_err"], res["k_bar"] = compare_k(gk[m], ek[m], t["out_fmt"])
    res["v_ok"], res["v_exact"] = compare_v(gv[m], ev[m], wire, t["out_fmt"], t["scale_dtype"])
    # padding rows of ragged blocks: never written, so still the sentinel
    res["padding_ok"] = bool(np.array_equal(gk[~m], ek[~m]) and np.array_equal(gv[~m], ev[~m]))
    res["ok"] = all(res[x] for x in ("codes_ok", "scales_ok", "k_ok", "v_ok", "padding_ok"))
    res["seconds"] = time.perf_counter() - t0
    return res


def default_procs(per_proc_bytes=2 << 30):
    """One process per core of the affinity mask, as many as half the free
    host memory holds at about 2 GB each."""
    cores = len(os.sched_getaffinity(0))
    try:
        free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        free = 16 << 30
    return max(1, min(cores, int(free / 2 // per_proc_bytes)))


class OraclePool:
    """check_chunk in spawned processes with a bounded window of chunks in
    flight; results() returns every chunk's report."""

    def __init__(self, procs=None, window=None):
        import multiprocessing as mp
        self.procs = procs or default_procs()
        self.window = window or 2 * self.procs
        self._saved = {k: os.environ.get(k) for k in THREAD_VARS}
        os.environ.update({k: "1" for k in THREAD_VARS})      # one thread per worker
        self._ex = ProcessPoolExecutor(max_workers=self.procs, mp_context=mp.get_context("spawn"))
        self._pending = set()
        self._done = []
        self.t0 = time.perf_counter()

    def submit(self, task):
        while len(self._pending) >= self.window:
            done, self._pending = wait(self._pending, return_when=FIRST_COMPLETED)
            self._done += [f.result() for f in done]
        self._pending.add(self._ex.submit(check_chunk, task))

    def results(self):
        """Every report since the last call (waits for the chunks in flight)."""
        done, _ = wait(self._pending)
        self._done += [f.result() for f in done]
        self._pending = set()
        out, self._done = self._done, []
        return out

    def close(self):
        self._ex.shutdown(wait=True, cancel_futures=True)
        for k, val in self._saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def summarize(results):
    """Totals over the chunk reports and the failing ones."""
    bad = [r for r in results if not r["ok"]]
    return {"chunks": len(results), "blocks": sum(r["blocks"] for r in results),
            "tokens": sum(r["tokens"] for r in results),
            "k_max_err": max((r["k_max_err"] for r in results), default=0.0),
            "v_exact": all(r["v_exact"] for r in results),
            "oracle_cpu_s": sum(r["seconds"] for r in results), "failed": bad[:3]}
