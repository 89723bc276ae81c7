"""The parallel oracle timing leg of bench.py (host only): spawned
single-threaded processes each time one oracle pass on their own sample, and
the leg reports aggregate bytes over the wall time."""
import bench
import workloads


def test_parallel_oracle_leg_runs_and_reports():
    w = workloads.qwen3_8b()
    blk = w.blocks[0]
    r = bench.cpu_baseline_parallel(w, blk, nb=4, procs=2)
    assert "unavailable" not in r, r
    assert r["cores"] == 2 and r["kind"] == "oracle" and r["unit"] == "GB/s"
    assert r["value"] > 0 and r["tokens_per_s"] > 0
    assert "2 processes x 1 layer x 4 of 2048 blocks" in r["sample"]


def test_parallel_oracle_shape_is_bounded():
    w = workloads.qwen3_8b()
    blk = w.blocks[0]
    single = {"sample_blocks": 2048, "seconds": 4.0}
    procs, nb = bench.parallel_oracle_shape(w, blk, single, budget_s=15.0, procs=4)
    assert 1 <= procs <= 4 and 16 <= nb <= blk.nb
    procs, nb = bench.parallel_oracle_shape(w, blk, {"sample_blocks": 16, "seconds": 100.0}, 15.0, 3)
    assert nb == 16


def test_parallel_oracle_leg_reports_a_failing_worker():
    """A worker that raises (here: an unknown source dtype) makes the leg an
    `unavailable` object instead of a number, without hanging the bench."""
    import copy
    w = copy.copy(workloads.qwen3_8b())
    w.src_dtype = "no-such-dtype"
    r = bench.cpu_baseline_parallel(w, w.blocks[0], nb=4, procs=2)
    assert "unavailable" in r and "value" not in r, r


def test_oracle_leg_of_the_per_layer_workloads():
    """The layered lines' oracle leg: one layer, the first blocks of one block
    size, the workload's wire and value distribution."""
    for name, wire in (("ragged", "int4"), ("llama3_70b", "fp8")):
        w = workloads.WORKLOADS[name]()
        r = bench.cpu_baseline_workload(w, w.blocks[0], wire, budget_s=0.3)
        assert r["kind"] == "oracle" and r["cores"] == 1 and r["unit"] == "GB/s"
        assert r["value"] > 0 and r["tokens_per_s"] > 0 and f"of {name}, {wire}" in r["sample"]
