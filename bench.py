"""Benchmark of the KV wire codec hot path on the Qwen3-8B-shaped workload.

One step = one pass of the whole path over one batch: encode every cached
block of all 36 layers from the fp16 paged buffer to the FP8 E4M3 wire
(gather + amax + scale + quantize + wire write), build the delta-m rotation
table, and fetch every block back (dequantize + rotate K by delta-m +
scatter into a bf16 paged buffer through a shuffled block table).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is algorithmic bytes moved per second over
the whole job (all ranks), with inputs resident in HBM; `e2e` is the same
metric with the source copied from pinned host memory and the result copied
back inside the timed region; `cpu_baseline` / `--impl reference` time the
float64 oracle on the host cores on a bounded sample of the same workload.
`workloads` adds the two per-layer workloads, each call timed with CUDA
events: the Llama-3-70B-shaped layer-streamed fetch (80 layers, FP8, against
70% of the nominal 8 TB/s per layer) and the ragged INT4 sweep (36 layers,
blocks of 16 and 64); these run after the step's own timed region.
Under torchrun each rank runs an independent replica (weak scaling: the path
has no exchange step).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV fetch+rotate+scatter GB/s and tokens/s; % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = {
    "k_encode": ["encode.cu", "encode_common.cuh", "crc_math.h", "crc_fields.cuh", "hc_internal.cuh",
                 "fastdiv.h"],
    "k_fetch": ["fetch_impl.cuh", "fetch_fp8.cu", "hc_internal.cuh", "fastdiv.h"],
    "k_encode_fp8_rows": ["encode_rows.cu", "encode_common.cuh", "hc_internal.cuh", "fastdiv.h"],
    "k_fetch_fp8_rows": ["fetch_impl.cuh", "fetch_fp8_rows.cu", "hc_internal.cuh", "fastdiv.h"],
    "k_crc32": ["crc32.cu", "crc_fields.cuh", "crc_math.h", "hc_internal.cuh"],
}
# Integer ALU pipe of one SM: 4 schedulers x 16 lanes (ncu's pct_of_peak for
# the pipe is taken against this rate); GB300's maximum SM clock.
ALU_LANES_PER_SM = 64
MAX_SM_MHZ = 2070.0
CODECS = {
    "fp8": "FP8 E4M3 wire (per-block-head fp32 scale)",
    "fp8_rows": "FP8 E4M3 wire (per-token-head fp16 scale, the pages' frame layout)",
}


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max_sum(seconds, units, backend_group=None):
    """(max seconds over ranks, sum of units over ranks); identity at N = 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return seconds, units
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([float(units)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel):
    """Hash of the kernel's sources with comments and blank space removed, so
    that a profile stays valid across edits that cannot change the kernel."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "kv_cache_quantization_hc_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_values(kernel, workload, keys):
    """Per-launch counters recorded by ncu in profiles/<kernel>_<workload>.md
    (lines `key: value`), if the kernel's sources are unchanged since the
    capture; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    want = tuple(keys) + ("source_sha256", "capture")
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(want):
            k, v = line.split(":", 1)
            vals[k.strip().strip("-* `")] = v.strip().strip("`")
    if vals.get("source_sha256") != kernel_source_hash(kernel):
        return None
    try:
        out = {k: int(vals[k]) for k in keys}
    except (KeyError, ValueError):
        return None
    out["capture"] = vals.get("capture")
    out["source"] = f"profiles/{kernel}_{workload}.md"
    return out


def profiled_traffic(kernel, workload):
    """DRAM traffic of one launch recorded by ncu in profiles/ (a capture of
    the full-size launch), if the kernel's sources are unchanged since; else
    None.  Returns {"traffic", "read", "write", "capture", "source"}."""
    v = profiled_values(kernel, workload, ("dram_read_bytes_per_launch", "dram_write_bytes_per_launch"))
    if v is None:
        return None
    rd, wr = v["dram_read_bytes_per_launch"], v["dram_write_bytes_per_launch"]
    return {"traffic": rd + wr, "read": rd, "write": wr, "capture": v["capture"], "source": v["source"]}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7], float(parts[7])))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r[3] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in loaded for n, v in zip(names, r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


# ------------------------------------------------------------------ workload
def algorithmic_bytes(w, blk, codec="fp8"):
    """Bytes the method must move, per kernel, for one call over all layers."""
    L, H, d, T, NB = w.L, w.H, w.d, blk.tokens(), blk.nb
    src_b = {"f32": 4, "f16": 2, "bf16": 2}[w.src_dtype]
    out_b = {"f32": 4, "f16": 2, "bf16": 2}[w.out_dtype]
    kv_elems = 2 * L * T * H * d
    codes = kv_elems
    scales = L * NB * 2 * H * 4 if codec == "fp8" else 2 * L * T * H * 2
    n_distinct = len(np.unique(blk.delta_m))
    table = n_distinct * (d // 2) * 8
    encode = kv_elems * src_b + codes + scales + NB * 4
    fetch = codes + scales + kv_elems * out_b + table + NB * 3 * 4
    return {"encode": encode, "table": table + n_distinct * 4, "fetch": fetch}


def setup_device(w, blk, device, codec="fp8"):
    import torch
    from kv_cache_quantization_hc_gb300 import path as kvpath
    import workloads
    src_k = workloads.device_pool(w, blk, range(w.L), 0, device)
    src_v = workloads.device_pool(w, blk, range(w.L), 1, device)
    shape = (w.L, blk.num_dst_slots, blk.B, w.H, w.d)
    dst_k = torch.empty(shape, dtype=torch.bfloat16, device=device)
    dst_v = torch.empty(shape, dtype=torch.bfloat16, device=device)
    p = kvpath.from_blocks(w, blk, codec, device=device, scale_dtype="f16")
    return p, src_k, src_v, dst_k, dst_v


def run_ours(args):
    import torch
    import __graft_entry__
    import workloads

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    __graft_entry__.build()

    w = workloads.qwen3_8b()
    if args.layers:
        w.L = args.layers
    blk = w.blocks[0]
    p, src_k, src_v, dst_k, dst_v = setup_device(w, blk, device, args.codec)
    nbytes = algorithmic_bytes(w, blk, args.codec)
    step_bytes = sum(nbytes.values())
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device=device)

    def step(ev=None):
        # KVPath.step's schedule, with events: the table (it needs only
        # delta-m) on a side stream beside the encode, after the work already
        # queued (an earlier fetch reads the table); the fetch waits for both.
        queued, built = torch.cuda.Event(), torch.cuda.Event()
        queued.record(stream)
        side.wait_event(queued)
        if ev: ev[2].record(side)
        p.build_table(stream=side)
        if ev: ev[3].record(side)
        built.record(side)
        if ev: ev[0].record(stream)
        p.encode(src_k, src_v, stream=stream)
        if ev: ev[1].record(stream)
        stream.wait_event(built)
        p.fetch(dst_k, dst_v, stream=stream)
        if ev: ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if p.error_bits():
        raise RuntimeError(f"device error flag {p.error_bits()}")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize(device)
        start.record(stream)
        for i in range(args.steps):
            step(events[i])
        end.record(stream)
        torch.cuda.synchronize(device)
        barrier()
    total_s = start.elapsed_time(end) / 1e3
    per = {"encode": [], "table": [], "fetch": []}
    for ev in events:
        # The table waits on the side stream for SM room (the persistent
        # encode fills every SM), so its own span is mostly queueing; what it
        # costs the step is the time it ends after the encode.  The fetch
        # starts at the later of the two ends.
        after = max(0.0, ev[1].elapsed_time(ev[3]))
        per["encode"].append(ev[0].elapsed_time(ev[1]) / 1e3)
        per["table"].append(after / 1e3)
        per["fetch"].append((ev[1].elapsed_time(ev[4]) - after) / 1e3)
    if p.error_bits():
        raise RuntimeError(f"device error flag {p.error_bits()}")

    max_s, total_bytes = reduce_max_sum(total_s, step_bytes * args.steps)
    _, total_tokens = reduce_max_sum(total_s, blk.tokens() * args.steps)
    peak, peak_kind = measured_peaks()
    kern = {}
    for k in ("encode", "table", "fetch"):
        avg = statistics.mean(per[k])
        kern[k] = {"avg_ms": avg * 1e3, "median_ms": statistics.median(per[k]) * 1e3,
                   "min_ms": min(per[k]) * 1e3,
                   "bytes_per_launch": nbytes[k], "gbs": nbytes[k] / avg / 1e9 if avg > 0 else None}
    kern["table"]["timing"] = "time the table ends after the encode (it runs on a side stream)"
    for k in ("encode", "fetch"):   # context tokens (all layers of the call) per second
        kern[k]["tokens_per_s"] = blk.tokens() / (kern[k]["avg_ms"] / 1e3)
    dominant = max(("encode", "fetch"), key=lambda k: kern[k]["avg_ms"])
    kname = {"encode": "k_encode", "fetch": "k_fetch"}[dominant]
    if args.codec == "fp8_rows":
        kname += "_fp8_rows"
    prof = profiled_traffic(kname, "qwen3_8b") if not args.layers else None
    achieved = kern[dominant]["gbs"]

    crc = run_crc(args, p, device, src_k, src_v) if args.crc else None
    e2e = None
    if "e2e" in args.legs:
        e2e = run_e2e(args, w, blk, p, src_k, src_v, dst_k, dst_v, step_bytes, device,
                      device_step_s=total_s / args.steps)
    wl = None
    if "workloads" in args.legs and not args.layers:
        del p, src_k, src_v, dst_k, dst_v
        torch.cuda.empty_cache()
        with ClockSampler(local) as wl_clocks:
            wl = workload_lines(args, device)
        wl["clocks"] = wl_clocks.summary()
    cpu = None
    if "cpu" in args.legs and rank == 0 and world == 1:
        cpu = cpu_baseline(w, blk, budget_s=args.cpu_seconds)
        if args.cpu_procs != 1:
            procs, nb = parallel_oracle_shape(w, blk, cpu, args.cpu_seconds, max(args.cpu_procs, 0))
            cpu["parallel"] = cpu_baseline_parallel(w, blk, nb, procs)

    if rank == 0:
        line = {
            "metric": METRIC, "value": total_bytes / max_s / 1e9, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": max_s / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"qwen3_8b: {w.L} layers x {w.H} KV heads x d{w.d}, "
                                   f"{blk.tokens()} tokens, block {blk.B}, fp16 paged -> "
                                   f"{CODECS[args.codec]} -> bf16 paged, delta-m +4096, "
                                   f"half-split RoPE base 1e6, shuffled block tables",
                       "layers": w.L, "tokens": blk.tokens(), "block_size": blk.B,
                       "storage": {"source": w.src_dtype, "wire": "e4m3",
                                   "scales": "f32 per block-head" if args.codec == "fp8" else "f16 per token-head",
                                   "destination": w.out_dtype},
                       "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (working set %.1f GB per step)" % (step_bytes / 1e9),
                       "parallelism": f"replicas x{world}"},
            "tokens_per_s": total_tokens / max_s,
            "hbm_frac": total_bytes / max_s / 1e9 / world / peak,
            "hbm_frac_nominal": total_bytes / max_s / 1e9 / world / NOMINAL_HBM_GBS,
            "kernels": kern,
            "roofline": {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None if prof is None else prof["traffic"],
                         "traffic_detail": prof,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, a 1:1 copy)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "nominal_peak": f"{NOMINAL_HBM_GBS:.0f} GB/s, the nominal ~8 TB/s HBM3e "
                                         f"figure (frac is against the measured copy peak)",
                         "algorithmic_bytes_per_launch": nbytes[dominant]},
            "gpu_launches": 3 * args.steps,
            "clocks": clocks.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        if crc is not None:
            line["crc32"] = crc
        if wl is not None:
            line["workloads"] = wl
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def crc_alu_roofline(p, seconds, sms):
    """The CRC kernel against its bound, the integer ALU pipe: ALU-pipe
    warp instructions of one full-size launch (ncu, recorded in profiles/)
    over the live launch time, against SMs x 64 lanes x the maximum SM
    clock.  None unless the recorded launch is this one (the Qwen3-8B FP8
    wire, as many units) and the kernel is unchanged since."""
    if p.wire_name != "fp8":
        return None
    v = profiled_values("k_crc32", "qwen3_8b", ("alu_warp_instructions_per_launch", "units_per_launch"))
    if v is None or v["units_per_launch"] != p.L * p.nb:
        return None
    achieved = v["alu_warp_instructions_per_launch"] * 32 / seconds / 1e12
    peak_t = sms * ALU_LANES_PER_SM * MAX_SM_MHZ * 1e6 / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak_t,
            "unit": "T integer-ALU thread instructions/s", "frac": achieved / peak_t,
            "alu_warp_instructions_per_launch": v["alu_warp_instructions_per_launch"],
            "peak_rule": f"{sms} SMs x {ALU_LANES_PER_SM} ALU lanes x {MAX_SM_MHZ:.0f} MHz",
            "source": v["source"]}


def run_crc(args, p, device, src_k, src_v):
    """CRC-32 of the step's wire (one unit per (layer, block): its codes, then
    its scales), timed alone with CUDA events after the step's own timing.
    For the FP8 wire, also the encode with the fused per-slab CRC
    (hc_encode_fp8_crc) against the plain encode."""
    import torch
    stream = torch.cuda.current_stream(device)
    out = torch.empty(p.L * p.nb, dtype=torch.int32, device=device)
    nbytes = p.codes.numel() * p.codes.element_size() + p.scales.numel() * p.scales.element_size()
    for _ in range(3):
        p.crc32(out, stream)
    reps = max(3, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        p.crc32(out, stream)
        b.record(stream)
    torch.cuda.synchronize(device)
    avg = statistics.mean(a.elapsed_time(b) / 1e3 for a, b in evs)
    peak, _ = measured_peaks()
    out_d = {"kernel": "k_crc32", "units": p.L * p.nb, "bytes_per_launch": nbytes, "launches": reps,
             "avg_ms": avg * 1e3, "gbs": nbytes / avg / 1e9, "frac": nbytes / avg / 1e9 / peak,
             "bound": "integer ALU: field extraction for the 5-bit table lookups (the traffic is "
                      "read-only HBM)",
             "roofline": crc_alu_roofline(
                 p, avg, torch.cuda.get_device_properties(device).multi_processor_count)}
    if args.codec == "fp8":
        slab_crc = torch.empty((p.L, p.nb, 2, p.H), dtype=torch.int32, device=device)

        def timed(fn):
            for _ in range(3):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in ev:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize(device)
            return statistics.mean(a.elapsed_time(b) / 1e3 for a, b in ev)
        plain = timed(lambda: p.encode(src_k, src_v, stream=stream))
        fused = timed(lambda: p.encode(src_k, src_v, stream=stream, crc=slab_crc))
        out_d["fused_encode"] = {"kernel": "k_encode (fused slab CRC)", "units": slab_crc.numel(),
                                 "encode_ms": plain * 1e3, "encode_with_crc_ms": fused * 1e3,
                                 "separate_crc_ms": avg * 1e3}
    return out_d


def run_e2e(args, w, blk, p, src_k, src_v, dst_k, dst_v, step_bytes, device, device_step_s=None):
    """Same step through the C ABI with host buffers, layer-streamed (the
    public LayerStream schedule): per layer, the fp16 source is copied from
    pinned host memory, encoded and fetched, and the bf16 result copied back;
    uploads, kernels and downloads of neighbouring layers overlap on three
    streams.  The block tables are uploaded every step as well, and the steps
    are streamed back to back (one step's last downloads overlap the next
    step's first uploads).  Every copy is inside the timed region.  `overlap` compares the step with its parts run
    alone (whole upload, the device step, whole download): hidden_frac is the
    share of the shorter parts' time that the pipeline hid (1 = the step takes
    only as long as its longest part)."""
    import copy
    import torch
    from kv_cache_quantization_hc_gb300 import path as kvpath
    from kv_cache_quantization_hc_gb300.stream import LayerStream
    stream = torch.cuda.current_stream(device)
    h_src_k = torch.empty(src_k.shape, dtype=src_k.dtype, pin_memory=True)
    h_src_v = torch.empty(src_v.shape, dtype=src_v.dtype, pin_memory=True)
    h_src_k.copy_(src_k)
    h_src_v.copy_(src_v)
    h_dst_k = torch.empty(dst_k.shape, dtype=dst_k.dtype, pin_memory=True)
    h_dst_v = torch.empty(dst_v.shape, dtype=dst_v.dtype, pin_memory=True)
    w1 = copy.copy(w)
    w1.L = 1
    p1 = kvpath.from_blocks(w1, blk, args.codec, device=device, scale_dtype="f16")
    ls = LayerStream(p1, src_k.shape[1:], src_k.dtype, dst_k.shape[1:], dst_k.dtype, device)
    tables = [p1.src_slots, p1.dst_slots, p1.delta_m, p1.delta_idx]
    h_tables = [t.cpu().pin_memory() for t in tables]
    h2d = sum(t.numel() * t.element_size() for t in (h_src_k, h_src_v, *h_tables))
    d2h = sum(t.numel() * t.element_size() for t in (h_dst_k, h_dst_v)) + 4
    h_err = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    steps = max(1, min(args.steps, args.e2e_steps))

    def passes(n):
        # n steps streamed back to back: every step uploads its block tables
        # and sources and downloads its results; the shuffled destination
        # table covers every slot (checked by the full-size parity test), so
        # the destination need not be uploaded
        ls.run(h_src_k, h_src_v, h_dst_k, h_dst_v, h_err, preserve_dst=False, passes=n,
               tables=list(zip(tables, h_tables)))

    passes(2)
    torch.cuda.synchronize(device)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    passes(steps)
    b.record(stream)
    torch.cuda.synchronize(device)
    if int(h_err.item()):
        raise RuntimeError("device error flag set in e2e leg")
    secs, total = reduce_max_sum(a.elapsed_time(b) / 1e3, step_bytes * steps)
    overlap = None
    if device_step_s:
        # each part alone: the whole source up, the whole result down
        def alone(fn):
            # the best of three runs: a part's own time, free of interference
            fn()
            torch.cuda.synchronize(device)
            best = None
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(device)
                t = e0.elapsed_time(e1) / 1e3
                best = t if best is None else min(best, t)
            return best
        up = alone(lambda: (src_k.copy_(h_src_k, non_blocking=True), src_v.copy_(h_src_v, non_blocking=True)))
        down = alone(lambda: (h_dst_k.copy_(dst_k, non_blocking=True), h_dst_v.copy_(dst_v, non_blocking=True)))
        serial = up + device_step_s + down
        e2e_s = secs / steps
        longest = max(up, device_step_s, down)
        overlap = {"upload_ms": up * 1e3, "compute_ms": device_step_s * 1e3, "download_ms": down * 1e3,
                   "serial_ms": serial * 1e3, "e2e_ms": e2e_s * 1e3,
                   "hidden_frac": (serial - e2e_s) / (serial - longest) if serial > longest else None}
    return {"value": total / secs / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": secs / steps * 1e3,
            "schedule": "layer-streamed: upload l+1 / compute l / download l-1 on three streams; "
                        "steps streamed back to back",
            "overlap": overlap}


# ------------------------------------------------------------------ oracle timing
def oracle_sample(w, blk, n_blocks, seed=0):
    """A bounded sample of the workload for the oracle: one layer, the first
    n_blocks blocks, source drawn on the host with the workload's distribution."""
    r = np.random.default_rng(seed)
    B, H, d = blk.B, w.H, w.d
    from oracle.numerics import round_to
    shape = (1, n_blocks, B, H, d)
    k = round_to(r.standard_normal(shape) * 0.5, w.src_dtype)
    v = round_to(r.standard_normal(shape) * 0.5, w.src_dtype)
    return k, v


def time_oracle_step(w, blk, k, v):
    """One oracle pass over the sample: encode FP8, decode, rotate+scatter."""
    from oracle import paged, rope
    nb = k.shape[1]
    th = rope.inv_freq(w.d, w.rope_base)
    t0 = time.perf_counter()
    codes, scales = paged.encode_fp8(k, v, np.arange(nb))
    vals = paged.decode_fp8(codes, scales)
    dm_vals = np.unique(blk.delta_m[:nb])
    paged.delta_sincos_table(dm_vals, th)
    out = np.zeros((1, nb, blk.B, w.H, w.d))
    paged.fetch_rotate_scatter(vals, blk.delta_m[:nb], th, w.pairing, np.arange(nb), out, out,
                               w.out_dtype)
    return time.perf_counter() - t0


def sample_bytes(w, blk, nb):
    sub = type(blk)(blk.B, blk.src_slots[:nb], blk.dst_slots[:nb], blk.n_valid[:nb],
                    blk.delta_m[:nb], nb, nb)
    import copy
    w1 = copy.copy(w)
    w1.L = 1
    return sum(algorithmic_bytes(w1, sub).values()), int(sub.tokens())


def cpu_baseline(w, blk, budget_s=15.0):
    nb = 16
    k, v = oracle_sample(w, blk, nb)
    t = time_oracle_step(w, blk, k, v)                 # calibrate
    nb = int(min(blk.nb, max(16, nb * budget_s / max(t, 1e-3) / 1.1)))
    k, v = oracle_sample(w, blk, nb)
    t = time_oracle_step(w, blk, k, v)
    b, toks = sample_bytes(w, blk, nb)
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"1 of {w.L} layers x {nb} of {blk.nb} blocks ({toks} tokens) of qwen3_8b, "
                      f"encode FP8 + table + fetch, float64 numpy, one thread; {t:.1f} s",
            "tokens_per_s": toks / t, "sample_blocks": nb, "seconds": t}


def _oracle_worker(i, w, blk, nb, barrier, out):
    """One process of the parallel oracle leg: its own seeded sample (a
    different layer's draw), then one timed oracle pass once every process
    has its sample ready."""
    try:
        k, v = oracle_sample(w, blk, nb, seed=1 + i)
        barrier.wait(timeout=120)
        t0 = time.perf_counter()
        time_oracle_step(w, blk, k, v)
        out.put((i, t0, time.perf_counter()))
    except Exception as e:                                  # reported by the parent
        out.put((i, None, repr(e)))


def cpu_baseline_parallel(w, blk, nb, procs):
    """The same oracle pass run by `procs` single-threaded processes at once,
    one sample (one layer's blocks) each: aggregate bytes / wall time from the
    first start to the last end.  Processes are spawned (never forked after
    CUDA work); BLAS and OpenMP pools are pinned to one thread each."""
    import multiprocessing as mp
    import queue
    ctx = mp.get_context("spawn")
    barrier, out = ctx.Barrier(procs), ctx.Queue()
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update({k: "1" for k in saved})
    ps = [ctx.Process(target=_oracle_worker, args=(i, w, blk, nb, barrier, out)) for i in range(procs)]
    res, why = {}, None
    try:
        for pr in ps:
            pr.start()
        deadline = time.monotonic() + 300
        while len(res) < procs and why is None:
            try:
                r = out.get(timeout=1.0)
                res[r[0]] = r
            except queue.Empty:
                # a process that ended without reporting (killed, failed to start)
                dead = [i for i, pr in enumerate(ps) if pr.exitcode is not None and i not in res]
                if dead:
                    why = f"process {dead[0]} exited with code {ps[dead[0]].exitcode}"
                elif time.monotonic() > deadline:
                    why = "timeout"
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
        for pr in ps:
            if why is not None and pr.is_alive():
                pr.terminate()
            pr.join(timeout=60)
            if pr.is_alive():
                pr.terminate()
    failed = [r[2] for r in res.values() if r[1] is None]
    if why is not None or failed:
        return {"unavailable": "a worker failed: " + (why or failed[0])}
    res = list(res.values())
    wall = max(r[2] for r in res) - min(r[1] for r in res)
    b, toks = sample_bytes(w, blk, nb)
    return {"value": procs * b / wall / 1e9, "unit": "GB/s", "cores": procs, "kind": "oracle",
            "sample": f"{procs} processes x 1 layer x {nb} of {blk.nb} blocks ({toks} tokens each) "
                      f"of qwen3_8b, encode FP8 + table + fetch, float64 numpy, one thread each; "
                      f"{wall:.1f} s wall",
            "tokens_per_s": procs * toks / wall}


def parallel_oracle_shape(w, blk, single, budget_s, procs=0):
    """Processes and blocks per process for the parallel oracle leg: one per
    core of this process's affinity (or `procs`), each sample sized for about
    half the single-thread budget, and the set held to half the free host
    memory (about 4 MB of float64 working set per 16-token block)."""
    cores = procs or len(os.sched_getaffinity(0))
    try:
        free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        free = 16 << 30
    per_block = 4e6 * blk.B / 16
    nb_time = int(single["sample_blocks"] * budget_s / 2 / max(single["seconds"], 1e-3))
    nb = max(16, min(blk.nb, nb_time))
    cores = max(1, min(cores, int(free / 2 / (per_block * nb))))
    return cores, nb


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads
    w = workloads.qwen3_8b()
    blk = w.blocks[0]
    nb = args.ref_blocks
    k, v = oracle_sample(w, blk, nb)
    for _ in range(args.warmup):
        time_oracle_step(w, blk, k, v)
    times = [time_oracle_step(w, blk, k, v) for _ in range(args.steps)]
    total = sum(times)
    b, toks = sample_bytes(w, blk, nb)
    value = b * args.steps / total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "qwen3_8b (bounded sample per step)", "layers": 1, "blocks": nb},
        "tokens_per_s": toks * args.steps / total,
        "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": 1,
                         "sample": f"1 layer x {nb} blocks ({toks} tokens) of qwen3_8b per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------ small workloads
SMALL_WIRES = ("fp8", "int4", "fp8_rows")


def small_bytes(w, blk, wire):
    """Algorithmic bytes of one pass (all layers) of a small workload."""
    if wire != "int4":
        return algorithmic_bytes(w, blk, wire)
    L, H, d, T, NB = w.L, w.H, w.d, blk.tokens(), blk.nb
    src_b = {"f32": 4, "f16": 2, "bf16": 2}[w.src_dtype]
    out_b = {"f32": 4, "f16": 2, "bf16": 2}[w.out_dtype]
    kv_elems = 2 * L * T * H * d
    wire_b = kv_elems // 2 + 2 * L * T * H * (d // 32) * 2      # g32 nibbles + fp16 scales
    n_distinct = len(np.unique(blk.delta_m))
    table = n_distinct * (d // 2) * 8
    return {"encode": kv_elems * src_b + wire_b + NB * 4, "table": table + n_distinct * 4,
            "fetch": wire_b + kv_elems * out_b + table + NB * 3 * 4}


def oracle_small(w, blk, k, v, wire):
    """The float64 oracle over the whole small workload for one wire."""
    from oracle import paged, rope
    th = rope.inv_freq(w.d, w.rope_base)
    t0 = time.perf_counter()
    if wire == "fp8":
        codes, scales = paged.encode_fp8(k, v, blk.src_slots, blk.n_valid)
        vals = paged.decode_fp8(codes, scales)
    elif wire == "int4":
        codes, scales = paged.encode_int4(k, v, blk.src_slots, blk.n_valid, 32, "f16")
        vals = paged.decode_int4(codes, scales, 32)
    else:
        codes, scales = paged.encode_fp8_rows(k, v, blk.src_slots, blk.n_valid, "f16")
        vals = paged.decode_fp8_rows(codes, scales)
    paged.delta_sincos_table(np.unique(blk.delta_m), th)
    out = np.zeros((w.L, blk.num_dst_slots, blk.B, w.H, w.d))
    paged.fetch_rotate_scatter(vals, blk.delta_m, th, w.pairing, blk.dst_slots, out, out,
                               w.out_dtype, n_valid=blk.n_valid)
    return time.perf_counter() - t0


def host_sample(w, nb, B, seed=0):
    """K and V for nb blocks of one layer, drawn on the host with the
    workload's value distribution and rounded to its source dtype."""
    from oracle.numerics import round_to
    r = np.random.default_rng(seed)
    shape = (1, nb, B, w.H, w.d)
    dist = w.extra.get("dist", ("normal", 1.0))

    def draw():
        if dist[0] == "student_t":
            x = r.standard_t(dist[1], shape) * dist[2]
        else:
            x = r.standard_normal(shape) * dist[1]
            if dist[0] == "normal_outliers":        # dist[2] channels per head, times dist[3]
                for h in range(w.H):
                    x[..., h, r.choice(w.d, size=dist[2], replace=False)] *= dist[3]
        return round_to(x, w.src_dtype)
    return draw(), draw()


def cpu_baseline_workload(w, blk, wire, budget_s=15.0):
    """The oracle on a bounded sample of a per-layer workload: one layer, the
    first blocks of one block size (as many as fit the budget), with the
    workload's wire, encode + table + fetch."""
    import copy
    w1 = copy.copy(w)
    w1.L = 1

    def sub(nb):
        ids = np.arange(nb, dtype=np.int32)
        return type(blk)(blk.B, ids, ids.copy(), blk.n_valid[:nb].copy(), blk.delta_m[:nb].copy(),
                         nb, nb)
    nb = 8
    k, v = host_sample(w1, nb, blk.B)
    t = oracle_small(w1, sub(nb), k, v, wire)        # calibrate
    nb = int(min(blk.nb, max(8, nb * budget_s / max(t, 1e-3) / 1.1)))
    s = sub(nb)
    k, v = host_sample(w1, nb, blk.B)
    t = oracle_small(w1, s, k, v, wire)
    b = sum(small_bytes(w1, s, wire).values())
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"1 of {w.L} layers x {nb} of {blk.nb} blocks of {blk.B} tokens "
                      f"({s.tokens()} tokens) of {w.name}, {wire} encode + table + fetch, "
                      f"float64 numpy, one thread; {t:.1f} s",
            "tokens_per_s": s.tokens() / t}


def run_small(args):
    """The small workloads (tiny, gqa_reorder): every wire's encode + table +
    fetch over all layers, with L2 flushed before every timed pass (their
    working sets fit in L2), and the oracle over the same inputs in full."""
    import torch
    import __graft_entry__
    import workloads
    from kv_cache_quantization_hc_gb300 import path as kvpath

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    __graft_entry__.build()
    w, _ = workloads.WORKLOADS[args.workload]()
    blk = w.blocks[0]
    stream = torch.cuda.current_stream(device)
    src_k = workloads.device_pool(w, blk, range(w.L), 0, device)
    src_v = workloads.device_pool(w, blk, range(w.L), 1, device)
    shape = (w.L, blk.num_dst_slots, blk.B, w.H, w.d)
    dst_k = torch.empty(shape, dtype=workloads.torch_dtype(w.out_dtype), device=device)
    dst_v = torch.empty_like(dst_k)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=device)
    peak, peak_kind = measured_peaks()
    res = {}
    with ClockSampler(local) as clocks:
        for wire in SMALL_WIRES:
            p = kvpath.from_blocks(w, blk, wire, device=device, scale_dtype="f16")
            nbytes = small_bytes(w, blk, wire)

            def step(ev=None):
                if ev: ev[0].record(stream)
                p.encode(src_k, src_v, stream=stream)
                if ev: ev[1].record(stream)
                p.build_table(stream=stream)
                if ev: ev[2].record(stream)
                p.fetch(dst_k, dst_v, stream=stream)
                if ev: ev[3].record(stream)

            for _ in range(args.warmup):
                flush.zero_()
                step()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
            torch.cuda.synchronize(device)
            for e in evs:
                flush.zero_()
                step(e)
            torch.cuda.synchronize(device)
            if p.error_bits():
                raise RuntimeError(f"device error flag {p.error_bits()}")
            t = {"encode": [], "table": [], "fetch": [], "step": []}
            for e in evs:
                t["encode"].append(e[0].elapsed_time(e[1]) / 1e3)
                t["table"].append(e[1].elapsed_time(e[2]) / 1e3)
                t["fetch"].append(e[2].elapsed_time(e[3]) / 1e3)
                t["step"].append(e[0].elapsed_time(e[3]) / 1e3)
            kern = {k: {"median_us": statistics.median(t[k]) * 1e6, "min_us": min(t[k]) * 1e6,
                        "bytes_per_launch": nbytes[k],
                        "gbs": nbytes[k] / statistics.median(t[k]) / 1e9} for k in nbytes}
            step_bytes = sum(nbytes.values())
            med = statistics.median(t["step"])
            # the same pass as a CUDA graph (table on a side branch, overlapping the encode)
            g = p.capture(src_k, src_v, dst_k, dst_v)
            for _ in range(args.warmup):
                flush.zero_()
                g.replay()
            gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
            for e in gev:
                flush.zero_()
                e[0].record(stream)
                g.replay()
                e[1].record(stream)
            torch.cuda.synchronize(device)
            if p.error_bits():
                raise RuntimeError(f"device error flag {p.error_bits()}")
            gt = [e[0].elapsed_time(e[1]) / 1e3 for e in gev]
            gmed = statistics.median(gt)
            res[wire] = {"gbs": step_bytes / gmed / 1e9, "hbm_frac": step_bytes / gmed / 1e9 / peak,
                         "median_step_us": gmed * 1e6, "min_step_us": min(gt) * 1e6,
                         "bytes_per_step": step_bytes, "tokens_per_s": blk.tokens() * w.L / gmed,
                         "eager": {"gbs": step_bytes / med / 1e9, "median_step_us": med * 1e6,
                                   "kernels": kern}}
            del g, p
    cpu = None
    if "cpu" in args.legs and rank == 0:
        k = src_k.double().cpu().numpy()
        v = src_v.double().cpu().numpy()
        cpu = {}
        for wire in SMALL_WIRES:
            ts = oracle_small(w, blk, k, v, wire)
            cpu[wire] = {"value": sum(small_bytes(w, blk, wire).values()) / ts / 1e9, "unit": "GB/s",
                         "seconds": ts}
        cpu = {"value": cpu["fp8"]["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole workload ({w.L} layers x {blk.nb} blocks), float64 numpy, "
                         f"one thread", "wires": cpu}
    if rank == 0:
        fp8 = res["fp8"]
        kern = fp8["eager"]["kernels"]
        dom = max(("encode", "fetch"), key=lambda k: kern[k]["median_us"])
        achieved = kern[dom]["gbs"]
        print(json.dumps({
            "metric": METRIC, "value": fp8["gbs"], "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": fp8["median_step_us"] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.L} layers x {w.H} KV heads x d{w.d}, "
                                   f"{blk.tokens()} tokens, block {blk.B}, {w.src_dtype} -> wire -> "
                                   f"{w.out_dtype}", "value_wire": "fp8",
                       "l2": f"flushed before every timed pass ({2 * l2 >> 20} MB write, not timed)",
                       "timing": "median of per-pass CUDA events; value: the pass replayed as a "
                                 "CUDA graph (KVPath.capture); wires.*.eager: the three calls "
                                 "launched one by one, timed per kernel"},
            "wires": res,
            "roofline": {"kernel": {"encode": "k_encode", "fetch": "k_fetch"}[dom], "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None,
                         "note": "launch-bound: the whole pass moves a few tens of MB"},
            "gpu_launches": 2 * 3 * args.steps * len(SMALL_WIRES),
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
        }))


# ------------------------------------------------------------------ per-layer workloads
def layered_bytes(w, blk, wire, group=32):
    """Algorithmic bytes of one layer's encode and fetch for one block size."""
    T, H, d, NB = blk.tokens(), w.H, w.d, blk.nb
    kv_elems = 2 * T * H * d
    src_b = {"f32": 4, "f16": 2, "bf16": 2}[w.src_dtype]
    out_b = {"f32": 4, "f16": 2, "bf16": 2}[w.out_dtype]
    if wire == "fp8":
        wire_b = kv_elems + NB * 2 * H * 4
    else:  # INT4, fp16 scales; padding rows carry no payload the method needs
        wire_b = kv_elems // 2 + 2 * T * H * (d // group) * 2
    n_distinct = len(np.unique(blk.delta_m))
    enc = kv_elems * src_b + wire_b + NB * 8
    fet = wire_b + kv_elems * out_b + n_distinct * (d // 2) * 8 + NB * 12
    return enc, fet


def fetch_target_us(fetch_bytes, frac=0.7, nominal_gbs=8000.0):
    """Time a fetch call may take at `frac` of the nominal ~8 TB/s HBM peak."""
    return fetch_bytes / (frac * nominal_gbs * 1e9) * 1e6


def measure_layered(w, wire, device, steps, warmup, K=2, distinct_layers=False):
    """Per-layer calls of a workload (one call per layer and block size), in
    three timed passes over all layers:

    * encode alone: the encodes back to back on one stream, each call between
      CUDA events on that stream;
    * fetch alone: the fetches back to back on a side stream, each timed;
    * layered: layer l encoded on encode stream l % K and then fetched on
      fetch stream l % K after an event, so neighbouring layers overlap (the
      layer-streamed schedule); timed as a whole.

    With `distinct_layers`, every layer has its own wire and its own slice of
    an all-layer destination cache (the layer-streamed fetch into one paged
    cache); otherwise each block size keeps a ring of 2K wire buffers
    (layer l encodes into slot l % 2K only after the fetch that last read it
    has finished) and each fetch stream writes its own destination pool.  The
    sources are two drawn layers per block size, used alternately (each is
    larger than L2)."""
    import torch
    import workloads
    from kv_cache_quantization_hc_gb300 import path as kvpath

    K = max(1, K)
    R = w.L if distinct_layers else 2 * K
    main = torch.cuda.current_stream(device)
    enc_streams = [main] + [torch.cuda.Stream(device=device) for _ in range(K - 1)]
    fet_streams = [torch.cuda.Stream(device=device) for _ in range(K)]
    odt = workloads.torch_dtype(w.out_dtype)
    groups = []
    for blk in w.blocks:
        p = kvpath.from_blocks(w, blk, wire, device=device, n_layers=R, scale_dtype="f16")
        srcs = [(workloads.device_pool(w, blk, range(i, i + 1), 0, device),
                 workloads.device_pool(w, blk, range(i, i + 1), 1, device)) for i in range(2)]
        n_dst = w.L if distinct_layers else K
        shape = (n_dst, blk.num_dst_slots, blk.B, w.H, w.d)
        dst = (torch.empty(shape, dtype=odt, device=device), torch.empty(shape, dtype=odt, device=device))
        p.build_table(stream=main)
        groups.append(dict(blk=blk, p=p, srcs=srcs, dst=dst, bytes=layered_bytes(w, blk, wire)))

    def wire_of(g, layer):
        i = layer % R
        return g["p"].codes[i:i + 1], g["p"].scales[i:i + 1]

    def dst_of(g, layer, fs_index):
        i = layer if distinct_layers else fs_index
        return g["dst"][0][i:i + 1], g["dst"][1][i:i + 1]

    def encode_pass(rec):
        for layer in range(w.L):
            for gi, g in enumerate(groups):
                codes, scales = wire_of(g, layer)
                sk, sv = g["srcs"][layer % 2]
                if rec: rec[layer][gi][0].record(main)
                g["p"].encode(sk, sv, stream=main, codes=codes, scales=scales)
                if rec: rec[layer][gi][1].record(main)

    def fetch_pass(rec):
        fs = fet_streams[0]
        fs.wait_stream(main)
        for layer in range(w.L):
            for gi, g in enumerate(groups):
                codes, scales = wire_of(g, layer)
                dk, dv = dst_of(g, layer, 0)
                if rec: rec[layer][gi][0].record(fs)
                g["p"].fetch(dk, dv, stream=fs, codes=codes, scales=scales)
                if rec: rec[layer][gi][1].record(fs)
        main.wait_stream(fs)

    def layered_pass():
        for st in enc_streams[1:] + fet_streams:
            st.wait_stream(main)
        fetched = {}
        for layer in range(w.L):
            es, fs = enc_streams[layer % K], fet_streams[layer % K]
            for gi, g in enumerate(groups):
                codes, scales = wire_of(g, layer)
                if layer >= R:                       # the slot's previous reader is done
                    es.wait_event(fetched[(layer - R, gi)])
                sk, sv = g["srcs"][layer % 2]
                g["p"].encode(sk, sv, stream=es, codes=codes, scales=scales)
                done = torch.cuda.Event()
                done.record(es)
                fs.wait_event(done)
                dk, dv = dst_of(g, layer, layer % K)
                g["p"].fetch(dk, dv, stream=fs, codes=codes, scales=scales)
                fetched[(layer, gi)] = torch.cuda.Event()
                fetched[(layer, gi)].record(fs)
        for st in enc_streams[1:] + fet_streams:
            main.wait_stream(st)

    def call_events():
        return [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in groups]
                for _ in range(w.L)]

    for _ in range(warmup):
        encode_pass(None)
        fetch_pass(None)
        layered_pass()
    torch.cuda.synchronize(device)
    enc_rec = [call_events() for _ in range(steps)]
    fet_rec = [call_events() for _ in range(steps)]
    for i in range(steps):
        encode_pass(enc_rec[i])
    for i in range(steps):
        fetch_pass(fet_rec[i])
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for _ in range(steps):
        layered_pass()
    end.record(main)
    torch.cuda.synchronize(device)
    if any(g["p"].error_bits() for g in groups):
        raise RuntimeError("device error flag set")
    pass_s = start.elapsed_time(end) / 1e3 / steps
    peak, _ = measured_peaks()
    per_kernel = {}
    for name, recs, bi in (("encode", enc_rec, 0), ("fetch", fet_rec, 1)):
        per_kernel[name] = {}
        for gi, g in enumerate(groups):
            ts = [r[layer][gi][0].elapsed_time(r[layer][gi][1]) / 1e3 for r in recs for layer in range(w.L)]
            med = statistics.median(ts)
            b = g["bytes"][bi]
            per_kernel[name][f"B{g['blk'].B}"] = {
                "median_us": med * 1e6, "min_us": min(ts) * 1e6, "calls": len(ts),
                "bytes_per_call": b, "gbs": b / med / 1e9, "frac": b / med / 1e9 / peak,
                # context tokens through all layers per second at this call's rate
                "tokens_per_s": g["blk"].tokens() / (med * w.L)}
    pass_bytes = sum(g["bytes"][0] + g["bytes"][1] for g in groups) * w.L
    tokens = sum(g["blk"].tokens() for g in groups)
    out = {"layers": w.L, "tokens": tokens, "wire": wire,
           "blocks": "/".join(f"{g['blk'].nb}xB{g['blk'].B}" for g in groups),
           "encode": per_kernel["encode"], "fetch": per_kernel["fetch"],
           "pass": {"gbs": pass_bytes / pass_s / 1e9, "frac": pass_bytes / pass_s / 1e9 / peak,
                    "ms_per_pass": pass_s * 1e3, "per_layer_us": pass_s / w.L * 1e6,
                    "tokens_per_s": tokens / pass_s, "bytes_per_pass": pass_bytes,
                    "schedule": f"layer l: encode on stream l % {K}, then fetch on fetch stream "
                                f"l % {K} after an event"},
           "timing": f"CUDA events on the launching stream, {steps} passes after {warmup} warm-up "
                     "passes; per-call figures from the passes of that kernel alone",
           "buffers": ("one wire and one destination-cache slice per layer" if distinct_layers else
                       f"wire ring of {R} per block size, {K} destination pools"),
           "peak_gbs": peak}
    for g in groups:
        del g["p"], g["srcs"], g["dst"]
    return out


def run_layered(args):
    """The per-layer workloads on their own (llama3_70b: FP8, one wire and
    destination slice per layer; ragged: --wire, rings), one JSON line."""
    import torch
    import __graft_entry__
    import workloads

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    __graft_entry__.build()
    w = workloads.WORKLOADS[args.workload]()
    if args.layers:
        w.L = args.layers
    wire = "fp8" if args.workload == "llama3_70b" else args.wire
    with ClockSampler(local) as clocks:
        res = measure_layered(w, wire, device, args.steps, args.warmup, K=args.layer_streams,
                              distinct_layers=args.workload == "llama3_70b")
    ps = res["pass"]
    print(json.dumps({
        "metric": METRIC, "value": ps["gbs"], "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ps["ms_per_pass"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.L} layers, per-layer encode + fetch, wire {wire}, "
                               f"blocks {res['blocks']}", "tokens": res["tokens"],
                   "layer_streams": args.layer_streams, "buffers": res["buffers"]},
        "tokens_per_s": ps["tokens_per_s"], "per_layer_us": ps["per_layer_us"],
        "kernels": {"encode": res["encode"], "fetch": res["fetch"]},
        "cpu_baseline": (cpu_baseline_workload(w, w.blocks[0], wire, args.cpu_seconds)
                         if "cpu" in args.legs and rank == 0 else None),
        "peak": res["peak_gbs"], "gpu_launches": 4 * w.L * len(w.blocks) * args.steps,
        "clocks": clocks.summary()}))


def workload_lines(args, device):
    """Compact objects for the two per-layer workloads, carried by the default
    line: the Llama-3-70B-shaped layer-streamed fetch (80 layers, FP8, against
    the 70%-of-8-TB/s time per layer) and the ragged INT4 sweep (36 layers,
    blocks of 16 and 64)."""
    import workloads
    steps = max(3, min(args.steps, 20))
    out = {}
    w = workloads.llama3_70b()
    r = measure_layered(w, "fp8", device, steps, 3, K=2, distinct_layers=True)
    f = r["fetch"]["B64"]
    r["fetch_target"] = {"max_us_per_layer": fetch_target_us(f["bytes_per_call"]),
                         "median_us_per_layer": f["median_us"],
                         "met": f["median_us"] <= fetch_target_us(f["bytes_per_call"]),
                         "rule": "70% of the nominal ~8 TB/s for one layer's fetch bytes"}
    out["llama3_70b"] = r
    w = workloads.ragged()
    out["ragged_int4"] = measure_layered(w, "int4", device, steps, 3, K=2)
    return out


def run_blend(args):
    """Drift-ranked token selection on 64 sequences x 2048 tokens x hidden 4096
    (bf16): drift of every token (both hidden-state arrays read once) and the
    top-15% selection per sequence, one hc_drift_select call per step."""
    import torch
    import __graft_entry__
    import workloads
    from kv_cache_quantization_hc_gb300 import hc

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    __graft_entry__.build()
    w = workloads.blend_selection()
    cached, fresh = workloads.blend_hidden(w, device)
    k = hc.selection_size(w.n_tokens)
    drift = torch.empty((w.n_seq, w.n_tokens), dtype=torch.float32, device=device)
    sel = torch.empty((w.n_seq, k), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    es = cached.element_size()
    nbytes = 2 * cached.numel() * es + drift.numel() * 4 + sel.numel() * 4
    for _ in range(max(args.warmup, 3)):
        hc.drift_select(cached, fresh, k, drift, sel, stream)
    torch.cuda.synchronize(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize(device)
        for a, b in evs:
            a.record(stream)
            hc.drift_select(cached, fresh, k, drift, sel, stream)
            b.record(stream)
        torch.cuda.synchronize(device)
    times = [a.elapsed_time(b) / 1e3 for a, b in evs]
    avg = statistics.mean(times)
    peak, peak_kind = measured_peaks()
    print(json.dumps({
        "metric": "drift-ranked token selection GB/s (layer-0 hidden states read once)",
        "value": nbytes / avg / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": avg * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.n_seq} sequences x {w.n_tokens} tokens x hidden "
                               f"{w.hidden}, {w.dtype}, k = {k} (ceil 15%)",
                   "bytes_per_step": nbytes,
                   "l2": "inputs larger than L2 (%.2f GB per step)" % (nbytes / 1e9)},
        "tokens_per_s": w.n_seq * w.n_tokens / avg,
        "roofline": {"kernel": "k_drift + k_select", "bound": "hbm", "achieved": nbytes / avg / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": nbytes / avg / 1e9 / peak, "traffic": None,
                     "peak_source": peak_kind},
        "gpu_launches": 2 * args.steps, "min_ms": min(times) * 1e3,
        "clocks": clocks.summary()}))


def run_hashing(args):
    """Host-side block digests (hc_block_digests, one core): the prefix and
    content BLAKE2b-128 digests of 445,722 token ids in blocks of 16 and of
    64, per tenant key; the oracle (hashlib) timed beside it."""
    from kv_cache_quantization_hc_gb300 import hc
    from oracle import hashing
    import __graft_entry__
    __graft_entry__.build()
    r = np.random.default_rng(7)
    tokens = r.integers(0, 151936, 445722).astype(np.int32)     # a Qwen3-sized vocabulary
    key = hc.tenant_key(b"bench master secret", "tenant-0")
    out = {}
    for B in (16, 64):
        hc.block_digests(tokens, B, key)
        reps = max(1, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(reps):
            hc.block_digests(tokens, B, key)
        dt = (time.perf_counter() - t0) / reps
        n_blocks = -(-len(tokens) // B)
        sample = tokens[: 64 * B]
        t1 = time.perf_counter()
        hashing.block_digests(sample, B, key)
        dto = (time.perf_counter() - t1) * len(tokens) / len(sample)
        out[f"B{B}"] = {"blocks_per_s": n_blocks / dt, "ms_per_pass": dt * 1e3,
                        "token_bytes_per_s": 4 * len(tokens) / dt,
                        "oracle_blocks_per_s": n_blocks / dto}
    print(json.dumps({
        "metric": "block digests per second (host, one core; two BLAKE2b-128 per block)",
        "value": out["B16"]["blocks_per_s"], "unit": "blocks/s", "n_gpus": 0, "steps": reps,
        "higher_is_better": True, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "445,722 token ids (vocabulary 151,936), blocks of 16 and 64, "
                               "tenant-keyed prefix and content digests"},
        "blocks": out, "cores": 1}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling a smaller case)")
    ap.add_argument("--workload", choices=["qwen3_8b", "llama3_70b", "ragged", "blend", "hashing",
                                           "tiny", "gqa_reorder"],
                    default="qwen3_8b",
                    help="qwen3_8b: the step the JSON line reports by default; llama3_70b / ragged "
                         "time the per-layer calls of the layer-streamed and ragged workloads; blend "
                         "times the drift-ranked token selection; hashing the host-side block "
                         "digests")
    ap.add_argument("--legs", default="device,e2e,cpu,workloads",
                    help="comma list of: device, e2e, cpu, workloads (the per-layer Llama-3-70B "
                         "and ragged INT4 objects of the default line)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--cpu-procs", type=int, default=0,
                    help="processes of the parallel oracle leg: 0 = one per core of the affinity "
                         "mask (bounded by host memory), 1 = skip it")
    ap.add_argument("--ref-blocks", type=int, default=16)
    ap.add_argument("--wire", choices=["int4", "fp8"], default="int4", help="ragged workload's wire format")
    ap.add_argument("--layer-streams", type=int, default=2,
                    help="per-layer workloads: encode and fetch streams the layers alternate over")
    ap.add_argument("--codec", choices=sorted(CODECS), default="fp8",
                    help="wire of the qwen3_8b step: per-block-head FP8 (default) or per-row FP8")
    ap.add_argument("--crc", action="store_true",
                    help="also time the CRC-32 of the step's wire (reported as crc32)")
    args = ap.parse_args(argv)
    args.legs = set(args.legs.split(","))
    args.warmup = max(args.warmup, 3)          # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "blend":
        run_blend(args)
    elif args.workload == "hashing":
        run_hashing(args)
    elif args.workload in ("tiny", "gqa_reorder"):
        run_small(args)
    elif args.workload != "qwen3_8b":
        run_layered(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
