"""The hot path composed from the C-ABI calls on torch-owned device buffers.

One ``KVPath`` holds, for one block size, the device-side block tables and the
wire / table / error-flag buffers of a call, and runs the three steps:

  encode  (hc_encode_fp8 or hc_encode_int4): paged source -> wire
  table   (hc_build_delta_sincos):           distinct delta-m -> (cos, sin)
  fetch   (hc_fetch_rotate_scatter):         wire -> rotated K, V in the paged destination

PyTorch supplies device memory and streams only; every arithmetic step runs
in libhc.so's kernels.
"""
import numpy as np
import torch

from . import hc

WIRES = {"fp8": hc.HC_WIRE_FP8, "int4": hc.HC_WIRE_INT4, "raw": hc.HC_WIRE_RAW,
         "fp8_rows": hc.HC_WIRE_FP8_ROWS}
_TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


class KVPath:
    def __init__(self, *, n_layers, H, d, B, n_blocks, src_slots, dst_slots, n_valid,
                 delta_m_distinct, delta_idx, wire, pairing, rope_base, paged_dtype,
                 group=32, scale_dtype="f16", device="cuda", inv_freq=None):
        self.L, self.H, self.d, self.B, self.nb = n_layers, H, d, B, n_blocks
        self.wire = WIRES[wire]
        self.wire_name = wire
        self.pairing = hc.PAIRING_NAMES[pairing]
        self.rope_base = float(rope_base)
        self.group = group
        self.scale_dtype = hc.DTYPE_NAMES[scale_dtype]
        self.paged_dtype = paged_dtype
        dev = torch.device(device)
        i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32), device=dev)
        self.src_slots = i32(src_slots)
        self.dst_slots = i32(dst_slots)
        full = n_valid is None or bool(np.all(np.asarray(n_valid) == B))
        self.n_valid = None if full else i32(n_valid)
        self.delta_m = i32(delta_m_distinct)
        self.delta_idx = i32(delta_idx)
        self.n_distinct = len(delta_m_distinct)
        self.inv_freq = None if inv_freq is None else torch.as_tensor(
            np.asarray(inv_freq, np.float64), device=dev)
        cshape, cdt, sshape = hc.wire_shapes(n_layers, n_blocks, H, B, d, self.wire, group)
        if self.wire == hc.HC_WIRE_RAW:
            self.codes = torch.zeros(cshape, dtype=_TORCH[paged_dtype], device=dev)
            self.scales = None
        else:
            self.codes = torch.zeros(cshape, dtype=torch.uint8, device=dev)
            sdt = torch.float32 if (self.wire == hc.HC_WIRE_FP8 or scale_dtype == "f32") else torch.float16
            self.scales = torch.zeros(sshape, dtype=sdt, device=dev)
        self.table = torch.zeros((max(self.n_distinct, 1), d // 2, 2), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    # -- steps ----------------------------------------------------------------
    def encode(self, src_k, src_v, desc=None, stream=None, codes=None, scales=None, crc=None):
        """Encode; with `crc` (device int32/uint32 [L, NB, 2, H], FP8 wire only)
        the same pass writes each slab's CRC-32 (its codes, then its scale)."""
        desc = desc or hc.paged_desc(src_k)
        codes = self.codes if codes is None else codes
        scales = self.scales if scales is None else scales
        if crc is not None and self.wire != hc.HC_WIRE_FP8:
            raise ValueError("the fused CRC is built for the FP8 wire")
        if self.wire == hc.HC_WIRE_FP8 and crc is not None:
            hc.hc_encode_fp8_crc(src_k, src_v, desc, self.src_slots, self.n_valid, self.nb,
                                 codes, scales, crc, self.err, stream)
        elif self.wire == hc.HC_WIRE_FP8:
            hc.hc_encode_fp8(src_k, src_v, desc, self.src_slots, self.n_valid, self.nb,
                             codes, scales, self.err, stream)
        elif self.wire == hc.HC_WIRE_INT4:
            hc.hc_encode_int4(src_k, src_v, desc, self.src_slots, self.n_valid, self.nb,
                              self.group, self.scale_dtype, codes, scales, self.err, stream)
        elif self.wire == hc.HC_WIRE_FP8_ROWS:
            hc.hc_encode_fp8_rows(src_k, src_v, desc, self.src_slots, self.n_valid, self.nb,
                                  self.scale_dtype, codes, scales, self.err, stream)
        else:
            raise ValueError("the RAW wire has no encode step")

    def build_table(self, stream=None):
        hc.hc_build_delta_sincos(self.delta_m, self.n_distinct, self.d, self.rope_base,
                                 self.inv_freq, self.table, stream)

    def fetch(self, dst_k, dst_v, desc=None, stream=None, codes=None, scales=None):
        desc = desc or hc.paged_desc(dst_k)
        codes = self.codes if codes is None else codes
        scales = self.scales if scales is None else scales
        hc.hc_fetch_rotate_scatter(self.wire, codes, scales, self.group, self.scale_dtype,
                                   self.table, self.delta_idx, self.n_distinct, self.pairing,
                                   self.dst_slots, self.n_valid, self.nb, dst_k, dst_v, desc,
                                   self.err, stream)

    def step(self, src_k, src_v, dst_k, dst_v, stream=None, side=None):
        """One pass: encode, then fetch, on `stream` (default: the current
        stream). The table depends only on delta-m, so it is built on the
        `side` stream (default: a stream of this path), overlapping the
        encode. The side stream first waits for the work already queued on
        `stream`, since an earlier fetch may still read the table. The fetch
        waits for the table."""
        stream = torch.cuda.current_stream(self.table.device) if stream is None else stream
        if side is None:
            if getattr(self, "_side", None) is None:
                self._side = torch.cuda.Stream(device=self.table.device)
            side = self._side
        queued, built = torch.cuda.Event(), torch.cuda.Event()
        queued.record(stream)
        side.wait_event(queued)
        self.build_table(stream=side)
        built.record(side)
        self.encode(src_k, src_v, stream=stream)
        stream.wait_event(built)
        self.fetch(dst_k, dst_v, stream=stream)

    def capture(self, src_k, src_v, dst_k, dst_v):
        """A CUDA graph of `step` over these buffers: replaying it runs the
        three kernels with no host work per launch, which is what bounds calls
        of a few tens of MB. The buffers must stay alive and in place while
        the graph is used."""
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=self.table.device)
        side = torch.cuda.Stream(device=self.table.device)
        cap.wait_stream(torch.cuda.current_stream(self.table.device))
        with torch.cuda.graph(g, stream=cap):
            self.step(src_k, src_v, dst_k, dst_v, stream=cap, side=side)
        return g

    def crc32(self, out=None, stream=None):
        """CRC-32 of every (layer, block)'s wire bytes: its codes for K and V,
        then its scales (device uint32 [n_layers * n_blocks], layer-major)."""
        L, nb = self.L, self.nb
        out = torch.empty(L * nb, dtype=torch.int32, device=self.codes.device) if out is None else out
        a_bytes = self.codes[0, 0].numel() * self.codes.element_size()
        if self.scales is None:
            hc.hc_crc32(self.codes, a_bytes, a_bytes, None, 0, 0, L * nb, out, stream)
        else:
            b_bytes = self.scales[0, 0].numel() * self.scales.element_size()
            hc.hc_crc32(self.codes, a_bytes, a_bytes, self.scales, b_bytes, b_bytes, L * nb, out,
                        stream)
        return out

    def error_bits(self):
        return int(self.err.item())


def from_blocks(w, blk, wire, device="cuda", n_layers=None, **kw):
    """KVPath for workload ``w`` and its Blocks entry ``blk``."""
    vals, idx = blk.distinct()
    return KVPath(n_layers=w.L if n_layers is None else n_layers, H=w.H, d=w.d, B=blk.B,
                  n_blocks=blk.nb, src_slots=blk.src_slots, dst_slots=blk.dst_slots,
                  n_valid=blk.n_valid, delta_m_distinct=vals, delta_idx=idx, wire=wire,
                  pairing=w.pairing, rope_base=w.rope_base, paged_dtype=w.out_dtype,
                  device=device, **kw)
