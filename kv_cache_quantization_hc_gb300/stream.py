"""Layer-streamed evict + fetch between host memory and the GPU.

Pages: waiting for every layer of a long cache to arrive before computing
leaves the GPU idle; transferring layer l+1 into a staging buffer while layer
l is being processed hides most of the transfer ["HyperCache - Distributed
KV-cache quantization and relative RoPE reuse", "Core Design", layer-wise
pipelining paragraph].

``LayerStream`` applies that schedule to one pass of the hot path with host
buffers.  Per layer l it issues:

  copy stream A : host K/V of layer l  -> device ring slot l % R
  compute stream: hc_encode_fp8 / hc_encode_int4 (ring slot -> wire ring slot),
                  hc_fetch_rotate_scatter (wire -> device output ring slot)
  copy stream B : device output ring slot -> host K/V of layer l

with events so that layer l's compute waits for its upload, its download
waits for its compute, and a ring slot is reused only after its previous
reader finished.  Host-to-device and device-to-host copies run on separate
streams, so the two directions of the host link overlap each other and the
kernels.  The block tables and the rotation table are shared by all layers.

Torch provides the streams, events and buffers; every arithmetic step is a
C-ABI call.
"""
import torch

from . import hc
from .path import KVPath



class LayerStream:
    def __init__(self, path: KVPath, src_shape, src_dtype, dst_shape, dst_dtype, device,
                 ring=3):
        """``src_shape`` / ``dst_shape``: one layer's pool [num_slots, B, H, d]."""
        if path.L != 1:
            raise ValueError("LayerStream drives a single-layer KVPath per call")
        self.p = path
        self.ring = ring
        dev = torch.device(device)
        self.src = [(torch.empty(src_shape, dtype=src_dtype, device=dev),
                     torch.empty(src_shape, dtype=src_dtype, device=dev)) for _ in range(ring)]
        self.dst = [(torch.empty(dst_shape, dtype=dst_dtype, device=dev),
                     torch.empty(dst_shape, dtype=dst_dtype, device=dev)) for _ in range(ring)]
        self.codes = [torch.empty_like(path.codes) for _ in range(ring)]
        self.scales = [None if path.scales is None else torch.empty_like(path.scales)
                       for _ in range(ring)]
        self.up = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        self.compute = torch.cuda.Stream(device=dev)
        self.dev = dev

    def run(self, h_src_k, h_src_v, h_dst_k, h_dst_v, h_err=None, preserve_dst=True, passes=1,
            tables=()):
        """One pass over all layers: h_src_* [L, num_slots, B, H, d] pinned host
        tensors in, h_dst_* [L, ...] pinned host tensors out.  Enqueues
        everything and returns; the caller synchronizes.  If ``h_err`` (a pinned
        int32 tensor of one element) is given, the device error flag is copied
        into it after the last layer.

        Whole destination layers are copied back.  With ``preserve_dst`` (the
        default) each destination layer is first uploaded too, so slots the
        fetch does not write keep their host contents; a caller whose block
        table writes every slot of the destination can turn it off and save
        that upload.

        ``passes`` > 1 streams that many passes back to back with no join
        between them, so one pass's last downloads overlap the next pass's
        first uploads.  ``tables`` is a list of (device tensor, pinned host
        tensor) pairs, such as the block tables, uploaded at the start of
        every pass once the previous pass's last compute (which reads them)
        has finished."""
        L = h_src_k.shape[0]
        p = self.p
        n = passes * L
        uploaded = [None] * n
        computed = [None] * n
        downloaded = [None] * n
        cur = torch.cuda.current_stream(self.dev)
        for s in (self.up, self.down, self.compute):
            s.wait_stream(cur)
        for it in range(n):
            layer, slot = it % L, it % self.ring
            sk, sv = self.src[slot]
            dk, dv = self.dst[slot]
            with torch.cuda.stream(self.up):
                if layer == 0 and tables:
                    if it > 0:                              # the last pass's compute read them
                        self.up.wait_event(computed[it - 1])
                    for d_t, h_t in tables:
                        d_t.copy_(h_t, non_blocking=True)
                if it >= self.ring:                         # slot's previous reader done
                    self.up.wait_event(computed[it - self.ring])
                sk.copy_(h_src_k[layer], non_blocking=True)
                sv.copy_(h_src_v[layer], non_blocking=True)
                if preserve_dst:
                    if it >= self.ring:                     # output slot downloaded
                        self.up.wait_event(downloaded[it - self.ring])
                    dk.copy_(h_dst_k[layer], non_blocking=True)
                    dv.copy_(h_dst_v[layer], non_blocking=True)
                uploaded[it] = torch.cuda.Event()
                uploaded[it].record(self.up)
            self.compute.wait_event(uploaded[it])
            if it >= self.ring:                             # output slot downloaded
                self.compute.wait_event(downloaded[it - self.ring])
            if layer == 0:
                with torch.cuda.stream(self.compute):
                    p.build_table(stream=self.compute)
            desc_s = hc.paged_desc(sk)
            desc_d = hc.paged_desc(dk)
            p.encode(sk, sv, desc=desc_s, stream=self.compute, codes=self.codes[slot],
                     scales=self.scales[slot])
            p.fetch(dk, dv, desc=desc_d, stream=self.compute, codes=self.codes[slot],
                    scales=self.scales[slot])
            computed[it] = torch.cuda.Event()
            computed[it].record(self.compute)
            with torch.cuda.stream(self.down):
                self.down.wait_event(computed[it])
                h_dst_k[layer].copy_(dk, non_blocking=True)
                h_dst_v[layer].copy_(dv, non_blocking=True)
                downloaded[it] = torch.cuda.Event()
                downloaded[it].record(self.down)
        if h_err is not None:
            with torch.cuda.stream(self.down):
                self.down.wait_event(computed[n - 1])
                h_err.copy_(p.err, non_blocking=True)
        for s in (self.up, self.down, self.compute):
            cur.wait_stream(s)
