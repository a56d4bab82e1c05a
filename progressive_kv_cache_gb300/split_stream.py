"""Split-stream arrival of a quantized cache on one GPU.

The Lynx reading (section 4, "Speculation at the communication boundary")
sends the anchor planes first and the residual planes after them: decoding
starts on the anchor-only draft as soon as the anchors are in, and the cache is
refined when the residuals land. Here the network is emulated by host-to-device
copies from pinned memory, optionally paced to a link rate: anchors (with the
metadata) go first on a high-priority stream, residuals follow on a
low-priority one, layer by layer. Decode attention over each layer runs in
anchor mode as soon as that layer's anchors are in, and again in full mode once
its residuals are in. Every step of the path runs in the library's kernels;
this module only orders copies and launches.
"""
from __future__ import annotations

import time

import torch

from . import MODE_ANCHOR, MODE_FULL, QuantizedKV, decode_attn, decode_attn_workspace

__all__ = ["pinned_copy", "split_stream_decode", "sequential_decode"]


def pinned_copy(q: QuantizedKV) -> QuantizedKV:
    """A pinned host copy of a device-resident quantized tensor (the sender)."""
    def pin(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h
    return QuantizedKV(pin(q.anchor), pin(q.residual), pin(q.page_meta), pin(q.chunk_meta))


class _Link:
    """Issues copies in order, paced on the host to `gbps` gigabits per second
    (None: as fast as the copy engines go). Copies are split into pieces of at
    most `piece` bytes so that pacing is smooth."""

    def __init__(self, gbps, piece=8 << 20):
        self.rate = None if gbps is None else gbps * 1e9 / 8.0
        self.piece = piece
        self.sent = 0
        self.t0 = None

    def start(self):
        self.t0 = time.perf_counter()
        self.sent = 0

    def send(self, dst, src, stream):
        d, s = dst.reshape(-1).view(torch.uint8), src.reshape(-1).view(torch.uint8)
        for o in range(0, d.numel(), self.piece):
            n = min(self.piece, d.numel() - o)
            if self.rate is not None:
                wait = self.t0 + (self.sent + n) / self.rate - time.perf_counter()
                if wait > 0:
                    time.sleep(wait)
            with torch.cuda.stream(stream):
                d[o:o + n].copy_(s[o:o + n], non_blocking=True)
            self.sent += n


def _anchor_parts(q: QuantizedKV, l):
    return [q.anchor[l], q.page_meta[l], q.chunk_meta[l]]


def split_stream_decode(host_k: QuantizedKV, host_v: QuantizedKV, dev_k: QuantizedKV, dev_v: QuantizedKV,
                        q, page_table, ctx_lens, sm_scale, link_gbps=None, order=None):
    """Receive K and V (anchors first, then residuals, layer by layer in
    `order`) into dev_k/dev_v and decode: anchor-mode attention for a layer as
    soon as its anchors are in, full-mode attention once its residuals are in.
    Returns (outputs in anchor mode [L], outputs in full mode [L], timings in ms
    from the first copy: anchors in, anchor decode done, residuals in, full
    decode done)."""
    L = dev_k.shape[0]
    order = list(range(L)) if order is None else list(order)
    dev = q.device
    s_anchor = torch.cuda.Stream(device=dev, priority=-1)      # high priority
    s_resid = torch.cuda.Stream(device=dev, priority=0)        # low priority
    c_anchor = torch.cuda.Stream(device=dev, priority=-1)
    c_full = torch.cuda.Stream(device=dev, priority=0)
    B, Hq, _ = q.shape
    ws_a = torch.zeros(decode_attn_workspace(B, Hq, page_table.shape[1]), dtype=torch.uint8, device=dev)
    ws_f = torch.zeros_like(ws_a)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e_start, e_anchor_in, e_anchor_done, e_resid_in, e_full_done = ev(), ev(), ev(), ev(), ev()
    a_in = [torch.cuda.Event() for _ in range(L)]
    r_in = [torch.cuda.Event() for _ in range(L)]
    out_a = [torch.empty((B, Hq, 128), dtype=torch.float32, device=dev) for _ in range(L)]
    out_f = [torch.empty_like(out_a[0]) for _ in range(L)]
    cur = torch.cuda.current_stream(dev)
    for s in (s_anchor, s_resid, c_anchor, c_full):
        s.wait_stream(cur)

    link = _Link(link_gbps)
    e_start.record(s_anchor)
    link.start()
    for l in order:                                   # anchor stream
        for hq, dq in ((host_k, dev_k), (host_v, dev_v)):
            for dst, src in zip(_anchor_parts(dq, l), _anchor_parts(hq, l)):
                link.send(dst, src, s_anchor)
        a_in[l].record(s_anchor)
        c_anchor.wait_event(a_in[l])
        decode_attn(q, dev_k, dev_v, l, page_table, ctx_lens, sm_scale, MODE_ANCHOR, out=out_a[l],
                    workspace=ws_a, stream=c_anchor)
    e_anchor_in.record(s_anchor)
    e_anchor_done.record(c_anchor)
    s_resid.wait_stream(s_anchor)                     # the link carries residuals after the anchors
    for l in order:                                   # residual stream
        link.send(dev_k.residual[l], host_k.residual[l], s_resid)
        link.send(dev_v.residual[l], host_v.residual[l], s_resid)
        r_in[l].record(s_resid)
        c_full.wait_event(r_in[l])
        c_full.wait_event(a_in[l])
        decode_attn(q, dev_k, dev_v, l, page_table, ctx_lens, sm_scale, MODE_FULL, out=out_f[l],
                    workspace=ws_f, stream=c_full)
    e_resid_in.record(s_resid)
    e_full_done.record(c_full)
    for s in (s_anchor, s_resid, c_anchor, c_full):
        cur.wait_stream(s)
    torch.cuda.synchronize(dev)
    t = {"anchors_in": e_start.elapsed_time(e_anchor_in), "anchor_decode_done": e_start.elapsed_time(e_anchor_done),
         "residuals_in": e_start.elapsed_time(e_resid_in), "full_decode_done": e_start.elapsed_time(e_full_done)}
    return out_a, out_f, t


def sequential_decode(host_k: QuantizedKV, host_v: QuantizedKV, dev_k: QuantizedKV, dev_v: QuantizedKV,
                      q, page_table, ctx_lens, sm_scale, link_gbps=None):
    """The baseline without the split: the whole cache crosses the link, then
    every layer is decoded in full mode. Returns (outputs [L], ms)."""
    L = dev_k.shape[0]
    dev = q.device
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    B, Hq, _ = q.shape
    ws = torch.zeros(decode_attn_workspace(B, Hq, page_table.shape[1]), dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    link = _Link(link_gbps)
    e0.record(s)
    link.start()
    for l in range(L):
        for hq, dq in ((host_k, dev_k), (host_v, dev_v)):
            for dst, src in zip(_anchor_parts(dq, l) + [dq.residual[l]], _anchor_parts(hq, l) + [hq.residual[l]]):
                link.send(dst, src, s)
    outs = [torch.empty((B, Hq, 128), dtype=torch.float32, device=dev) for _ in range(L)]
    for l in range(L):
        decode_attn(q, dev_k, dev_v, l, page_table, ctx_lens, sm_scale, MODE_FULL, out=outs[l], workspace=ws,
                    stream=s)
    e1.record(s)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    return outs, e0.elapsed_time(e1)
