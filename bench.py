"""Benchmark of the Lynx progressive KV quantizer hot path on one GB300.

One step = one pass of the whole path over the full worked-example cache
(94 layers x 4 KV heads x 131072 tokens x 128, bf16 K and V, ~23.5 GiB):
  lynx_quantize_pages (K, V) -> lynx_dequant_anchor (K, V) ->
  lynx_refine_residual (K, V) -> lynx_decode_attn through all 94 layers, anchor
  mode and full mode (batch 1, 64 query heads, group 16).
Inputs are seeded synthetic Laplace values with per-channel scales 10^U(-2,0)
and 2% outlier channels x100, generated on the device before timing; every
buffer is larger than L2, so no flush is needed between steps.

value = algorithmic bytes of the whole step / step time (GB/s). Per-kernel
GB/s, decode tokens/s and roofline fractions are reported alongside.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torchrun: every rank runs the same per-GPU workload (weak
scaling, no collective on the data path); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import lynx_synth as S  # noqa: E402

METRIC = "quantize/dequant HBM GB/s and decode-attn tokens/s vs HBM roofline (1 GB300)"
W3 = S.WORKLOADS[3]
HQ = 64
D = 128
# algorithmic bytes per element (K or V) and per (token, KV head)
B_QUANT = 2 + 0.5 + 0.5 + 8 / 256 + 4 / 32          # 3.15625
B_DEQ_ANCHOR = 0.5 + 8 / 256 + 4 / 32 + 2            # 2.65625
B_REFINE = 1.0 + 8 / 256 + 4 / 32 + 2                # 3.15625
B_ATTN_ANCHOR = 64 + 64 + 16 + 16 + 4 + 4            # 168
B_ATTN_FULL = B_ATTN_ANCHOR + 128                    # 296


def max_over_ranks(ms_step, world, device):
    """Per-step time of the whole job: the slowest rank's (every rank runs its
    own replica of the workload; no collective touches the data path)."""
    if world <= 1:
        return float(ms_step)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank, world, ms_step):
    """Weak scaling: every rank moves bytes_per_rank per step."""
    return world * bytes_per_rank / (ms_step * 1e-3) / 1e9


def measured_traffic(group, units_per_launch):
    """DRAM bytes per launch of `group` from the committed ncu capture, or None
    when there is none or the kernel source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(group)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
        return None
    return rec["bytes_per_unit"] * units_per_launch / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# reference arm / CPU baseline: the oracle on a bounded sample of the workload
# --------------------------------------------------------------------------

def oracle_sample(pages=128, heads=4, layer=0):
    """Inputs of a bounded sample: `heads` KV heads x `pages` pages of one layer."""
    T = pages * 256
    ks, vs = W3.scales(S.S_K), W3.scales(S.S_V)
    kx = S.laplace_bf16(W3.key(S.S_K), ks, W3.L, W3.H, W3.T, layers=[layer], heads=range(heads), t0=0, t1=T)
    vx = S.laplace_bf16(W3.key(S.S_V), vs, W3.L, W3.H, W3.T, layers=[layer], heads=range(heads), t0=0, t1=T)
    return kx, vx, W3.queries_bf16()


def oracle_step(orc, kx, vx, qb):
    """The same sequence of operations as one GPU step, on the sample; returns
    the algorithmic bytes it stands for."""
    _, H, T, _ = kx.shape
    k = orc.quantize(kx)
    v = orc.quantize(vx)
    for t in (k, v):
        orc.dequant(t, False)
        orc.dequant(t, True)
    table = np.arange(T // 256, dtype=np.int32)[None, :]
    ctx = np.array([T], np.int32)
    orc.decode_attn(qb, k, v, 0, table, ctx, D ** -0.5, False)
    orc.decode_attn(qb, k, v, 0, table, ctx, D ** -0.5, True)
    el = 2 * H * T * D
    return el * (B_QUANT + B_DEQ_ANCHOR + B_REFINE) + H * T * (B_ATTN_ANCHOR + B_ATTN_FULL)


def run_oracle(steps, warmup, pages, min_seconds=0.0):
    """The oracle on the sample: `steps` passes, and more until `min_seconds`
    have gone by. Returns (GB/s, seconds, threads, passes)."""
    import oracle as orc
    orc.build()
    kx, vx, qb = oracle_sample(pages=pages)
    for _ in range(warmup):
        oracle_step(orc, kx, vx, qb)
    t0 = time.perf_counter()
    nbytes = 0.0
    n = 0
    while n < steps or time.perf_counter() - t0 < min_seconds:
        nbytes += oracle_step(orc, kx, vx, qb)
        n += 1
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt, orc.num_threads(), n


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class Workload:
    def __init__(self, torch, lx, layers=None, device="cuda"):
        self.torch, self.lx = torch, lx
        L = W3.L if layers is None else layers
        self.L, self.H, self.T = L, W3.H, W3.T
        dev = torch.device(device)
        self.dev = dev
        gen = S.DeviceGenerator(device)
        self.x = {}
        for s in (S.S_K, S.S_V):
            x = torch.empty((L, self.H, self.T, D), dtype=torch.bfloat16, device=dev)
            gen.fill(x, W3.key(s), W3.scales(s)[:L])
            self.x[s] = x
        self.q = {s: lx.QuantizedKV.empty(L, self.H, self.T, dev) for s in (S.S_K, S.S_V)}
        self.dense = {s: torch.empty((L, self.H, self.T, D), dtype=torch.bfloat16, device=dev)
                      for s in (S.S_K, S.S_V)}
        qb = W3.queries_bf16()
        self.qt = torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16)
        self.table = torch.arange(self.T // 256, dtype=torch.int32, device=dev)[None, :].contiguous()
        self.ctx = torch.full((1,), self.T, dtype=torch.int32, device=dev)
        self.ws = torch.empty(lx.decode_attn_workspace(1, HQ, self.T // 256), dtype=torch.uint8, device=dev)
        self.out = {m: torch.empty((L, 1, HQ, D), dtype=torch.float32, device=dev) for m in (0, 1)}
        self.elements = L * self.H * self.T * D          # per tensor
        self.token_heads = L * self.H * self.T           # per attention pass

    def launches_per_step(self):
        return 6 + 2 * 2 * self.L

    GROUPS = ("quantize", "dequant_anchor", "refine", "decode_attn_anchor", "decode_attn_full")

    def units(self):
        """Each timed unit: (group name, callable issuing its library calls)."""
        lx = self.lx
        out = []
        for s in (S.S_K, S.S_V):
            out.append(("quantize", lambda s=s: lx.quantize_pages(self.x[s], self.q[s])))
        for s in (S.S_K, S.S_V):
            out.append(("dequant_anchor", lambda s=s: lx.dequant_anchor(self.q[s], self.dense[s])))
        for s in (S.S_K, S.S_V):
            out.append(("refine", lambda s=s: lx.refine_residual(self.q[s], self.dense[s])))
        for mode, name in ((lx.MODE_ANCHOR, "decode_attn_anchor"), (lx.MODE_FULL, "decode_attn_full")):
            def attn(mode=mode):
                for l in range(self.L):
                    lx.decode_attn(self.qt, self.q[S.S_K], self.q[S.S_V], l, self.table, self.ctx, D ** -0.5,
                                   mode, out=self.out[mode][l], workspace=self.ws)
            out.append((name, attn))
        return out

    def capture(self, only=None):
        """One CUDA graph per timed unit (the same library calls, replayed
        without per-call host overhead)."""
        torch = self.torch
        self.graphs = []
        for name, fn in self.units():
            if only is not None and name != only:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            self.graphs.append((name, g))
        torch.cuda.synchronize()

    def step(self, ev=None, only=None, graphs=True):
        """ev: optional dict name -> list of (start, end) event pairs to record;
        only: run just this kernel group (single-kernel measurements)."""
        torch = self.torch
        st = torch.cuda.current_stream()
        seq = self.graphs if graphs else [(n, f) for n, f in self.units() if only is None or n == only]
        for name, item in seq:
            run = item.replay if graphs else item
            if ev is None:
                run()
                continue
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            run()
            b.record(st)
            ev.setdefault(name, []).append((a, b))

    def algorithmic_bytes(self):
        e = self.elements
        return {
            "quantize": 2 * e * B_QUANT,
            "dequant_anchor": 2 * e * B_DEQ_ANCHOR,
            "refine": 2 * e * B_REFINE,
            "decode_attn_anchor": self.token_heads * B_ATTN_ANCHOR,
            "decode_attn_full": self.token_heads * B_ATTN_FULL,
        }


def e2e_measure(torch, lx, layers, steps, warmup):
    """End to end through the public API with host buffers: per step, the bf16
    K and V of `layers` layers go host->device from pinned memory, the whole
    path runs, and the planes, metadata and attention outputs come back."""
    wl = Workload(torch, lx, layers=layers)
    hx = {s: torch.empty(wl.x[s].shape, dtype=torch.bfloat16, pin_memory=True) for s in wl.x}
    for s in hx:
        hx[s].copy_(wl.x[s])
    hq = {s: {n: torch.empty(getattr(wl.q[s], n).shape, dtype=getattr(wl.q[s], n).dtype, pin_memory=True)
              for n in ("anchor", "residual", "page_meta", "chunk_meta")} for s in wl.q}
    hout = {m: torch.empty(wl.out[m].shape, dtype=torch.float32, pin_memory=True) for m in wl.out}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for d in hq.values() for t in d.values()) + \
        sum(t.numel() * t.element_size() for t in hout.values())

    # Layer by layer: the bf16 K and V of layer l go in on their own copy
    # streams while layer l - 1 is computed and layer l - 2's planes come
    # back, so the link's two directions and the kernels overlap (the section-4
    # point of overlapping transfer with compute). The work and the bytes are
    # those of the whole-tensor step.
    K_, V_ = S.S_K, S.S_V
    NH = 1                                           # copy streams per tensor (more were slower: 760 vs 870 GB/s)
    st_h = {(s, i): torch.cuda.Stream() for s in (K_, V_) for i in range(NH)}
    st_c, st_d = torch.cuda.Stream(), torch.cuda.Stream()
    L, Hh = wl.L, wl.H // NH

    def body():
        cur = torch.cuda.current_stream()
        for st in list(st_h.values()) + [st_c, st_d]:
            st.wait_stream(cur)
        for l in range(L):
            landed = []
            for (s, i), st in st_h.items():
                with torch.cuda.stream(st):
                    wl.x[s][l, i * Hh:(i + 1) * Hh].copy_(hx[s][l, i * Hh:(i + 1) * Hh], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(st)
                    landed.append(e)
            for e in landed:
                st_c.wait_event(e)
            with torch.cuda.stream(st_c):
                for s in (K_, V_):
                    lx.quantize_pages(wl.x[s][l:l + 1], wl.q[s].layers(l, l + 1), stream=st_c)
                for s in (K_, V_):
                    lx.dequant_anchor(wl.q[s].layers(l, l + 1), wl.dense[s][l:l + 1], stream=st_c)
                for s in (K_, V_):
                    lx.refine_residual(wl.q[s].layers(l, l + 1), wl.dense[s][l:l + 1], stream=st_c)
                for mode in (lx.MODE_ANCHOR, lx.MODE_FULL):
                    lx.decode_attn(wl.qt, wl.q[K_], wl.q[V_], l, wl.table, wl.ctx, D ** -0.5, mode,
                                   out=wl.out[mode][l], workspace=wl.ws, stream=st_c)
                done = torch.cuda.Event()
                done.record(st_c)
            st_d.wait_event(done)
            with torch.cuda.stream(st_d):
                for s in hq:
                    for n, t in hq[s].items():
                        t[l].copy_(getattr(wl.q[s], n)[l], non_blocking=True)
                for m in hout:
                    hout[m][l].copy_(wl.out[m][l], non_blocking=True)
        for st in list(st_h.values()) + [st_c, st_d]:
            cur.wait_stream(st)

    body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    one = graph.replay
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    total = sum(wl.algorithmic_bytes().values())
    # the host link alone, for the record: one plain pinned copy each way of
    # the K input (the e2e figure is bound by it)
    link = {}
    for name, dst, src in (("h2d_gbs", wl.x[K_], hx[K_]), ("d2h_gbs", hx[K_], wl.x[K_])):
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        link[name] = src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
    del wl, hx, hq, hout
    torch.cuda.empty_cache()
    return {"value": total / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "layers": layers, "link": link,
            "note": f"{layers} of the 94 layers per step (host buffers pinned), same path and byte accounting; "
                    "layer-pipelined: host-to-device, kernels and device-to-host of different layers overlap"}


def progressive_arrival(torch, lx, w=None, top=32, keep=False):
    """Progressive arrival: every layer starts as the anchor-only draft; residual
    planes land layer by layer in a seeded order. On each arrival the layer's
    dense K and V caches are refined in place and decode attention reruns over
    all layers, full mode for arrived layers and anchor mode for the rest.
    Returns a report per arrival: the arrived layer's output change (anchor ->
    full, max abs and relative L2) and the agreement of its top-`top` keys by
    score between the anchor and the full pass, plus per-arrival GPU time."""
    w = S.WORKLOADS[5] if w is None else w
    L, H, T, B, Hq = w.L, w.H, w.T, w.B, w.Hq
    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    x = torch.empty((L, H, T, D), dtype=torch.bfloat16, device=dev)
    qkv, dense = {}, {}
    for s in (S.S_K, S.S_V):
        gen.fill(x, w.key(s), w.scales(s))
        qkv[s] = lx.QuantizedKV.empty(L, H, T, dev)
        lx.quantize_pages(x, qkv[s])
        dense[s] = torch.empty((L, H, T, D), dtype=torch.bfloat16, device=dev)
        lx.dequant_anchor(qkv[s], dense[s])            # the draft cache
    del x
    qb = w.queries_bf16()
    qt = torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16)
    table = torch.arange(T // 256, dtype=torch.int32, device=dev)[None, :].repeat(B, 1).contiguous()
    ctx = torch.full((B,), T, dtype=torch.int32, device=dev)
    ws = torch.empty(lx.decode_attn_workspace(B, Hq, T // 256), dtype=torch.uint8, device=dev)
    sm = D ** -0.5

    def attn(l, mode, scores=None):
        return lx.decode_attn(qt, qkv[S.S_K], qkv[S.S_V], l, table, ctx, sm, mode, scores=scores, workspace=ws)

    def topk_set(sc):
        return torch.topk(sc, top, dim=-1).indices

    out_anchor, top_anchor = [], []
    sc = torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
    for l in range(L):
        out_anchor.append(attn(l, lx.MODE_ANCHOR, sc).clone())
        top_anchor.append(topk_set(sc))
    order = [int(v) for v in S.arrival_order(w)]
    arrived, report = set(), []
    for l in order:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s in (S.S_K, S.S_V):
            lx.refine_residual(qkv[s].layers(l, l + 1), dense[s][l:l + 1])
        arrived.add(l)
        outs = [attn(m, lx.MODE_FULL if m in arrived else lx.MODE_ANCHOR) for m in range(L)]
        e1.record()
        torch.cuda.synchronize()
        full = outs[l]
        attn(l, lx.MODE_FULL, sc)
        tf = topk_set(sc)
        agree = (tf[..., :, None] == top_anchor[l][..., None, :]).any(-1).float().sum(-1) / top
        d = (full - out_anchor[l]).double()
        report.append({
            "layer": l,
            "ms_refine_plus_attention": e0.elapsed_time(e1),
            "delta_max_abs": float(d.abs().max()),
            "delta_rel_l2": float(d.norm() / out_anchor[l].double().norm()),
            "top_agreement_mean": float(agree.mean()),
            "top_agreement_min": float(agree.min()),
            "pending_layers_unchanged": all(torch.equal(outs[m], out_anchor[m]) for m in range(L)
                                            if m not in arrived),
        })
    result = {"workload": w.name, "order": order, "top": top, "arrivals": report}
    if keep:
        result.update(qkv=qkv, dense=dense, qb=qb, outs=outs, out_anchor=out_anchor)
    return result


def append_report(args):
    """Quantize-on-append at the batched-decode workload's shape on the 94-layer
    model: the growing last page of each of 32 requests (ragged contexts,
    seeded physical pages) re-encoded for 94 layers x 8 KV heads per step
    (24,064 pages), one lynx_quantize_append call per tensor. Algorithmic bytes
    are the encoder's 3.15625 B per element. The oracle is timed on a sample of
    the same tails beside it."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx

    w = S.WORKLOADS[4]
    L, H, n = (args.layers or W3.L), w.H, w.B
    ctx, pool, table = S.batched_layout(w)
    last = (ctx - 1) // 256
    phys = torch.from_numpy(table[np.arange(n), last].astype(np.int32)).cuda()
    valid = torch.from_numpy((ctx - 256 * last).astype(np.int32)).cuda()

    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        sc = S.channel_scales(w.seed, S.S_K, 1, H, n_outliers=w.n_outliers, factor_log10=w.factor_log10)
        xs = S.laplace_bf16(w.key(S.S_K), sc, 1, H, 8 * 256)          # 64 sample tails
        pv = np.resize(valid.cpu().numpy(), 8)
        orc.quantize(xs, pv)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            orc.quantize(xs, pv)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * xs.size * B_QUANT / dt / 1e9, "unit": "GB/s", "cores": orc.num_threads(),
               "kind": "oracle", "sample": f"{H * 8} tail pages (8 KV heads x 8 tails), {reps} passes, {dt:.1f} s"}

    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    tails, qkv = {}, {}
    for s in (S.S_K, S.S_V):
        x = torch.empty((n, L, H, 256, D), dtype=torch.bfloat16, device=dev)
        sc = S.channel_scales(w.seed, s, n * L, H, n_outliers=w.n_outliers, factor_log10=w.factor_log10)
        gen.fill(x.view(n * L, H, 256, D), w.key(s), sc)
        tails[s] = x
        qkv[s] = lx.QuantizedKV.empty(L, H, pool * 256, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        for s in (S.S_K, S.S_V):
            lx.quantize_append(tails[s], phys, valid, qkv[s], dev_err=err)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    if int(err.item()) != 0:
        raise RuntimeError("lynx_quantize_append flagged a page")
    nbytes = 2 * n * L * H * 256 * D * B_QUANT
    hbm, peak_kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {"report": "append", "metric": "quantize-on-append HBM GB/s vs HBM roofline (1 GB300)", "value": gbs,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16 in, 4+4-bit planes", "data": "synthetic",
            "config": {"workload": f"{w.name} tails on a {L}-layer model", "requests": n, "layers": L,
                       "kv_heads": H, "pages_per_step": 2 * n * L * H, "l2": "inputs larger than L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "peak_kind": peak_kind, "traffic": None},
            "cpu_baseline": cpu, "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
    print(json.dumps(line))


def batched_report(args):
    """Batched decode attention at the batched-decode workload: 32 requests
    with seeded context lengths in [4K, 16K] (ragged last pages) on a seeded
    random page table, 8 KV heads, 64 query heads (GQA group 8), one layer.
    One call is one decode step of every request. Algorithmic bytes count the
    tokens each request attends to: 168 B (anchor) or 296 B (full) per (token,
    KV head). The oracle runs beside it on a sample of two requests."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx

    w = S.WORKLOADS[4]
    H, B, Hq = w.H, w.B, w.Hq
    ctx_np, pool, table_np = S.batched_layout(w)
    T = pool * 256
    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    qkv = {}
    x = torch.empty((1, H, T, D), dtype=torch.bfloat16, device=dev)
    for s_ in (S.S_K, S.S_V):
        gen.fill(x, w.key(s_), w.scales(s_))
        qkv[s_] = lx.QuantizedKV.empty(1, H, T, dev)
        lx.quantize_pages(x, qkv[s_])
    del x
    qb = w.queries_bf16()
    qt = torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16)
    table = torch.from_numpy(table_np).to(dev)
    ctx = torch.from_numpy(ctx_np.astype(np.int32)).to(dev)
    max_pages = table_np.shape[1]
    ws = torch.empty(lx.decode_attn_workspace(B, Hq, max_pages), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sm = D ** -0.5
    token_heads = int(ctx_np.sum()) * H
    hbm, peak_kind = peaks()
    modes = {}
    for mode, name, per in ((lx.MODE_ANCHOR, "anchor", B_ATTN_ANCHOR), (lx.MODE_FULL, "full", B_ATTN_FULL)):
        def call():
            lx.decode_attn(qt, qkv[S.S_K], qkv[S.S_V], 0, table, ctx, sm, mode, out=out, workspace=ws,
                           dev_err=err)
        for _ in range(max(args.warmup, 3)):
            call()
        torch.cuda.synchronize()
        reps = max(args.steps, 200)          # long enough for the clock sampler
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clk:
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = token_heads * per / (ms * 1e-3) / 1e9
        modes[name] = {"ms": ms, "GB/s": gbs, "frac_of_measured_hbm": gbs / hbm,
                       "request_steps_per_s": B / (ms * 1e-3), "kv_token_heads_per_s": token_heads / (ms * 1e-3),
                       "clocks": clk.summary()}
    if int(err.item()) != 0:
        raise RuntimeError("lynx_decode_attn flagged the page table or a context length")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        n_s, ctx_s = 2, 2048
        sc_k = S.channel_scales(w.seed, S.S_K, 1, 1, n_outliers=w.n_outliers, factor_log10=w.factor_log10)
        sc_v = S.channel_scales(w.seed, S.S_V, 1, 1, n_outliers=w.n_outliers, factor_log10=w.factor_log10)
        ks = orc.quantize(S.laplace_bf16(w.key(S.S_K), sc_k, 1, 1, ctx_s))
        vs = orc.quantize(S.laplace_bf16(w.key(S.S_V), sc_v, 1, 1, ctx_s))
        tb = np.tile(np.arange(ctx_s // 256, dtype=np.int32), (n_s, 1))
        cl = np.full(n_s, ctx_s, np.int32)
        qs = qb[:n_s, :Hq // H]
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            orc.decode_attn(qs, ks, vs, 0, tb, cl, sm, False)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * n_s * ctx_s * B_ATTN_ANCHOR / dt / 1e9, "unit": "GB/s", "cores": orc.num_threads(),
               "kind": "oracle", "sample": f"anchor mode, 1 KV head x 8 query heads, {n_s} requests x {ctx_s} "
                                           f"tokens, {reps} calls, {dt:.1f} s"}
    a = modes["anchor"]
    line = {"report": "batched", "metric": "batched decode attention: GB/s and decode steps/s vs HBM roofline (1 GB300)",
            "value": a["GB/s"], "unit": "GB/s", "n_gpus": 1, "steps": max(args.steps, 200),
            "warmup": max(args.warmup, 3), "ms_per_step": a["ms"], "higher_is_better": True,
            "dtype": "4+4-bit planes, fp32 accumulation", "data": "synthetic",
            "config": {"workload": f"{w.name}: {B} requests, contexts {int(ctx_np.min())}..{int(ctx_np.max())} "
                                   f"tokens, {H} KV heads, {Hq} query heads, one layer",
                       "token_heads_per_call": token_heads, "page_pool": pool, "max_pages": max_pages,
                       "l2": f"{token_heads * B_ATTN_ANCHOR / 1e6:.0f} MB read per anchor call, larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "decode_attn_anchor", "achieved": a["GB/s"], "peak": hbm,
                         "unit": "GB/s", "frac": a["GB/s"] / hbm, "peak_kind": peak_kind, "traffic": None},
            "modes": modes, "cpu_baseline": cpu, "gpu_launches": 2 * 2 * max(args.steps, 200),
            "clocks": a["clocks"]}
    print(json.dumps(line))


def split_stream_report(args):
    """Split-stream arrival (Lynx section 4) emulated on one GPU at the
    progressive-arrival workload's shape (8 layers x 8 KV heads x 64K tokens, 8
    requests sharing the context, 64 query heads): anchors and metadata cross
    an emulated link first (high-priority stream), residuals after
    (low-priority stream); each layer is decoded in anchor mode as soon as its
    anchors are in and in full mode once its residuals are in. Compared with
    the sequential baseline (whole cache, then full decode), unpaced and with
    the link paced to 400 and 100 Gb/s."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    from progressive_kv_cache_gb300 import split_stream as ss

    w = S.WORKLOADS[5]
    L, H, T, B, Hq = w.L, w.H, w.T, w.B, w.Hq
    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    src = {}
    x = torch.empty((L, H, T, D), dtype=torch.bfloat16, device=dev)
    for s in (S.S_K, S.S_V):
        gen.fill(x, w.key(s), w.scales(s))
        src[s] = lx.QuantizedKV.empty(L, H, T, dev)
        lx.quantize_pages(x, src[s])
    del x
    host = {s: ss.pinned_copy(src[s]) for s in src}
    dst = {s: lx.QuantizedKV.empty(L, H, T, dev) for s in src}
    qt = torch.from_numpy(w.queries_bf16().view(np.int16)).to(dev).view(torch.bfloat16)
    table = torch.arange(T // 256, dtype=torch.int32, device=dev)[None, :].repeat(B, 1).contiguous()
    ctx = torch.full((B,), T, dtype=torch.int32, device=dev)
    sm = D ** -0.5
    lx.decode_attn(qt, src[S.S_K], src[S.S_V], 0, table, ctx, sm, lx.MODE_FULL)   # first call: set-up
    torch.cuda.synchronize()
    a_bytes = sum(t.numel() * t.element_size() for q in src.values() for t in (q.anchor, q.page_meta, q.chunk_meta))
    r_bytes = sum(q.residual.numel() for q in src.values())
    runs = []
    for gbps in (None, 400.0, 100.0):
        best = None
        for _ in range(2 if gbps is not None else 4):
            _, _, t = ss.split_stream_decode(host[S.S_K], host[S.S_V], dst[S.S_K], dst[S.S_V], qt, table, ctx, sm,
                                             link_gbps=gbps, order=S.arrival_order(w))
            _, seq_ms = ss.sequential_decode(host[S.S_K], host[S.S_V], dst[S.S_K], dst[S.S_V], qt, table, ctx, sm,
                                             link_gbps=gbps)
            if best is None or t["anchor_decode_done"] < best[0]["anchor_decode_done"]:
                best = (t, seq_ms)
        t, seq_ms = best
        runs.append({"link_gbps": gbps, "ms": t, "sequential_ms": seq_ms,
                     "first_decode_speedup": seq_ms / t["anchor_decode_done"],
                     "full_decode_vs_sequential": t["full_decode_done"] / seq_ms})
    print(json.dumps({"report": "split-stream", "workload": w.name, "layers": L, "kv_heads": H, "tokens": T,
                      "batch": B, "q_heads": Hq, "anchor_bytes": a_bytes, "residual_bytes": r_bytes,
                      "runs": runs}))


def verify_report(args):
    """Multi-token verify attention at the Qwen3-235B-like layer shape (4 KV
    heads x 32K tokens, 64 query heads, batch 1) with a block of 64 draft
    positions: 4,096 query rows over the full cache, causal within the block.
    The dense contraction is tensor-bound: achieved = algorithmic FLOPs (QK^T
    and PV, 2 per multiply-add, causal counts) / kernel time, against the
    measured bf16 tensor peak (f16 operands: the same nominal rate). The
    acceptance proxy: per drafted position, the fraction of (head) outputs
    whose argmax channel agrees between the anchor-only and the full pass."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx

    w = S.WORKLOADS[2]
    H, T, Hq, Tq = w.H, w.T, w.Hq, 64
    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    x = torch.empty((1, H, T, D), dtype=torch.bfloat16, device=dev)
    qkv = {}
    for s in (S.S_K, S.S_V):
        gen.fill(x, w.key(s), w.scales(s))
        qkv[s] = lx.QuantizedKV.empty(1, H, T, dev)
        lx.quantize_pages(x, qkv[s])
    del x
    qb = S.laplace_bf16(S.key(w.seed, S.S_Q * 1000 + 64), np.ones((1, Tq * Hq, D), np.float32), 1, Tq * Hq, 1)
    qt = torch.from_numpy(qb.reshape(1, Tq, Hq, D).view(np.int16)).to(dev).view(torch.bfloat16)
    table = torch.arange(T // 256, dtype=torch.int32, device=dev)[None].contiguous()
    ctx = torch.full((1,), T, dtype=torch.int32, device=dev)
    ws = torch.empty(lx.verify_attn_workspace(1, Tq, Hq, T // 256), dtype=torch.uint8, device=dev)
    sm = D ** -0.5
    outs = {}
    for m in (lx.MODE_ANCHOR, lx.MODE_FULL):
        outs[m] = lx.verify_attn(qt, qkv[S.S_K], qkv[S.S_V], 0, table, ctx, sm, m, workspace=ws).clone()
    res = {}
    for name, m in (("full", lx.MODE_FULL), ("anchor", lx.MODE_ANCHOR)):
        for _ in range(max(args.warmup, 3)):
            lx.verify_attn(qt, qkv[S.S_K], qkv[S.S_V], 0, table, ctx, sm, m, workspace=ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clk:
            e0.record()
            for _ in range(args.steps):
                lx.verify_attn(qt, qkv[S.S_K], qkv[S.S_V], 0, table, ctx, sm, m, workspace=ws)
            e1.record()
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        visible = sum(T - Tq + i + 1 for i in range(Tq))
        flops = 4.0 * Hq * visible * D
        res[name] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                     "hbm_gbs": H * T * (B_ATTN_FULL if m == lx.MODE_FULL else B_ATTN_ANCHOR) / (ms * 1e-3) / 1e9,
                     "clocks": clk.summary()}
    agree = (outs[lx.MODE_ANCHOR].argmax(-1) == outs[lx.MODE_FULL].argmax(-1)).float().mean(dim=(0, 2))
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"] \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        kx = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, H, T, heads=[0], t0=0, t1=8192)
        vx = S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), 1, H, T, heads=[0], t0=0, t1=8192)
        kq, vq = orc.quantize(kx), orc.quantize(vx)
        qs = qb.reshape(1, Tq, Hq, D)[:, :4, : Hq // H]
        pt = np.arange(32, dtype=np.int32)[None]
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            orc.verify_attn(qs, kq, vq, 0, pt, np.array([8192], np.int32), sm, True)
            reps += 1
        dt = time.perf_counter() - t0
        fl = reps * 4.0 * (Hq // H) * sum(8192 - 4 + i + 1 for i in range(4)) * D
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
               "sample": f"1 KV head, 8K tokens, 4 draft positions x 16 heads, full mode, {reps} passes, {dt:.1f} s"}
    f = res["full"]
    print(json.dumps({
        "report": "verify", "metric": "verify attention TFLOP/s vs tensor roofline (1 GB300)",
        "value": f["tflops"], "unit": "TFLOP/s", "ms_per_call": f["ms"], "steps": args.steps,
        "config": {"workload": f"{w.name}, block of {Tq} draft positions", "kv_heads": H, "tokens": T,
                   "q_heads": Hq, "draft": Tq, "batch": 1},
        "roofline": {"bound": "tensor", "achieved": f["tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": f["tflops"] / peak, "peak_kind": "measured bf16 (f16 operands, same nominal rate)",
                     "note": "algorithmic FLOPs; the hi/lo split costs three MMAs per product"},
        "modes": res, "acceptance_proxy_per_position": [round(float(v), 4) for v in agree.cpu()],
        "acceptance_proxy_mean": float(agree.mean()), "cpu_baseline": cpu}))


ABLATION = [
    ("lynx (C=32, 4+4, alpha=255)", {}),
    ("C=16", {"chunk": 16}), ("C=64", {"chunk": 64}),
    ("alpha=15", {"alpha": 15.0}), ("alpha=63", {"alpha": 63.0}), ("alpha=1023", {"alpha": 1023.0}),
    ("split 2+4 (6-bit codes)", {"anchor_bits": 2, "residual_bits": 4}),
    ("split 3+3 (6-bit codes)", {"anchor_bits": 3, "residual_bits": 3}),
    ("split 6+2", {"anchor_bits": 6, "residual_bits": 2}),
    ("no page normalisation", {"flags": 1}), ("no chunk isolation", {"flags": 2}),
    ("no log map (linear grid)", {"alpha": 0.0}), ("no bias", {"flags": 4}), ("no sign-aware mapping", {"flags": 8}),
    ("lynx 4-bit code (split 2+2)", {"anchor_bits": 2, "residual_bits": 2}),
    ("uniform INT4 per page-channel", {"uniform_bits": 4}), ("uniform INT8 per page-channel", {"uniform_bits": 8}),
    ("uniform INT4 per token", {"uniform_bits": 4, "flags": 16}),
    ("uniform INT8 per token", {"uniform_bits": 8, "flags": 16}),
]


def ablation_report(args):
    """Section 7's unmeasured knobs on synthetic data: vNMSE (sum (x_hat - x)^2
    / sum x^2) of the anchor-only and the full reconstruction for each variant
    of the quantizer and for the uniform comparators, on the K and V of the
    Qwen3-235B-like layer (4 KV heads x 32K tokens, Laplace with outlier
    channels); the vNMSE of the attention output over that layer (section 5's
    measure); and the variant encoder's throughput on 2 layers of the full
    cache's shape (268 MB of bf16 per tensor, larger than L2)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx

    w = S.WORKLOADS[2]
    dev = torch.device("cuda")
    gen = S.DeviceGenerator()
    xs = {}
    for s_ in (S.S_K, S.S_V):
        xs[s_] = torch.empty((1, w.H, w.T, D), dtype=torch.bfloat16, device=dev)
        gen.fill(xs[s_], w.key(s_), w.scales(s_))
    # attention-output vNMSE: one decode step of B_Q requests x 64 query heads
    # over the layer, the reconstruction's output against the output over the
    # original (bf16) values, both through the same fp32 dense attention
    n_req = 8
    q = torch.from_numpy(w.queries_bf16(n_req, w.Hq).view(np.int16)).to(dev).view(torch.bfloat16)
    kf, vf = (xs[s_].view(w.H, w.T, D).float() for s_ in (S.S_K, S.S_V))
    o_ref = lx.dense_attn(q, kf, vf).double()
    ref_sq = float((o_ref * o_ref).sum())
    del kf, vf
    rows = []
    for name, kw in ABLATION:
        r = {"name": name, "knobs": kw}
        rec = {}
        for s_, lab in ((S.S_K, "k"), (S.S_V, "v")):
            g = lx.quantize_variant(xs[s_], recon=True, **kw)
            e = g["err"].sum(dim=(0, 1)).cpu().numpy()
            r[lab] = {"anchor": float(e[1] / e[0]), "full": float(e[2] / e[0])}
            rec[lab] = g
        r["attn"] = {}
        for part in ("anchor", "full"):
            o = lx.dense_attn(q, rec["k"]["x_" + part].view(w.H, w.T, D), rec["v"]["x_" + part].view(w.H, w.T, D))
            r["attn"][part] = float(((o.double() - o_ref) ** 2).sum()) / ref_sq
        del rec
        rows.append(r)
    by = {r["name"]: r for r in rows}
    base, two = "lynx (C=32, 4+4, alpha=255)", "lynx 4-bit code (split 2+2)"
    ratio = {  # vNMSE of uniform INT4 / vNMSE of a Lynx reconstruction from 4 bits a value
        f"{u} / lynx {lab_l}": {t: by[u][t]["full"] / by[l][t][part] for t in ("k", "v", "attn")}
        for u in ("uniform INT4 per page-channel", "uniform INT4 per token")
        for lab_l, l, part in (("anchor-only of 4+4", base, "anchor"), ("4-bit code (2+2)", two, "full"))}
    ratio.update({  # uniform INT8 / the full 8-bit Lynx reconstruction
        f"{u} / lynx full 4+4": {t: by[u][t]["full"] / by[base][t]["full"] for t in ("k", "v", "attn")}
        for u in ("uniform INT8 per page-channel", "uniform INT8 per token")})
    del xs
    # throughput: the base variant and the comparator, errors only
    wt = S.WORKLOADS[3]
    big = torch.empty((2, wt.H, wt.T, D), dtype=torch.bfloat16, device=dev)
    gen.fill(big, wt.key(S.S_K), wt.scales(S.S_K)[:2])
    elems = big.numel()
    hbm, kind = peaks()
    timing = {}
    for name, kw in (("lynx", {}), ("C=16", {"chunk": 16}), ("C=64", {"chunk": 64}), ("uniform INT4", {"uniform_bits": 4})):
        for _ in range(max(args.warmup, 3)):
            lx.quantize_variant(big, **kw)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(args.steps, 400)          # long enough for the clock sampler to see the region
        with ClockSampler(0) as clk:
            e0.record()
            for _ in range(reps):
                lx.quantize_variant(big, **kw)
            e1.record()
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        timing[name] = {"ms": ms, "gbs": 2.0 * elems / (ms * 1e-3) / 1e9, "clocks": clk.summary()}
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import variants as V
        xc = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, w.H, w.T, heads=[0], t0=0, t1=4096)
        xc = xc.reshape(1, 4096, D)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 8.0:
            V.encode(xc)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": 2.0 * xc.size * reps / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"1 KV head x 4096 tokens (16 pages), base variant, {reps} passes, {dt:.1f} s (numpy)"}
    g = timing["lynx"]["gbs"]
    print(json.dumps({
        "report": "ablation",
        "metric": "quantizer variants: vNMSE on synthetic KV, and the variant encoder's GB/s vs HBM roofline (1 GB300)",
        "value": g, "unit": "GB/s", "steps": args.steps,
        "config": {"workload": f"quality: {w.name} (K and V, {n_req} requests x {w.Hq} query heads for the "
                               f"attention output); throughput: 2 layers x {wt.H} KV heads x {wt.T} tokens (K), "
                               f"errors only",
                   "vnmse": "k, v: sum (x_hat - x)^2 / sum x^2; attn: sum (o_hat - o)^2 / sum o^2, o the fp32 "
                            "decode attention over the original bf16 K and V, o_hat over the reconstruction"},
        "roofline": {"bound": "hbm", "achieved": g, "peak": hbm, "unit": "GB/s", "frac": g / hbm,
                     "peak_kind": kind, "note": "algorithmic bytes: 2 B read per element, outputs negligible"},
        "timing": timing, "variants": rows, "uniform_int4_over_lynx_4bit_vnmse": ratio,
        "cpu_baseline": cpu}))


def realism(workloads=(2, 3, 4), pages=32):
    """How concentrated the synthetic values are inside each page-channel's
    range: for every (page, channel) of a sample, the width of the interval
    holding the central 50 % of its 256 values (25th to 75th percentile by
    rank), as a fraction of the page range max - min. The Lynx reading
    (section 2, "Not all bits are equal") reports that on real KV half the
    elements sit inside the middle 17 % of the value range. Host only: the
    seeded generator gives the same values the GPU draws. Per workload: the
    median and mean over the sampled page-channels of K and V, the median
    over outlier and over ordinary channels, and the share at or below 17 %."""
    import numpy as np
    import lynx_synth as S
    out = {}
    for wi in workloads:
        w = S.WORKLOADS[wi]
        T = w.T if w.T else S.batched_layout(w)[1] * S.PAGE
        fr, is_out = [], []
        for s in (S.S_K, S.S_V):
            sc = w.scales(s)
            base = np.median(sc, axis=-1, keepdims=True)
            for l, h in ((0, 0), (w.L - 1, w.H - 1)):
                xb = S.laplace_bf16(w.key(s), sc, w.L, w.H, T, layers=[l], heads=[h], t1=pages * S.PAGE)
                x = S.bf16_bits_to_f32(xb)[0, 0].reshape(pages, S.PAGE, S.D).astype(np.float64)
                xs = np.sort(x, axis=1)
                rng = xs[:, -1] - xs[:, 0]
                mid = xs[:, 3 * S.PAGE // 4 - 1] - xs[:, S.PAGE // 4]
                fr.append((mid / np.where(rng > 0, rng, 1)).ravel())
                is_out.append(np.broadcast_to(sc[l, h] > 5 * base[l, h], (pages, S.D)).ravel())
        fr, is_out = np.concatenate(fr), np.concatenate(is_out)
        out[w.name] = dict(median=float(np.median(fr)), mean=float(fr.mean()),
                           median_outlier_channels=float(np.median(fr[is_out])) if is_out.any() else None,
                           median_other_channels=float(np.median(fr[~is_out])),
                           share_at_or_below_17pct=float((fr <= 0.17).mean()),
                           page_channels=int(fr.size))
    return {"central_half_of_range": out, "page_reading": 0.17,
            "definition": "(x_(192) - x_(64)) / (max - min) over the 256 tokens of a page-channel"}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import progressive_kv_cache_gb300 as lx

    # CPU baseline first (rank 0 only, before any GPU work that could interfere)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, cores, n = run_oracle(1, 0, args.cpu_pages, min_seconds=10.0)
        cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"layer 0, {W3.H} KV heads x {args.cpu_pages} pages (K and V) of the full cache: "
                         f"encode, both decodes, decode attention both modes; {n} passes, {dt:.1f} s"}

    wl = Workload(torch, lx, layers=args.layers)
    only = args.only
    use_graphs = not args.no_graph
    wl.step(only=only, graphs=False)          # first calls: module load, kernel attributes
    torch.cuda.synchronize()
    if use_graphs:
        wl.capture(only=only)
    for _ in range(args.warmup):
        wl.step(only=only, graphs=use_graphs)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    ev = {}
    with ClockSampler(local) as clk:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.steps):
            wl.step(ev, only=only, graphs=use_graphs)
        end.record()
        torch.cuda.synchronize()
    ms_step = max_over_ranks(start.elapsed_time(end) / args.steps, world, "cuda")
    if world > 1:
        dist.barrier()

    nbytes = wl.algorithmic_bytes()
    if only is not None:
        nbytes = {only: nbytes[only]}
    hbm, peak_kind = peaks()
    per = {}
    for name, pairs in ev.items():
        tot = sum(a.elapsed_time(b) for a, b in pairs)            # ms over all steps
        n_launch = len(pairs)
        per_launch_ms = tot / n_launch
        gbs = nbytes[name] * args.steps / (tot * 1e-3) / 1e9
        rec = {"ms_per_step": tot / args.steps, "GB/s": gbs, "frac_of_measured_hbm": gbs / hbm,
               "frac_of_8tbs_nominal": gbs / 8000.0, "share": None, "timed_units": n_launch,
               "ms_per_timed_unit": per_launch_ms}
        if name.startswith("decode_attn"):
            rec["tokens_per_s"] = 1.0 / (tot / args.steps * 1e-3)   # batch 1: one token per pass
            rec["kv_token_heads_per_s"] = wl.token_heads / (tot / args.steps * 1e-3)
        per[name] = rec
    tot_all = sum(p["ms_per_step"] for p in per.values())
    for p in per.values():
        p["share"] = p["ms_per_step"] / tot_all
    dom = max(per, key=lambda n: per[n]["ms_per_step"])
    # one launch: one tensor (quantize, decoders) or one layer (attention, split + combine)
    if dom in ("quantize", "dequant_anchor", "refine"):
        launch_units, launch_bytes = wl.elements, nbytes[dom] / 2
        launch_ms = per[dom]["ms_per_timed_unit"]
    else:
        launch_units, launch_bytes = wl.H * wl.T, nbytes[dom] / wl.L
        launch_ms = per[dom]["ms_per_step"] / wl.L
    ach = launch_bytes / (launch_ms * 1e-3) / 1e9
    traffic = measured_traffic(dom, launch_units)
    total_bytes = sum(nbytes.values())
    wl_layers = wl.L
    value = whole_job_gbs(total_bytes, world, ms_step)

    e2e = None
    if not args.no_e2e and only is None:
        del wl
        torch.cuda.empty_cache()
        e2e = e2e_measure(torch, lx, args.e2e_layers, max(1, min(args.steps, 3)), 1)
        e2e["value"] *= world

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": W3.name if wl_layers == W3.L else f"{W3.name} (first {wl_layers} layers)",
                       "launch": "CUDA graph per kernel group" if use_graphs else "eager",
                       "layers": wl_layers, "kv_heads": W3.H, "tokens": W3.T, "head_dim": D,
                       "only": only,
                       "q_heads": HQ, "batch": 1, "io": "bf16 in, 4+4-bit planes, bf16 dense cache",
                       "parallelism": f"replicas x{world}", "l2": "every input larger than L2, no flush"},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                         "frac": ach / hbm, "peak_kind": peak_kind, "traffic": traffic,
                         "traffic_unit": "GB per launch", "algorithmic": launch_bytes / 1e9},
            "per_kernel": per,
            "decode_tokens_per_s": {m: per[f"decode_attn_{m}"]["tokens_per_s"] for m in ("anchor", "full")
                                    if f"decode_attn_{m}" in per},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": wl_launches(args.steps, wl_layers, only),
            "clocks": clk.summary(),
            "realism": {k: round(v["median"], 4) for k, v in realism()["central_half_of_range"].items()},
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def wl_launches(steps, L, only=None):
    # quantize x2, dequant x2, refine x2, attention split+combine x2 modes x L layers
    per = {"quantize": 2, "dequant_anchor": 2, "refine": 2, "decode_attn_anchor": 2 * L, "decode_attn_full": 2 * L}
    return steps * (sum(per.values()) if only is None else per[only])


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    v, dt, cores, _ = run_oracle(args.steps, args.warmup, args.ref_pages)
    sample = (f"layer 0, {W3.H} KV heads x {args.ref_pages} pages (K and V) of the full cache per step: "
              "encode, both decodes, decode attention both modes")
    line = {
        "metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": W3.name, "layers": W3.L, "kv_heads": W3.H, "tokens": W3.T, "head_dim": D,
                   "q_heads": HQ, "batch": 1, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-pages", type=int, default=512)
    ap.add_argument("--ref-pages", type=int, default=64)
    ap.add_argument("--e2e-layers", type=int, default=12)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["quantize", "dequant_anchor", "refine", "decode_attn_anchor",
                                       "decode_attn_full"], default=None,
                    help="time one kernel group only (for profiler captures on smaller cases)")
    ap.add_argument("--layers", type=int, default=None, help="layers of the cache (default: all 94)")
    ap.add_argument("--report", choices=["progressive", "append", "split-stream", "verify", "ablation", "batched",
                                         "realism"],
                    default=None,
                    help="progressive: residual layers arriving one by one (8 layers, 64K tokens); "
                         "append: quantize-on-append of 32 requests' tail pages over 94 layers x 8 KV heads; "
                         "split-stream: anchors then residuals over an emulated link, decode on anchors first; "
                         "verify: multi-token verify attention (64 draft positions, 32K context); "
                         "ablation: quantizer variants and uniform comparators, vNMSE and encoder GB/s; "
                         "batched: decode attention of 32 ragged requests, 8 KV heads, GQA group 8; "
                         "realism: share of each page-channel range holding the central half of the "
                         "synthetic values (host only)")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue every library call from Python instead of replaying CUDA graphs of them")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.report == "progressive":
        import torch
        import __graft_entry__
        __graft_entry__.build()
        import progressive_kv_cache_gb300 as lx
        print(json.dumps(progressive_arrival(torch, lx)))
    elif args.report == "append":
        append_report(args)
    elif args.report == "split-stream":
        split_stream_report(args)
    elif args.report == "verify":
        verify_report(args)
    elif args.report == "ablation":
        ablation_report(args)
    elif args.report == "batched":
        batched_report(args)
    elif args.report == "realism":
        print(json.dumps(realism()))
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
