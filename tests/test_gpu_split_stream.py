"""Split-stream arrival on one GPU: anchors (and metadata) cross an emulated
link first, residuals after; decode attention runs in anchor mode per layer as
soon as its anchors are in and in full mode once its residuals are in (the
Lynx reading, section 4). Every arrived layer's anchor-mode and full-mode
output is checked against the oracle's fp64 decode attention over the
oracle's own encoding of the same inputs; the transported planes equal the
source bit for bit; the outputs equal those of the same calls on a
device-resident cache; and with a paced link the anchor-mode decode is done
before the residuals arrive."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_attn_close, attn_sensitivity, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu

W = S.WORKLOADS[5]


@pytest.fixture(scope="module")
def setup():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    from progressive_kv_cache_gb300 import split_stream as ss
    L, H, T, B, Hq = 3, 2, 2048, 2, 8
    src, orq = {}, {}
    for s in (S.S_K, S.S_V):
        sc = S.channel_scales(W.seed, s, L, H, n_outliers=W.n_outliers, factor_log10=W.factor_log10)
        x = S.laplace_bf16(W.key(s), sc, L, H, T)
        q = lx.QuantizedKV.empty(L, H, T)
        lx.quantize_pages(bf16_dev(x), q)
        src[s] = q
        orq[s] = x
    qb = W.queries_bf16(B, Hq)
    q = bf16_dev(qb)
    table_np = np.stack([np.arange(T // 256), np.arange(T // 256)[::-1]]).astype(np.int32)
    ctx_np = np.array([T, T - 300], np.int32)
    table, ctx = i32_dev(table_np), i32_dev(ctx_np)
    ref = {m: [lx.decode_attn(q, src[S.S_K], src[S.S_V], l, table, ctx, 128 ** -0.5, m) for l in range(L)]
           for m in (lx.MODE_ANCHOR, lx.MODE_FULL)}
    torch.cuda.synchronize()
    host = dict(x=orq, qb=qb, table=table_np, ctx=ctx_np)
    return lx, ss, src, q, table, ctx, ref, host


def _fresh(lx, src):
    L, H, T = src.shape
    return lx.QuantizedKV.empty(L, H, T)


@pytest.mark.parametrize("gbps", [None, 2.0])
def test_split_stream_matches_resident_cache(setup, gbps):
    lx, ss, src, q, table, ctx, ref, _ = setup
    hk, hv = ss.pinned_copy(src[S.S_K]), ss.pinned_copy(src[S.S_V])
    dk, dv = _fresh(lx, src[S.S_K]), _fresh(lx, src[S.S_V])
    out_a, out_f, t = ss.split_stream_decode(hk, hv, dk, dv, q, table, ctx, 128 ** -0.5, link_gbps=gbps,
                                             order=[2, 0, 1])
    for l in range(len(out_a)):
        assert torch.equal(out_a[l], ref[lx.MODE_ANCHOR][l])
        assert torch.equal(out_f[l], ref[lx.MODE_FULL][l])
    for a, b in ((dk, src[S.S_K]), (dv, src[S.S_V])):
        for name in ("anchor", "residual", "page_meta", "chunk_meta"):
            assert torch.equal(getattr(a, name), getattr(b, name))
    assert t["anchors_in"] <= t["residuals_in"] and t["anchors_in"] <= t["anchor_decode_done"]
    assert t["residuals_in"] <= t["full_decode_done"]
    if gbps is not None:
        assert t["anchor_decode_done"] < t["residuals_in"]


def test_sequential_baseline_matches(setup):
    lx, ss, src, q, table, ctx, ref, _ = setup
    hk, hv = ss.pinned_copy(src[S.S_K]), ss.pinned_copy(src[S.S_V])
    dk, dv = _fresh(lx, src[S.S_K]), _fresh(lx, src[S.S_V])
    outs, ms = ss.sequential_decode(hk, hv, dk, dv, q, table, ctx, 128 ** -0.5)
    assert ms > 0
    for l in range(len(outs)):
        assert torch.equal(outs[l], ref[lx.MODE_FULL][l])


def test_split_stream_outputs_against_oracle(setup, orc):
    """Each layer's anchor-mode output (decoded as soon as its anchors are in)
    and full-mode output (once its residuals are in), from the split-stream
    run itself, against the oracle's fp64 decode attention over the oracle's
    encoding of the same bf16 K and V."""
    lx, ss, src, q, table, ctx, ref, host = setup
    hk, hv = ss.pinned_copy(src[S.S_K]), ss.pinned_copy(src[S.S_V])
    dk, dv = _fresh(lx, src[S.S_K]), _fresh(lx, src[S.S_V])
    out_a, out_f, _ = ss.split_stream_decode(hk, hv, dk, dv, q, table, ctx, 128 ** -0.5, link_gbps=None,
                                             order=[1, 2, 0])
    torch.cuda.synchronize()
    kr, vr = orc.quantize(host["x"][S.S_K]), orc.quantize(host["x"][S.S_V])
    for l in range(len(out_a)):
        for full, got in ((False, out_a[l]), (True, out_f[l])):
            want = orc.decode_attn(host["qb"], kr, vr, l, host["table"], host["ctx"], 128 ** -0.5, full)
            E = attn_sensitivity(orc, host["qb"], kr, vr, l, host["table"], host["ctx"], 128 ** -0.5, full)
            assert_attn_close(got.cpu().numpy(), want, E, f"split-stream layer {l} {'full' if full else 'anchor'}")
