"""GPU parity of the fused-dequant paged decode attention (lynx_decode_attn)
against the oracle's fp64 attention, anchor-only and full, within 2e-3 absolute."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_attn_close, attn_sensitivity, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def _cache(lx, orc, w, L, H, T, valid=None):
    out = {}
    for s in (S.S_K, S.S_V):
        xb = S.laplace_bf16(w.key(s), w.scales(s)[:L, :H], L, H, T)
        q = lx.QuantizedKV.empty(L, H, T)
        lx.quantize_pages(bf16_dev(xb), q, None if valid is None else i32_dev(valid))
        out[s] = (q, orc.quantize(xb, valid))
    return out


def _run(lx, orc, cache, qb, layer, table, ctx, mode, scores=False):
    """GPU output, oracle output (or (output, scores)), GPU scores, device error
    word, and the per-output score sensitivity E of the tolerance."""
    B, Hq, _ = qb.shape
    (kq, kr), (vq, vr) = cache[S.S_K], cache[S.S_V]
    sc = None
    if scores:
        sc = torch.empty((B, Hq, table.shape[1] * 256), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lx.decode_attn(bf16_dev(qb), kq, vq, layer, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode,
                         scores=sc, dev_err=err)
    ref = orc.decode_attn(qb, kr, vr, layer, table, ctx, 128 ** -0.5, mode == lx.MODE_FULL, want_scores=scores)
    E = attn_sensitivity(orc, qb, kr, vr, layer, table, ctx, 128 ** -0.5, mode == lx.MODE_FULL)
    return out.cpu().numpy(), ref, (None if sc is None else sc.cpu().numpy()), int(err.item()), E


def _check(out, ref, E, label="decode attention"):
    assert_attn_close(out, ref, E, label)


@pytest.mark.parametrize("mode", [0, 1])
def test_one_page(lx, orc, mode):
    w = S.WORKLOADS[1]
    cache = _cache(lx, orc, w, 1, 1, 256)
    qb = w.queries_bf16(1, 1)
    out, ref, _, e, E = _run(lx, orc, cache, qb, 0, np.zeros((1, 1), np.int32), np.array([256]), mode)
    _check(out, ref, E)
    assert e == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_qwen3_235b_like_layer(lx, orc, mode):
    """4 KV heads, 32K tokens, 64 query heads (group 16), batch 1."""
    w = S.WORKLOADS[2]
    cache = _cache(lx, orc, w, w.L, w.H, w.T)
    qb = w.queries_bf16()
    table = np.arange(w.pages, dtype=np.int32)[None, :]
    out, ref, _, e, E = _run(lx, orc, cache, qb, 0, table, np.array([w.T]), mode)
    _check(out, ref, E)
    assert e == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_batched_ragged_permuted(lx, orc, mode):
    """32 requests, ctx in [4K, 16K], 8 KV heads, 64 query heads, permuted pages."""
    w = S.WORKLOADS[4]
    ctx, pool, table = S.batched_layout(w)
    cache = _cache(lx, orc, w, 1, w.H, pool * 256)
    qb = w.queries_bf16()
    out, ref, _, e, E = _run(lx, orc, cache, qb, 0, table, ctx, mode)
    _check(out, ref, E)
    assert e == 0


def test_scores_and_edges(lx, orc):
    w = S.Workload("t", 300, L=2, H=2, T=6 * 256, n_outliers_fixed=4, factor_log10=(1, 2))
    cache = _cache(lx, orc, w, 2, 2, 6 * 256)
    qb = w.queries_bf16(5, 8)
    table = np.array([[5, 0, 3], [1, 2, 4], [0, 1, 2], [3, 3, 3], [4, 5, 0]], np.int32)
    ctx = np.array([0, 1, 700, 768, 513], np.int32)
    for mode in (0, 1):
        out, ref, sc, e, E = _run(lx, orc, cache, qb, 1, table, ctx, mode, scores=True)
        _check(out, ref[0], E)
        assert np.all(out[0] == 0)
        rs = ref[1]
        fin = np.isfinite(rs)
        assert np.array_equal(np.isfinite(sc), fin)
        assert np.all(np.isneginf(sc[~fin]))
        assert np.allclose(sc[fin], rs[fin], rtol=1e-4, atol=1e-3)
        assert e == 0


def test_device_errors_are_flagged_not_fatal(lx, orc):
    w = S.Workload("t", 301, L=1, H=1, T=2 * 256, n_outliers_fixed=2)
    cache = _cache(lx, orc, w, 1, 1, 512)
    (kq, _), (vq, _) = cache[S.S_K], cache[S.S_V]
    qb = bf16_dev(w.queries_bf16(2, 2))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = i32_dev(np.array([[0, 7], [1, 0]]))        # page 7 is outside the 2-page pool
    ctx = i32_dev(np.array([400, 100]))
    out = lx.decode_attn(qb, kq, vq, 0, table, ctx, 0.1, lx.MODE_FULL, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lx.DEVERR_PAGE
    assert torch.isfinite(out).all()
    err.zero_()
    lx.decode_attn(qb, kq, vq, 0, i32_dev(np.array([[0, 1], [1, 0]])), i32_dev(np.array([600, 100])), 0.1,
                   lx.MODE_FULL, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lx.DEVERR_CTX


def test_same_cache_through_views_and_layers(lx, orc):
    """Attention of layer l through the whole-pool descriptor equals attention of
    a one-layer view."""
    w = S.Workload("t", 302, L=3, H=2, T=2 * 256, n_outliers_fixed=3)
    cache = _cache(lx, orc, w, 3, 2, 512)
    (kq, _), (vq, _) = cache[S.S_K], cache[S.S_V]
    qb = bf16_dev(w.queries_bf16(1, 4))
    t, c = i32_dev(np.array([[1, 0]])), i32_dev(np.array([450]))
    a = lx.decode_attn(qb, kq, vq, 2, t, c, 0.1, lx.MODE_FULL)
    b = lx.decode_attn(qb, kq.layers(2, 3), vq.layers(2, 3), 0, t, c, 0.1, lx.MODE_FULL)
    assert torch.equal(a, b)


@pytest.mark.parametrize("G", [2, 12, 24, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_group_sizes(lx, orc, G, mode):
    """Groups other than 8 and 16: padded tensor-core rows (2, 12) and the
    CUDA-core kernel for groups above 16 (24, 32)."""
    w = S.Workload("t", 310 + G, L=1, H=2, T=5 * 256, n_outliers_fixed=3, factor_log10=(1, 2))
    cache = _cache(lx, orc, w, 1, 2, 5 * 256)
    qb = w.queries_bf16(2, 2 * G)
    table = np.array([[4, 0, 2, 1, 3], [1, 2, 3, 4, 0]], np.int32)
    ctx = np.array([1100, 77], np.int32)
    out, ref, _, e, E = _run(lx, orc, cache, qb, 0, table, ctx, mode)
    _check(out, ref, E)
    assert e == 0
