"""Pins of the fp64 decode-attention oracle.

Decode attention over the reconstructed cache is the textbook
softmax(sm_scale * q K^T) V ("KV-cache quantization" explainer, aicassindra,
"Middle row": the stored keys and values are expanded back to real numbers as
they are read, then go through Q.K^T, the softmax and the weighted sum over V). Pins: numpy's matmul/softmax over the
oracle's own dense reconstruction (through a permuted page table), single-token
and uniform-score special cases, the anchor/full identity when every residual is
centred, GQA head grouping, empty contexts and the scores output.
"""
import numpy as np
import pytest

import lynx_synth as S

PAGE, D = 256, 128


def _cache(seed, L, H, T, n_out=4):
    w = S.Workload("t", seed, L=L, H=H, T=T, n_outliers_fixed=n_out, factor_log10=(1.0, 2.0))
    xk = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), L, H, T)
    xv = S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), L, H, T)
    return w, xk, xv


def _numpy_attention(q, Kd, Vd, layer, table, ctx, sm, G):
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(ctx[b])
        if n == 0:
            continue
        rows = np.concatenate([np.arange(p * PAGE, p * PAGE + PAGE) for p in table[b]])[:n]
        for h in range(Hq):
            g = h // G
            K = Kd[layer, g, rows]
            V = Vd[layer, g, rows]
            s = sm * (K @ q[b, h])
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ V
    return out


@pytest.mark.parametrize("full", [False, True])
def test_matches_numpy_softmax_through_permuted_pages(orc, full):
    L, H, T, B, Hq = 2, 2, 6 * PAGE, 3, 8
    w, xk, xv = _cache(5, L, H, T)
    k, v = orc.quantize(xk), orc.quantize(xv)
    table = np.array([[4, 1, 0], [2, 5, 3], [3, 0, 5]], np.int32)
    ctx = np.array([700, 1, 768], np.int32)
    q = w.queries_bf16(B, Hq)
    sm = 1 / np.sqrt(D)
    got = orc.decode_attn(q, k, v, 1, table, ctx, sm, full)
    Kd, Vd = orc.dequant(k, full), orc.dequant(v, full)
    want = _numpy_attention(S.bf16_bits_to_f32(q).astype(np.float64), Kd, Vd, 1, table, ctx, sm, Hq // H)
    assert np.allclose(got, want, rtol=1e-10, atol=1e-9)


def test_single_token_returns_its_value_row(orc):
    w, xk, xv = _cache(6, 1, 1, PAGE)
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = w.queries_bf16(1, 4)
    out = orc.decode_attn(q, k, v, 0, np.array([[0]], np.int32), np.array([1], np.int32), 0.1, True)
    Vd = orc.dequant(v, True)
    assert np.array_equal(out[0], np.broadcast_to(Vd[0, 0, 0], (4, D)))


def test_zero_query_gives_mean_of_values(orc):
    w, xk, xv = _cache(7, 1, 1, 2 * PAGE)
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = np.zeros((1, 2, D), np.uint16)
    out = orc.decode_attn(q, k, v, 0, np.array([[1, 0]], np.int32), np.array([300], np.int32), 1.0, False)
    Vd = orc.dequant(v, False)[0, 0]
    rows = np.concatenate([np.arange(PAGE, 2 * PAGE), np.arange(0, 44)])
    assert np.allclose(out[0, 0], Vd[rows].mean(0), rtol=1e-12, atol=1e-12)


def test_anchor_equals_full_when_residuals_are_centred(orc):
    w, xk, xv = _cache(8, 1, 2, 2 * PAGE)
    k, v = orc.quantize(xk), orc.quantize(xv)
    for t in (k, v):
        t["residual"][:] = 0x77
    q = w.queries_bf16(2, 4)
    tab = np.array([[0, 1], [1, 0]], np.int32)
    ctx = np.array([512, 257], np.int32)
    a = orc.decode_attn(q, k, v, 0, tab, ctx, 0.09, False)
    f = orc.decode_attn(q, k, v, 0, tab, ctx, 0.09, True)
    assert np.array_equal(a, f)


def test_gqa_groups_are_contiguous(orc):
    """Query head h reads KV head h // G: give each KV head its own constant V."""
    w, xk, xv = _cache(9, 1, 4, PAGE)
    for g in range(4):
        xv[0, g] = S.f32_to_bf16_bits(np.full((PAGE, D), float(g + 1), np.float32))
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = w.queries_bf16(1, 16)
    out = orc.decode_attn(q, k, v, 0, np.array([[0]], np.int32), np.array([200], np.int32), 0.1, True)
    for h in range(16):
        assert np.allclose(out[0, h], h // 4 + 1, rtol=1e-13, atol=0)


def test_empty_context_and_scores(orc):
    w, xk, xv = _cache(10, 1, 1, 2 * PAGE)
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = w.queries_bf16(2, 2)
    tab = np.array([[1, 0], [0, 1]], np.int32)
    ctx = np.array([0, 300], np.int32)
    out, sc = orc.decode_attn(q, k, v, 0, tab, ctx, 0.5, True, want_scores=True)
    assert np.all(out[0] == 0)
    assert np.all(np.isneginf(sc[0]))
    assert np.all(np.isneginf(sc[1, :, 300:]))
    Kd = orc.dequant(k, True)[0, 0]
    qf = S.bf16_bits_to_f32(q).astype(np.float64)
    assert np.allclose(sc[1, 1, :256], 0.5 * Kd[:256] @ qf[1, 1], rtol=1e-12, atol=1e-12)
    assert np.allclose(sc[1, 1, 256:300], 0.5 * Kd[256:300] @ qf[1, 1], rtol=1e-12, atol=1e-12)


def test_rejects_out_of_range_page_and_length(orc):
    w, xk, xv = _cache(11, 1, 1, PAGE)
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = w.queries_bf16(1, 1)
    with pytest.raises(ValueError):
        orc.decode_attn(q, k, v, 0, np.array([[1]], np.int32), np.array([10], np.int32), 1.0, True)
    with pytest.raises(ValueError):
        orc.decode_attn(q, k, v, 0, np.array([[0]], np.int32), np.array([257], np.int32), 1.0, True)
