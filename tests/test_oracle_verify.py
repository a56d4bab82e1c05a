"""Pins of the fp64 verify-attention oracle (a block of draft positions per
request, causal within the block; the Lynx reading, section 4, verifies drafted
positions against the refined cache).

The oracle takes position i of request b as one decode step over the first
ctx_b - T_q + i + 1 tokens. Pinned here against a different formulation: one
numpy masked softmax per (request, head) over the oracle's dense
reconstruction, with the causal mask written as a T_q x ctx matrix, through a
permuted page table; plus the special cases T_q = 1 (plain decode) and
positions that see nothing (zeros)."""
import numpy as np
import pytest

import lynx_synth as S

PAGE, D = 256, 128


def _setup(orc, seed=31, L=2, H=2, T=1024):
    w = S.Workload("v", seed, L=L, H=H, T=T, n_outliers_fixed=4, factor_log10=(1.0, 2.0))
    k = orc.quantize(S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), L, H, T))
    v = orc.quantize(S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), L, H, T))
    return w, k, v


def _masked_numpy(q, Kd, Vd, layer, table, ctx, sm, G):
    B, Tq, Hq, _ = q.shape
    out = np.zeros((B, Tq, Hq, D))
    for b in range(B):
        n = int(ctx[b])
        rows = np.concatenate([np.arange(p * PAGE, p * PAGE + PAGE) for p in table[b]])[:n]
        pos = np.arange(Tq)[:, None]
        tok = np.arange(n)[None, :]
        mask = tok <= n - Tq + pos                  # [Tq, n]: draft position i sees draft tokens <= i
        for h in range(Hq):
            K = Kd[layer, h // G, rows]
            V = Vd[layer, h // G, rows]
            s = np.where(mask, sm * (q[b, :, h] @ K.T), -np.inf)
            m = s.max(1, keepdims=True)
            seen = np.isfinite(m[:, 0])
            p = np.where(seen[:, None], np.exp(s - np.where(seen[:, None], m, 0.0)), 0.0)
            den = p.sum(1, keepdims=True)
            out[b, :, h] = np.where(seen[:, None], (p / np.where(den > 0, den, 1.0)) @ V, 0.0)
    return out


@pytest.mark.parametrize("full", [False, True])
def test_matches_a_masked_softmax_through_permuted_pages(orc, full):
    w, k, v = _setup(orc)
    B, Tq, Hq, G = 2, 9, 4, 2
    table = np.array([[3, 0, 2, 1], [1, 3, 0, 2]], np.int32)
    ctx = np.array([1000, 517], np.int32)
    qb = S.laplace_bf16(w.key(S.S_Q), np.ones((1, B * Tq * Hq, D), np.float32), 1, B * Tq * Hq, 1)
    qb = qb.reshape(B, Tq, Hq, D)
    got = orc.verify_attn(qb, k, v, 1, table, ctx, 128 ** -0.5, full)
    q = (qb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = _masked_numpy(q, orc.dequant(k, full), orc.dequant(v, full), 1, table, ctx, 128 ** -0.5, G)
    assert np.allclose(got, want, rtol=1e-10, atol=1e-10)


def test_one_position_is_a_decode_step(orc):
    w, k, v = _setup(orc, seed=32)
    qb = S.laplace_bf16(w.key(S.S_Q), np.ones((1, 8, D), np.float32), 1, 8, 1).reshape(2, 1, 4, D)
    table = np.array([[0, 1, 2, 3], [2, 3, 0, 1]], np.int32)
    ctx = np.array([700, 1024], np.int32)
    got = orc.verify_attn(qb, k, v, 0, table, ctx, 0.1, True)
    want = orc.decode_attn(qb[:, 0], k, v, 0, table, ctx, 0.1, True)
    assert np.array_equal(got[:, 0], want)


def test_positions_that_see_nothing_are_zero(orc):
    w, k, v = _setup(orc, seed=33)
    qb = S.laplace_bf16(w.key(S.S_Q), np.ones((1, 12, D), np.float32), 1, 12, 1).reshape(1, 6, 2, D)
    got = orc.verify_attn(qb, k, v, 0, np.array([[1, 0, 2, 3]], np.int32), np.array([3], np.int32), 0.1, False)
    assert np.all(got[0, :3] == 0.0) and np.all(np.abs(got[0, 3:]).sum(-1) > 0)
