"""GPU parity of the multi-token verify attention (lynx_verify_attn) against the
oracle's fp64 verify attention, anchor-only and full, within the attention
tolerance of the decode path (2e-3 plus the first-order fp32 score bound),
per draft position."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_attn_close, attn_sensitivity, attn_tolerance, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def _cache(lx, orc, w, L, H, T):
    out = {}
    for s in (S.S_K, S.S_V):
        xb = S.laplace_bf16(w.key(s), w.scales(s)[:L, :H], L, H, T)
        q = lx.QuantizedKV.empty(L, H, T)
        lx.quantize_pages(bf16_dev(xb), q)
        out[s] = (q, orc.quantize(xb))
    return out


def _queries(w, B, Tq, Hq):
    qb = S.laplace_bf16(S.key(w.seed, S.S_Q * 1000 + 7), np.ones((1, B * Tq * Hq, 128), np.float32), 1,
                        B * Tq * Hq, 1)
    return qb.reshape(B, Tq, Hq, 128)


def _check(lx, orc, cache, qb, layer, table, ctx, mode, positions=None):
    (kq, kr), (vq, vr) = cache[S.S_K], cache[S.S_V]
    B, Tq, Hq, _ = qb.shape
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lx.verify_attn(bf16_dev(qb), kq, vq, layer, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode,
                         dev_err=err).cpu().numpy()
    full = mode == lx.MODE_FULL
    ref = orc.verify_attn(qb, kr, vr, layer, table, ctx, 128 ** -0.5, full)
    assert int(err.item()) == 0
    for i in (range(Tq) if positions is None else positions):
        n = np.maximum(np.asarray(ctx) - Tq + i + 1, 0)
        E = attn_sensitivity(orc, qb[:, i], kr, vr, layer, table, n, 128 ** -0.5, full)
        assert_attn_close(out[:, i], ref[:, i], E, f"verify position {i} mode {mode}")
    return out


@pytest.mark.parametrize("mode", [0, 1])
def test_one_page(lx, orc, mode):
    w = S.WORKLOADS[1]
    cache = _cache(lx, orc, w, 1, 1, 256)
    _check(lx, orc, cache, _queries(w, 1, 8, 1), 0, np.zeros((1, 1), np.int32), np.array([256]), mode)


@pytest.mark.parametrize("mode", [0, 1])
def test_group_16_block_of_64(lx, orc, mode):
    """Qwen3-235B-like heads (4 KV heads, 64 query heads): 64 draft positions x 16
    heads = 1024 query rows per KV head, eight row blocks."""
    w = S.WORKLOADS[2]
    T = 8192
    cache = _cache(lx, orc, w, 1, 4, T)
    table = np.arange(T // 256, dtype=np.int32)[None]
    _check(lx, orc, cache, _queries(w, 1, 64, 64), 0, table, np.array([T - 37]), mode,
           positions=[0, 1, 17, 40, 62, 63])


@pytest.mark.parametrize("mode", [0, 1])
def test_report_shape_sampled_positions(lx, orc, mode):
    """The verify report's workload and launch configuration: 4 KV heads x 32K
    tokens, 64 query heads, 64 draft positions (eight row blocks x four page
    ranges of 32 pages). Sampled positions are checked against the oracle's
    decode step over each one's visible prefix, which is what the oracle's
    verify attention computes position by position."""
    w = S.WORKLOADS[2]
    cache = _cache(lx, orc, w, 1, w.H, w.T)
    (kq, kr), (vq, vr) = cache[S.S_K], cache[S.S_V]
    Tq, Hq = 64, 64
    qb = _queries(w, 1, Tq, Hq)
    table = np.arange(w.pages, dtype=np.int32)[None]
    ctx = np.array([w.T])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lx.verify_attn(bf16_dev(qb), kq, vq, 0, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode,
                         dev_err=err).cpu().numpy()
    assert int(err.item()) == 0
    full = mode == lx.MODE_FULL
    for i in (0, 21, 63):
        n = ctx - Tq + i + 1
        ref = orc.decode_attn(qb[:, i], kr, vr, 0, table, n, 128 ** -0.5, full)
        E = attn_sensitivity(orc, qb[:, i], kr, vr, 0, table, n, 128 ** -0.5, full)
        assert_attn_close(out[:, i], ref, E, f"verify 32K position {i} mode {mode}")


@pytest.mark.parametrize("mode", [0, 1])
def test_batched_ragged_permuted(lx, orc, mode):
    """The batched-decode layout (ragged contexts, permuted pages, 8 KV heads x
    8 query heads each) for 6 of its requests, 16 draft positions."""
    w = S.WORKLOADS[4]
    ctx, pool, table = S.batched_layout(w)
    pick = [0, 5, 11, 17, 23, 31]
    ctx, table = ctx[pick], table[pick]
    cache = _cache(lx, orc, w, 1, 8, pool * 256)
    _check(lx, orc, cache, _queries(w, len(pick), 16, 64), 0, table, ctx, mode, positions=[0, 7, 15])


def test_positions_before_the_context_are_zero_and_bad_pages_flagged(lx, orc):
    w = S.WORKLOADS[1]
    cache = _cache(lx, orc, w, 1, 1, 512)
    (kq, _), (vq, _) = cache[S.S_K], cache[S.S_V]
    qb = _queries(w, 2, 6, 1)
    table = np.array([[0, 1], [1, 7]], np.int32)                 # page 7 is outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lx.verify_attn(bf16_dev(qb), kq, vq, 0, i32_dev(table), i32_dev([3, 400]), 128 ** -0.5, lx.MODE_FULL,
                         dev_err=err).cpu().numpy()
    assert np.all(out[0, :3] == 0.0) and np.all(np.abs(out[0, 3:]).sum(-1) > 0)
    assert int(err.item()) & 1


@pytest.mark.parametrize("mode", [0, 1])
def test_single_position_equals_decode_attention(lx, orc, mode):
    """A block of one draft position is one decode step: the verify kernel
    (tensor-memory accumulators, decoded tiles) and the decode kernel
    (register-direct level operands) must agree, each within its bound of the
    oracle, so within twice the bound of each other."""
    w = S.WORKLOADS[4]
    ctx, pool, table = S.batched_layout(w)
    pick = [1, 8, 30]
    ctx, table = ctx[pick], table[pick]
    cache = _cache(lx, orc, w, 1, 8, pool * 256)
    (kq, kr), (vq, vr) = cache[S.S_K], cache[S.S_V]
    qb = _queries(w, len(pick), 1, 64)
    full = mode == lx.MODE_FULL
    ov = lx.verify_attn(bf16_dev(qb), kq, vq, 0, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode).cpu().numpy()[:, 0]
    od = lx.decode_attn(bf16_dev(qb[:, 0]), kq, vq, 0, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode).cpu().numpy()
    E = attn_sensitivity(orc, qb[:, 0], kr, vr, 0, table, np.asarray(ctx), 128 ** -0.5, full)
    ref = orc.decode_attn(qb[:, 0], kr, vr, 0, table, np.asarray(ctx), 128 ** -0.5, full)
    assert_attn_close(ov, ref, E, f"verify one position mode {mode}")
    assert_attn_close(od, ref, E, f"decode one position mode {mode}")
    tol = attn_tolerance(orc, qb[:, 0], kr, vr, 0, table, np.asarray(ctx), 128 ** -0.5, full)
    assert np.all(np.abs(ov - od) <= 2 * tol)


@pytest.mark.parametrize("mode", [0, 1])
def test_odd_group_and_block(lx, orc, mode):
    """G = 5 (20 query heads over 4 KV heads) and a block of 37 positions: row
    blocks, head mapping and causal masks off every power-of-two boundary."""
    w = S.WORKLOADS[2]
    T = 2048
    cache = _cache(lx, orc, w, 1, 4, T)
    table = np.arange(T // 256, dtype=np.int32)[None]
    _check(lx, orc, cache, _queries(w, 1, 37, 20), 0, table, np.array([T - 300]), mode,
           positions=[0, 1, 18, 35, 36])
