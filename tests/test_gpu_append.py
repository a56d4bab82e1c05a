"""GPU parity of quantize-on-append (lynx_quantize_append): each tail page is
re-encoded into its physical page of every layer and KV head, bit-exact against
the oracle's encoding of that page with its valid-token count; every other page
of the pool is left as it was."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_planes_equal, bf16_dev, i32_dev, planes_np

pytestmark = pytest.mark.gpu

W = S.WORKLOADS[4]


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def _tails(n, L, H, stream):
    """bf16 bits [n, L, H, 256, 128]: tail i of layer l, head h is page i of a
    [L, H, n * 256] Laplace tensor with the batched workload's channel scales."""
    sc = S.channel_scales(W.seed, stream, L, H, n_outliers=W.n_outliers, factor_log10=W.factor_log10)
    x = S.laplace_bf16(W.key(stream), sc, L, H, n * 256)
    return np.ascontiguousarray(x.reshape(L, H, n, 256, 128).transpose(2, 0, 1, 3, 4))


def _page(planes, l, h, p):
    sl = slice(256 * p, 256 * p + 256)
    return dict(anchor=planes["anchor"][l, h, sl][None, None], residual=planes["residual"][l, h, sl][None, None],
                page_meta=planes["page_meta"][l, h, p][None, None, None],
                chunk_meta=planes["chunk_meta"][l, h, p][None, None, None])


def _pool(lx, L, H, P, stream):
    sc = S.channel_scales(W.seed, stream + 7, L, H, n_outliers=W.n_outliers, factor_log10=W.factor_log10)
    x = S.laplace_bf16(W.key(stream + 7), sc, L, H, P * 256)
    q = lx.QuantizedKV.empty(L, H, P * 256)
    lx.quantize_pages(bf16_dev(x), q)
    return q


@pytest.mark.parametrize("stream", [S.S_K, S.S_V])
def test_tails_match_the_oracle_and_nothing_else_moves(lx, orc, stream):
    L, H, P = 2, 3, 16
    valid = np.array([256, 1, 37, 128, 255, 0, 200], np.int32)
    phys = np.array([3, 0, 15, 7, 9, 12, 4], np.int32)
    n = len(phys)
    q = _pool(lx, L, H, P, stream)
    before = planes_np(q)
    tails = _tails(n, L, H, stream)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lx.quantize_append(bf16_dev(tails), i32_dev(phys), i32_dev(valid), q, dev_err=err)
    after = planes_np(q)
    assert int(err.item()) == 0
    for i in range(n):
        for l in range(L):
            for h in range(H):
                ref = orc.quantize(tails[i, l, h][None, None], np.array([valid[i]], np.int32))
                assert_planes_equal(_page(after, l, h, phys[i]), ref, f"tail {i} layer {l} head {h}: ")
    untouched = sorted(set(range(P)) - set(phys.tolist()))
    for l in range(L):
        for h in range(H):
            for p in untouched:
                assert_planes_equal(_page(after, l, h, p), _page(before, l, h, p), f"page {p}: ")


def test_out_of_pool_pages_are_skipped_and_flagged(lx, orc):
    L, H, P = 1, 2, 4
    q = _pool(lx, L, H, P, S.S_K)
    before = planes_np(q)
    tails = _tails(3, L, H, S.S_K)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lx.quantize_append(bf16_dev(tails), i32_dev([-1, 2, 4]), i32_dev([256, 100, 256]), q, dev_err=err)
    assert int(err.item()) & 1
    after = planes_np(q)
    for h in range(H):
        ref = orc.quantize(tails[1, 0, h][None, None], np.array([100], np.int32))
        assert_planes_equal(_page(after, 0, h, 2), ref)
        for p in (0, 1, 3):
            assert_planes_equal(_page(after, 0, h, p), _page(before, 0, h, p))


def test_empty_pool_flags_every_tail(lx):
    """A pool of 0 pages (tokens = 0, through the raw ABI, whose pointers must
    only be non-NULL and aligned): every tail is outside it, so the call
    succeeds, writes nothing and sets the page bit."""
    import ctypes
    tails = bf16_dev(_tails(2, 1, 2, S.S_K))
    scratch = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    base = scratch.data_ptr()
    d = lx.LynxQKV(1, 2, 0, 128, base, base + 256, base + 512, base + 768)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    phys, valid = i32_dev([0, 3]), i32_dev([256, 7])
    st = lx.library().lynx_quantize_append(ctypes.c_void_p(tails.data_ptr()), ctypes.c_void_p(phys.data_ptr()),
                                            ctypes.c_void_p(valid.data_ptr()), 2, ctypes.byref(d),
                                            ctypes.c_void_p(err.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == lx.OK
    assert int(err.item()) == 1
    assert int(scratch.count_nonzero().item()) == 0


def test_batched_decode_tails_full_size(lx, orc):
    """The batched-decode workload's growing last pages (32 requests, ragged
    contexts, seeded physical pages) over 8 layers x 8 KV heads; sampled pages
    checked against the oracle."""
    ctx, pool, table = S.batched_layout(W)
    L, H, n = 8, W.H, W.B
    last = (ctx - 1) // 256
    phys = table[np.arange(n), last].astype(np.int32)
    valid = (ctx - 256 * last).astype(np.int32)
    q = lx.QuantizedKV.empty(L, H, pool * 256)
    tails = _tails(n, L, H, S.S_V)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lx.quantize_append(bf16_dev(tails), i32_dev(phys), i32_dev(valid), q, dev_err=err)
    assert int(err.item()) == 0
    got = planes_np(q)
    rng = np.random.default_rng(11)
    for _ in range(24):
        i, l, h = int(rng.integers(n)), int(rng.integers(L)), int(rng.integers(H))
        ref = orc.quantize(tails[i, l, h][None, None], np.array([valid[i]], np.int32))
        assert_planes_equal(_page(got, l, h, phys[i]), ref, f"tail {i} layer {l} head {h}: ")
