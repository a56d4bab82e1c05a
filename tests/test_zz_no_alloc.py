"""lynx_decode_attn_noalloc: decode attention for callers that cannot allocate
device memory (for instance a serving engine whose memory pool already holds
all free memory, or a plugin that only receives its input and output buffers).
Its split-K scratch is a fixed array inside the library instead of a
caller-provided workspace.

Checked through the C ABI against lynx_decode_attn on the same inputs, on two
calls in a row (the second must not see anything of the first through the
shared array). Both calls run the same kernels with the same split plan, so
the outputs must be equal bit for bit; each is also checked against the
oracle's fp64 decode attention within the attention tolerance of the parity
tests. Plus the rejection of a batch shape that needs more scratch than the
array holds. This file is named so that pytest collects it last."""
import ctypes

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


def _noalloc(lx, qt, k, v, layer, table, ctx, mode, out):
    kd, vd = k.desc(), v.desc()
    return lx.library().lynx_decode_attn_noalloc(
        ctypes.c_void_p(qt.data_ptr()), ctypes.byref(kd), ctypes.byref(vd), layer,
        ctypes.c_void_p(table.data_ptr()), ctypes.c_void_p(ctx.data_ptr()), qt.shape[0], qt.shape[1],
        table.shape[1], ctypes.c_float(128 ** -0.5), mode, ctypes.c_void_p(out.data_ptr()), None, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lx, orc):
    w = S.Workload("t", 400, L=2, H=4, T=24 * 256, n_outliers_fixed=4, factor_log10=(1, 2))
    caches = {}
    for s in (S.S_K, S.S_V):
        xb = S.laplace_bf16(w.key(s), w.scales(s), w.L, w.H, w.T)
        q = lx.QuantizedKV.empty(w.L, w.H, w.T)
        lx.quantize_pages(bf16_dev(xb), q)
        caches[s] = (q, orc.quantize(xb))
    (kq, kr), (vq, vr) = caches[S.S_K], caches[S.S_V]
    # two different calls: the second has a different batch, layer, mode and lengths
    calls = [
        (w.queries_bf16(1, 64, step=0), 0, np.arange(24, dtype=np.int32)[None, :], np.array([24 * 256]), 0),
        (w.queries_bf16(3, 64, step=1), 1, np.stack([np.roll(np.arange(24, dtype=np.int32), r) for r in (0, 5, 11)]),
         np.array([6000, 1, 256 * 7 + 3]), 1),
    ]
    for qb, layer, table, ctx, mode in calls:
        qt, tt, ct = bf16_dev(qb), i32_dev(table), i32_dev(ctx)
        out = torch.full((qb.shape[0], 64, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(lx, qt, kq, vq, layer, tt, ct, mode, out)
        assert st == lx.OK, lx.library().lynx_status_string(st)
        ref = lx.decode_attn(qt, kq, vq, layer, tt, ct, 128 ** -0.5, mode)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        want = orc.decode_attn(qb, kr, vr, layer, table, ctx, 128 ** -0.5, mode == 1)
        E = attn_sensitivity(orc, qb, kr, vr, layer, table, ctx, 128 ** -0.5, mode == 1)
        assert_attn_close(out.cpu().numpy(), want, E, f"no-alloc layer {layer} mode {mode}")


def test_noalloc_rejects_shapes_beyond_its_scratch(lx):
    B, Hq, maxp = 64, 128, 4096
    need = lx.decode_attn_workspace(B, Hq, maxp)
    assert need > lx.NOALLOC_SCRATCH_BYTES
    w = S.Workload("t", 401, L=1, H=4, T=256, n_outliers_fixed=2)
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, 4, 256)
    q = lx.QuantizedKV.empty(1, 4, 256)
    lx.quantize_pages(bf16_dev(xb), q)
    qt = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, maxp), dtype=torch.int32, device="cuda")
    ctx = torch.full((B,), 256, dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, 128), 7.0, dtype=torch.float32, device="cuda")
    st = _noalloc(lx, qt, q, q, 0, table, ctx, 0, out)
    assert st == lx.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)          # nothing was launched
