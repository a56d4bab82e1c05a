"""GPU parity of the decoders: anchor-only dequant (lynx_dequant_anchor) and the
in-place refinement (lynx_refine_residual), against the oracle's fp64 decode."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_dequant_close, bf16_dev, dense_to_np, i32_dev, rng_per_element

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def _case(lx, seed, L, H, T, valid=None, n_out=4):
    w = S.Workload("t", seed, L=L, H=H, T=T, n_outliers_fixed=n_out, base_log10=(-2, 0),
                   factor_log10=(1, 2))
    xb = S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), L, H, T)
    q = lx.QuantizedKV.empty(L, H, T)
    lx.quantize_pages(bf16_dev(xb), q, None if valid is None else i32_dev(valid))
    return xb, q


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_anchor_then_refine(lx, orc, dtype):
    valid = np.array([256, 256, 77, 0], np.int32)
    xb, q = _case(lx, 200, 2, 3, 1024, valid)
    ref_q = orc.quantize(xb, valid)
    rng = rng_per_element(ref_q)
    dense = torch.empty((2, 3, 1024, 128), dtype=dtype, device="cuda")
    lx.dequant_anchor(q, dense)
    assert_dequant_close(dense_to_np(dense), orc.dequant(ref_q, False), rng, dtype == torch.bfloat16)
    lx.refine_residual(q, dense)
    assert_dequant_close(dense_to_np(dense), orc.dequant(ref_q, True), rng, dtype == torch.bfloat16)


def test_refine_of_anchor_equals_direct_full(lx):
    """refine(dequant_anchor(A)) is bitwise the full reconstruction, whatever the
    buffer held before."""
    xb, q = _case(lx, 201, 1, 4, 2048)
    a = torch.empty((1, 4, 2048, 128), dtype=torch.bfloat16, device="cuda")
    lx.dequant_anchor(q, a)
    lx.refine_residual(q, a)
    b = torch.full((1, 4, 2048, 128), 123.0, dtype=torch.bfloat16, device="cuda")
    lx.refine_residual(q, b)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_anchor_only_needs_no_residual_plane(lx, orc):
    xb, q = _case(lx, 202, 1, 2, 512)
    ref_q = orc.quantize(xb)
    dense = torch.empty((1, 2, 512, 128), dtype=torch.float32, device="cuda")
    lx.dequant_anchor(q.without_residual(), dense)
    assert_dequant_close(dense_to_np(dense), orc.dequant(ref_q, False), rng_per_element(ref_q), False)


def test_layer_view(lx, orc):
    """A descriptor view of one layer decodes that layer only."""
    xb, q = _case(lx, 203, 3, 2, 512)
    ref_q = orc.quantize(xb)
    dense = torch.zeros((1, 2, 512, 128), dtype=torch.float32, device="cuda")
    lx.refine_residual(q.layers(1, 2), dense)
    full = orc.dequant(ref_q, True)
    assert_dequant_close(dense_to_np(dense), full[1:2], rng_per_element(ref_q)[1:2], False)


def test_qwen3_235b_like_layer(lx, orc):
    w = S.WORKLOADS[2]
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), w.L, w.H, w.T)
    q = lx.QuantizedKV.empty(w.L, w.H, w.T)
    lx.quantize_pages(bf16_dev(xb), q)
    ref_q = orc.quantize(xb)
    rng = rng_per_element(ref_q)
    dense = torch.empty((w.L, w.H, w.T, 128), dtype=torch.bfloat16, device="cuda")
    lx.dequant_anchor(q, dense)
    assert_dequant_close(dense_to_np(dense), orc.dequant(ref_q, False), rng, True)
    lx.refine_residual(q, dense)
    assert_dequant_close(dense_to_np(dense), orc.dequant(ref_q, True), rng, True)
