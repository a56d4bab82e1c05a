"""Parity at the full worked-example shape (94 layers x 4 KV heads x 128K tokens,
~23.5 GiB of bf16 K+V) in the launch configuration the benchmark times: the
whole cache is encoded on the GPU, and sampled pages, sampled dense rows and two
whole layers of decode attention are recomputed by the oracle from the host
copy of the seeded generator."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_dequant_close, assert_attn_close, assert_planes_equal, attn_sensitivity, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu

W = S.WORKLOADS[3]


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


@pytest.fixture(scope="module")
def full_cache(lx):
    gen = S.DeviceGenerator()
    x = torch.empty((W.L, W.H, W.T, 128), dtype=torch.bfloat16, device="cuda")
    out = {}
    for s in (S.S_K, S.S_V):
        sc = W.scales(s)
        gen.fill(x, W.key(s), sc)
        q = lx.QuantizedKV.empty(W.L, W.H, W.T)
        lx.quantize_pages(x, q)
        rng = np.random.default_rng(100 + s)
        samples = [(int(rng.integers(W.L)), int(rng.integers(W.H)), int(rng.integers(W.pages))) for _ in range(16)]
        samples += [(0, 0, 0), (W.L - 1, W.H - 1, W.pages - 1)]
        inputs = {}
        for (l, h, p) in samples:
            inputs[(l, h, p)] = x[l, h, p * 256:(p + 1) * 256].view(torch.int16).cpu().numpy().view(np.uint16)
        out[s] = (q, sc, samples, inputs)
    del x
    torch.cuda.empty_cache()
    return out


def test_device_input_equals_host_generator(full_cache):
    for s, (q, sc, samples, inputs) in full_cache.items():
        for (l, h, p) in samples:
            host = S.laplace_bf16(W.key(s), sc, W.L, W.H, W.T, layers=[l], heads=[h], t0=p * 256, t1=p * 256 + 256)
            assert np.array_equal(inputs[(l, h, p)], host[0, 0]), (s, l, h, p)


def test_sampled_pages_bit_exact(lx, orc, full_cache):
    for s, (q, sc, samples, _) in full_cache.items():
        for (l, h, p) in samples:
            xb = S.laplace_bf16(W.key(s), sc, W.L, W.H, W.T, layers=[l], heads=[h], t0=p * 256, t1=p * 256 + 256)
            ref = orc.quantize(xb)
            got = dict(anchor=q.anchor[l, h, p * 256:(p + 1) * 256].cpu().numpy()[None, None],
                       residual=q.residual[l, h, p * 256:(p + 1) * 256].cpu().numpy()[None, None],
                       page_meta=q.page_meta[l, h, p:p + 1].cpu().numpy()[None, None],
                       chunk_meta=q.chunk_meta[l, h, p:p + 1].cpu().numpy().view(np.uint16)[None, None])
            assert_planes_equal(got, ref, f"tensor {s} page {(l, h, p)}: ")


def test_sampled_dense_rows(lx, orc, full_cache):
    """Anchor dequant and refine over the whole cache; sampled pages vs the oracle."""
    q, sc, samples, _ = full_cache[S.S_V]
    dense = torch.empty((W.L, W.H, W.T, 128), dtype=torch.bfloat16, device="cuda")
    lx.dequant_anchor(q, dense)
    anchor_pages = {k: dense[k[0], k[1], k[2] * 256:(k[2] + 1) * 256].clone() for k in samples[:6]}
    lx.refine_residual(q, dense)
    for (l, h, p) in samples[:6]:
        xb = S.laplace_bf16(W.key(S.S_V), sc, W.L, W.H, W.T, layers=[l], heads=[h], t0=p * 256, t1=p * 256 + 256)
        ref = orc.quantize(xb)
        rng = np.repeat(ref["page_meta"][..., 1, :], 256, axis=2)
        for t, full in ((anchor_pages[(l, h, p)], False), (dense[l, h, p * 256:(p + 1) * 256], True)):
            got = (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert_dequant_close(got[None, None], orc.dequant(ref, full), rng, True)
    del dense
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layer", [0, 57])
def test_decode_attention_whole_layer(lx, orc, full_cache, layer):
    """B = 1, 64 query heads (group 16), all 128K tokens of one layer."""
    (kq, ksc, _, _), (vq, vsc, _, _) = full_cache[S.S_K], full_cache[S.S_V]
    kx = S.laplace_bf16(W.key(S.S_K), ksc, W.L, W.H, W.T, layers=[layer])
    vx = S.laplace_bf16(W.key(S.S_V), vsc, W.L, W.H, W.T, layers=[layer])
    kr, vr = orc.quantize(kx), orc.quantize(vx)
    qb = W.queries_bf16()
    table = np.arange(W.pages, dtype=np.int32)[None, :]
    ctx = np.array([W.T], np.int32)
    for mode in (0, 1):
        out = lx.decode_attn(bf16_dev(qb), kq, vq, layer, i32_dev(table), i32_dev(ctx), 128 ** -0.5, mode)
        ref = orc.decode_attn(qb, kr, vr, 0, table, ctx, 128 ** -0.5, mode == 1)
        E = attn_sensitivity(orc, qb, kr, vr, 0, table, ctx, 128 ** -0.5, mode == 1)
        assert_attn_close(out.cpu().numpy(), ref, E, f"layer {layer} mode {mode}")
