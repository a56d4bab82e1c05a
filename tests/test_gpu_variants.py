"""GPU parity of the quantizer variants (lynx_quantize_variant) against the
variant oracle: codes, anchor and residual planes and metadata bit for bit,
per-page squared errors within fp32 rounding (the kernel evaluates the
reconstructions in fp32, the oracle in fp64). The default variant also
reproduces lynx_quantize_pages' planes."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import bf16_dev

pytestmark = pytest.mark.gpu

CASES = [
    dict(),
    dict(chunk=16), dict(chunk=64),
    dict(alpha=15.0), dict(alpha=1023.0), dict(alpha=0.0),
    dict(anchor_bits=2, residual_bits=4), dict(anchor_bits=6, residual_bits=2), dict(anchor_bits=3, residual_bits=3),
    dict(flags=1), dict(flags=2), dict(flags=4), dict(flags=8), dict(flags=15),
    dict(anchor_bits=2, residual_bits=2),
    dict(uniform_bits=4), dict(uniform_bits=8), dict(uniform_bits=4, flags=16), dict(uniform_bits=8, flags=16),
]
_KEYS = {"chunk": "chunk", "anchor_bits": "anchor_bits", "residual_bits": "residual_bits", "alpha": "alpha",
         "uniform_bits": "uniform_bits"}


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


@pytest.fixture(scope="module")
def xb():
    w = S.WORKLOADS[2]
    x = S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V)[:1, :2], 1, 2, 1024)
    return x.reshape(2, 1024, 128)


def _variant(case):
    from oracle import variants as V
    f = case.get("flags", 0)
    kw = {k: case[k] for k in _KEYS if k in case}
    return V.Variant(page_norm=not f & 1, chunk_isolation=not f & 2, bias=not f & 4, sign_aware=not f & 8,
                     uniform_per_token=bool(f & 16), **kw)


def _compare(o, g, case, pages=None):
    """o: the oracle's encoding of the pages compared; g: the GPU outputs, of
    which `pages` (all when None) are those pages."""
    sel = slice(None) if pages is None else list(pages)
    tok = slice(None) if pages is None else np.concatenate([np.arange(256 * p, 256 * p + 256) for p in pages])
    assert np.array_equal(g["page_meta"].cpu().numpy()[:, sel].view(np.uint32),
                          o["page_meta"].astype(np.float32).view(np.uint32))
    assert np.array_equal(g["codes"].cpu().numpy().astype(np.int32)[:, tok], o["codes"])
    if not case.get("uniform_bits"):
        ga = g["anchor"].cpu().numpy().astype(np.int32)[:, tok]
        gr = g["residual"].cpu().numpy().astype(np.int32)[:, tok]
        assert np.array_equal(ga, o["anchor"]) and np.array_equal(gr, o["residual"])
        assert np.array_equal(g["chunk_meta"].cpu().numpy().view(np.uint16)[:, sel], o["chunk_meta"])
    ge = g["err"].cpu().numpy()[:, sel]
    assert np.allclose(ge[..., 0], o["err"][..., 0], rtol=1e-4)
    assert np.allclose(ge[..., 1:], o["err"][..., 1:], rtol=2e-3, atol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()) or "default")
def test_variant_matches_oracle(lx, xb, case):
    from oracle import variants as V
    g = lx.quantize_variant(bf16_dev(xb), codes=True, planes=True, meta=True, **case)
    o = V.encode(xb, _variant(case))
    _compare(o, g, case)


def test_default_variant_is_the_production_encoder(lx, xb):
    g = lx.quantize_variant(bf16_dev(xb), planes=True, meta=True)
    q = lx.QuantizedKV.empty(1, 2, 1024)
    lx.quantize_pages(bf16_dev(xb).view(1, 2, 1024, 128), q)
    a = q.anchor.cpu().numpy().reshape(2, 1024, 64)
    r = q.residual.cpu().numpy().reshape(2, 1024, 64)
    ga = g["anchor"].cpu().numpy().astype(np.int32) & 15
    gr = g["residual"].cpu().numpy().astype(np.int32)
    assert np.array_equal(ga[..., 0::2] | (ga[..., 1::2] << 4), a.astype(np.int32))
    assert np.array_equal(gr[..., 0::2] | (gr[..., 1::2] << 4), r.astype(np.int32))
    assert torch.equal(g["page_meta"].view(torch.int32).reshape(-1), q.page_meta.view(torch.int32).reshape(-1))
    assert torch.equal(g["chunk_meta"].reshape(-1), q.chunk_meta.view(torch.int16).reshape(-1))


@pytest.mark.parametrize("case", [dict(), dict(chunk=16), dict(uniform_bits=4)], ids=["default", "C16", "int4"])
def test_report_size_sampled_pages(lx, case):
    """The ablation report's launch (K of the 4-head, 32K-token layer, 512
    pages) against the oracle on sampled pages."""
    from oracle import variants as V
    w = S.WORKLOADS[2]
    gen = S.DeviceGenerator()
    x = torch.empty((1, w.H, w.T, 128), dtype=torch.bfloat16, device="cuda")
    gen.fill(x, w.key(S.S_K), w.scales(S.S_K))
    g = lx.quantize_variant(x, codes=True, planes=True, meta=True, **case)
    xs = x.view(w.H, w.T, 128)
    pages = [0, 37, w.T // 256 - 1]
    sub = torch.cat([xs[:, 256 * p:256 * p + 256] for p in pages], dim=1).contiguous()
    o = V.encode(sub.view(torch.int16).cpu().numpy().view(np.uint16), _variant(case))
    _compare(o, g, case, pages=pages)


@pytest.mark.parametrize("case", [dict(), dict(chunk=16, flags=1), dict(flags=2), dict(uniform_bits=4),
                                  dict(uniform_bits=8, flags=16)],
                         ids=["default", "C16-nopagenorm", "noiso", "int4", "int8-token"])
def test_edge_pages(lx, case):
    """Degenerate pages: a constant channel (range 0), a channel with a NaN, an
    all-zero page, a channel whose chunk holds one outlier, +/-0 mixtures, and
    large magnitudes. Codes and metadata bit for bit; error sums where finite."""
    from oracle import variants as V
    rng = np.random.default_rng(11)
    x = rng.laplace(size=(2, 768, 128)).astype(np.float32)
    x[0, :256, 3] = 1.5                              # constant channel
    x[0, 17, 5] = np.nan                             # NaN channel (page 0)
    x[1, 256:512, :] = 0.0                           # all-zero page
    x[1, 300, 9] = -0.0
    x[0, 600, 7] = 3.0e4                             # one outlier in a chunk
    x[1, 512:, 11] *= 1.0e3                          # large magnitudes
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation to bf16 is fine for a test input
    g = lx.quantize_variant(bf16_dev(xb), codes=True, planes=True, meta=True, **case)
    o = V.encode(xb, _variant(case))
    assert np.array_equal(g["codes"].cpu().numpy().astype(np.int32), o["codes"])
    pm_g, pm_o = g["page_meta"].cpu().numpy(), o["page_meta"].astype(np.float32)
    assert np.array_equal(np.isnan(pm_g), np.isnan(pm_o))
    assert np.array_equal(np.nan_to_num(pm_g).view(np.uint32), np.nan_to_num(pm_o).view(np.uint32))
    if not case.get("uniform_bits"):
        assert np.array_equal(g["anchor"].cpu().numpy().astype(np.int32), o["anchor"])
        assert np.array_equal(g["residual"].cpu().numpy().astype(np.int32), o["residual"])
        cg = g["chunk_meta"].cpu().numpy().view(np.uint16)
        hg, ho = cg.view(np.float16), o["chunk_meta"].view(np.float16)
        nan = np.isnan(hg)                            # NaN payloads may differ: any NaN matches any NaN
        assert np.array_equal(nan, np.isnan(ho)) and np.array_equal(cg[~nan], o["chunk_meta"][~nan])
    ge, oe = g["err"].cpu().numpy(), o["err"]
    fin = np.isfinite(oe).all(axis=-1)
    assert np.array_equal(np.isfinite(ge).all(axis=-1), fin)
    assert np.allclose(ge[fin][:, 0], oe[fin][:, 0], rtol=1e-4)
    assert np.allclose(ge[fin][:, 1:], oe[fin][:, 1:], rtol=2e-3, atol=1e-9)


def _recon_bound(o, xb, case):
    """Per-element bound on |fp32 reconstruction - fp64 oracle reconstruction|:
    the kernel forms mn + rng mu and rng s sgn(c) in fp32, then one fused
    multiply-add with the level (each step within half an ulp), the
    comparator one fused multiply-add of the code with the fp32 step."""
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    N, T, D = x.shape
    if case.get("uniform_bits"):
        if case.get("flags", 0) & 16:
            mn, rng = x.min(axis=-1, keepdims=True), x.max(axis=-1, keepdims=True) - x.min(axis=-1, keepdims=True)
        else:
            pm = np.repeat(o["page_meta"].astype(np.float64), 256, axis=1).reshape(N, T, 2, D)
            mn, rng = pm[:, :, 0], pm[:, :, 1]
        m = np.abs(mn) + np.abs(rng)
    else:
        C = case.get("chunk", 32)
        pm = np.repeat(o["page_meta"].astype(np.float64), 256, axis=1).reshape(N, T, 2, D)
        cm = np.repeat(o["chunk_meta"].view(np.float16).astype(np.float64), C, axis=2).reshape(N, T, 2, D)
        m = np.abs(pm[:, :, 0]) + np.abs(pm[:, :, 1]) * (np.abs(cm[:, :, 0]) + np.abs(cm[:, :, 1]))
    return 2.0 ** -21 * m


@pytest.mark.parametrize("case", [dict(), dict(chunk=16), dict(anchor_bits=2, residual_bits=2), dict(flags=15),
                                  dict(alpha=0.0), dict(uniform_bits=4), dict(uniform_bits=8, flags=16)],
                         ids=["default", "C16", "2+2", "flags15", "linear", "int4", "int8-token"])
def test_reconstructions_match_oracle(lx, xb, case):
    """The optional fp32 reconstructions (anchor-only and full) against the
    oracle's fp64 ones, within the rounding of the kernel's fp32 decode."""
    from oracle import variants as V
    g = lx.quantize_variant(bf16_dev(xb), recon=True, meta=True, **case)
    o = V.encode(xb, _variant(case))
    bound = _recon_bound(o, xb, case)
    for key in ("x_anchor", "x_full"):
        d = np.abs(g[key].cpu().numpy().astype(np.float64) - o[key])
        assert np.all(d <= bound), (key, float((d / bound).max()))
    # the error sums are those of the stored reconstructions
    x = torch.from_numpy((xb.astype(np.uint32) << 16).view(np.float32)).cuda().double()
    ge = g["err"].sum(dim=1)
    for j, key in ((1, "x_anchor"), (2, "x_full")):
        e = ((g[key].double() - x) ** 2).sum(dim=(1, 2))
        assert torch.allclose(ge[:, j], e, rtol=1e-4, atol=1e-30)     # fp32 per-thread sums


def _attn_tol(q, k, v, sm):
    """fp32 bound per (request, head): each score is a 128-term fp32 dot
    product (error within 128 ulp of sum |q_i k_i|); an error d in the scores
    moves the output by at most 2 d max|v|, plus the fp32 sums over tokens."""
    qf = S.bf16_bits_to_f32(q).astype(np.float64)
    G = q.shape[1] // k.shape[0]
    ka = np.abs(k).max(axis=1)                      # [H, 128]
    mag = np.einsum("bhd,hd->bh", np.abs(qf), np.repeat(ka, G, axis=0)) * sm
    vmax = np.abs(v).max()
    return (2 * 128 * 2.0 ** -24 * mag * 2 + 1e-5)[..., None] * vmax


@pytest.mark.parametrize("H,Hq,T,B", [(1, 1, 1, 1), (2, 8, 300, 3), (4, 64, 4113, 2), (1, 2, 49152, 2)],
                         ids=["one-token", "ragged", "gqa16", "max-tokens"])
def test_dense_attention_matches_oracle(lx, H, Hq, T, B):
    from oracle import variants as V
    rng = np.random.default_rng(T)
    k = (rng.laplace(size=(H, T, 128)) * np.where(rng.random(128) < 0.03, 30.0, 1.0)).astype(np.float32)
    v = rng.laplace(size=(H, T, 128)).astype(np.float32)
    q = S.f32_to_bf16_bits(rng.laplace(size=(B, Hq, 128)).astype(np.float32))
    sm = 128 ** -0.5
    got = lx.dense_attn(torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16),
                        torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), sm).cpu().numpy()
    want = V.dense_attn(q, k, v, sm)
    assert np.all(np.abs(got - want) <= _attn_tol(q, k, v, sm))


def test_dense_attention_argument_errors(lx):
    q = torch.zeros((1, 3, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((2, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError):
        lx.dense_attn(q, k, k)                      # 3 query heads over 2 KV heads
    big = torch.zeros((1, 49153, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError):
        lx.dense_attn(q, big, big)
