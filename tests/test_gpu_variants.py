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
