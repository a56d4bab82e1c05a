"""Progressive arrival at full size (8 layers x 8 KV heads x 64K tokens, 8
requests sharing the context, 64 query heads): residual layers land in a
seeded order; each arrival refines that layer in place and reruns decode
attention over all layers. Checked against the oracle on sampled layers and
requests, plus the invariants of the procedure."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_attn_close, assert_dequant_close, attn_sensitivity

pytestmark = pytest.mark.gpu

W = S.WORKLOADS[5]


@pytest.fixture(scope="module")
def run():
    import __graft_entry__
    __graft_entry__.build()
    import bench
    import progressive_kv_cache_gb300 as lx
    return lx, bench.progressive_arrival(torch, lx, keep=True)


def test_report_shape_and_invariants(run):
    lx, r = run
    assert sorted(r["order"]) == list(range(W.L))
    for a in r["arrivals"]:
        assert a["pending_layers_unchanged"]
        assert 0.0 <= a["top_agreement_min"] <= a["top_agreement_mean"] <= 1.0
        assert a["delta_max_abs"] > 0 and np.isfinite(a["delta_rel_l2"])
        print(a)
    # after the last arrival every layer is the full reconstruction
    for l in range(W.L):
        direct = lx.decode_attn(torch.from_numpy(r["qb"].view(np.int16)).cuda().view(torch.bfloat16),
                                r["qkv"][S.S_K], r["qkv"][S.S_V], l,
                                torch.arange(W.pages, dtype=torch.int32, device="cuda")[None].repeat(W.B, 1)
                                .contiguous(), torch.full((W.B,), W.T, dtype=torch.int32, device="cuda"),
                                128 ** -0.5, lx.MODE_FULL)
        assert torch.equal(direct, r["outs"][l])


def test_refined_cache_and_attention_against_oracle(run, orc):
    lx, r = run
    order = r["order"]
    for l in (order[0], order[-1]):
        heads = [0, 5]
        kx = S.laplace_bf16(W.key(S.S_K), W.scales(S.S_K), W.L, W.H, W.T, layers=[l], heads=heads)
        vx = S.laplace_bf16(W.key(S.S_V), W.scales(S.S_V), W.L, W.H, W.T, layers=[l], heads=heads)
        kr, vr = orc.quantize(kx), orc.quantize(vx)
        # refined dense cache of the layer: sampled pages
        rng = np.repeat(vr["page_meta"][..., 1, :], 256, axis=2)
        full = orc.dequant(vr, True)
        for hi, h in enumerate(heads):
            got = r["dense"][S.S_V][l, h, :4096]
            got = (got.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert_dequant_close(got[None, None], full[:, hi:hi + 1, :4096], rng[:, hi:hi + 1, :4096], True)
        # attention of requests 0 and 3, query heads of KV heads 0 and 5, both modes
        G = W.Hq // W.H
        qsel = np.concatenate([np.arange(h * G, (h + 1) * G) for h in heads])
        qb = r["qb"][[0, 3]][:, qsel]
        table = np.arange(W.pages, dtype=np.int32)[None].repeat(2, 0)
        ctx = np.array([W.T, W.T], np.int32)
        for mode, got in ((0, r["out_anchor"][l]), (1, r["outs"][l])):
            ref = orc.decode_attn(qb, kr, vr, 0, table, ctx, 128 ** -0.5, mode == 1)
            E = attn_sensitivity(orc, qb, kr, vr, 0, table, ctx, 128 ** -0.5, mode == 1)
            g = got[[0, 3]][:, qsel].cpu().numpy()
            assert_attn_close(g, ref, E, f"progressive layer {l} mode {mode}")
