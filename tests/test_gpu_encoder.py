"""GPU parity of the encoder (lynx_quantize_pages) and of its stage-3 code path:
bit-exact against the oracle on seeded inputs."""
import numpy as np
import pytest
import torch

import lynx_synth as S
from gpu_helpers import assert_planes_equal, bf16_dev, i32_dev, planes_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lx():
    import __graft_entry__
    __graft_entry__.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def test_level_codes_exhaustive_nonnegative(lx, orc):
    """Every fp32 in [0, 1 + 64 ulp] through the encoder's bucket lookup equals the
    oracle's threshold count."""
    top = int(np.float32(1.0).view(np.uint32)) + 64
    step = 1 << 26
    for lo in range(0, top + 1, step):
        hi = min(lo + step, top + 1)
        w = np.arange(lo, hi, dtype=np.uint32).view(np.float32)
        got = lx.level_codes(torch.from_numpy(w).cuda()).cpu().numpy()
        want = orc.codes(w)
        if not np.array_equal(got, want):
            i = int(np.argmax(got != want))
            raise AssertionError(f"w={w[i]!r} bits={w.view(np.uint32)[i]:#x}: gpu {got[i]} oracle {want[i]}")


def test_level_codes_negative_and_special(lx, orc):
    """Negative values, subnormals, signed zeros and threshold neighbourhoods in
    the stage-3 domain |w| < 2 (stage 2 never produces |w| > 1 + 2^-23)."""
    rng = np.random.default_rng(3)
    w = -np.minimum(np.abs(rng.standard_normal(1 << 22)) * 10.0 ** rng.uniform(-8, 0, 1 << 22), 1.99)
    thr, _ = orc.tables()
    near = np.concatenate([np.arange(int(t) - 300, int(t) + 300, dtype=np.uint32) for t in thr[1:].view(np.uint32)])
    w = np.concatenate([w.astype(np.float32), -near.view(np.float32), near.view(np.float32),
                        np.array([0.0, -0.0, 1e-40, -1e-40, 1.0, -1.0], np.float32)])
    got = lx.level_codes(torch.from_numpy(w).cuda()).cpu().numpy()
    assert np.array_equal(got, orc.codes(w))


def _encode(lx, xb, page_valid=None):
    L, H, T, _ = xb.shape
    q = lx.QuantizedKV.empty(L, H, T)
    lx.quantize_pages(bf16_dev(xb), q, None if page_valid is None else i32_dev(page_valid))
    return planes_np(q)


def test_one_page(lx, orc):
    w = S.WORKLOADS[1]
    for s in (S.S_K, S.S_V):
        xb = S.laplace_bf16(w.key(s), w.scales(s), 1, 1, 256)
        assert_planes_equal(_encode(lx, xb), orc.quantize(xb), f"tensor {s}: ")


@pytest.mark.parametrize("valid", [[256, 100, 0, 33], [1, 31, 32, 255], [0, 0, 0, 0]])
def test_ragged_multi_layer(lx, orc, valid):
    w = S.Workload("t", 77, L=2, H=3, T=4 * 256, n_outliers_fixed=5, base_log10=(-2, 0))
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 2, 3, 4 * 256)
    pv = np.array(valid, np.int32)
    assert_planes_equal(_encode(lx, xb, pv), orc.quantize(xb, pv))


# c0: first channel of the planted pattern (0: the page's first channel half,
# 100: the second; the encoder handles the two halves of a page separately)
@pytest.mark.parametrize("c0", [0, 100])
def test_special_values(lx, orc, c0):
    """Constant channels, signed-zero extremes, huge and tiny magnitudes."""
    w = S.Workload("t", 78, L=1, H=1, T=512, n_outliers_fixed=3)
    xf = S.bf16_bits_to_f32(S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), 1, 1, 512)).copy()
    xf[..., c0 + 0] = 2.5
    xf[..., c0 + 1] = 0.0
    xf[..., c0 + 2] = np.abs(xf[..., c0 + 2])
    xf[0, 0, 5, c0 + 2] = 0.0
    xf[..., c0 + 3] *= 1e30
    xf[..., c0 + 4] *= 1e-30
    xf[0, 0, 0:32, c0 + 5] = 7.0      # a constant chunk inside a varying channel
    xb = S.f32_to_bf16_bits(xf)
    xb[0, 0, 7, c0 + 1] = 0x8000       # -0 among +0
    xb[0, 0, 9, c0 + 2] = 0x8000
    assert_planes_equal(_encode(lx, xb), orc.quantize(xb))


@pytest.mark.parametrize("c0", [0, 100])
def test_unrepresentable_statistics(lx, orc, c0):
    """NaN, infinite, overflowing-range and subnormal-range channels (coded as
    constant, NaN statistics stored as the quiet NaN) next to ordinary ones, in
    every chunk position; bit-exact, metadata included."""
    w = S.Workload("t", 79, L=1, H=2, T=512, n_outliers_fixed=3)
    xf = S.bf16_bits_to_f32(S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, 2, 512)).copy()
    xf[0, 0, 9, c0 + 4] = np.inf
    xf[0, 1, 300, c0 + 4] = -np.inf
    xf[0, 0, :, c0 + 5] = 1.0
    xf[0, 0, 3, c0 + 5], xf[0, 0, 200, c0 + 5] = -3.0e38, 3.0e38
    xf[0, 1, :256, c0 + 6] = 0.0
    xf[0, 1, 17, c0 + 6] = 2.0 ** -130
    xf[0, 1, 256:, c0 + 8] = 0.0
    xf[0, 1, 296, c0 + 8] = 2.0 ** -126
    xb = S.f32_to_bf16_bits(xf)
    xb[0, 0, 5, c0 + 3] = 0x7FC1
    xb[0, 1, 511, c0 + 7] = 0xFF80      # -inf in the last token
    xb[0, 1, 260, c0 + 9] = 0xFFC0      # negative NaN
    assert_planes_equal(_encode(lx, xb), orc.quantize(xb))


def test_page_count_around_the_grid(lx, orc):
    """153 pages (306 channel-half units): a little more work than one round of
    two CTAs per SM on a 152-SM part, so that a few CTAs take a second unit,
    with a ragged last page; bit-exact."""
    w = S.Workload("t", 80, L=1, H=1, T=153 * 256, n_outliers_fixed=4)
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, 1, 153 * 256)
    pv = np.full(153, 256, np.int32)
    pv[-1] = 77
    assert_planes_equal(_encode(lx, xb, pv), orc.quantize(xb, pv))


@pytest.mark.parametrize("which", ["u", "tree", "w", "mean"])
def test_contract_order_pages(lx, orc, which):
    """The pages that tell the contract's operation order apart from the
    plausible alternatives (u and w as products with a reciprocal, the
    stride-halving chunk sum, mean = sum / n_c): bit-exact with the oracle."""
    import test_oracle_contract_order as O
    chunk = {"u": [0x400E] * 32, "tree": O.SEQ_CHUNK, "w": O.W_CHUNK,
             "mean": [0x3D7F, 0x3D9E, 0x3F2B, 0x3B85, 0x3ECE, 0x0000, 0x3F33]}[which]
    xb, valid = O._page(chunk)
    assert_planes_equal(_encode(lx, xb, valid), orc.quantize(xb, valid))


def test_qwen3_235b_like_layer_every_page(lx, orc):
    """4 KV heads x 32K tokens, K and V: every page bit-exact."""
    w = S.WORKLOADS[2]
    for s in (S.S_K, S.S_V):
        xb = S.laplace_bf16(w.key(s), w.scales(s), w.L, w.H, w.T)
        assert_planes_equal(_encode(lx, xb), orc.quantize(xb), f"tensor {s}: ")


def test_device_generator_matches_host_generator(lx):
    w = S.WORKLOADS[2]
    gen = S.DeviceGenerator()
    out = torch.empty((1, 4, 2048, 128), dtype=torch.bfloat16, device="cuda")
    sc = w.scales(S.S_K)
    gen.fill(out, w.key(S.S_K), sc)
    host = S.laplace_bf16(w.key(S.S_K), sc, 1, 4, 2048)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), host)
