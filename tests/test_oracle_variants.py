"""Pins of the variant oracle (oracle/variants.py) to what the pages and the
mathematics fix: the default configuration reproduces the main oracle's codes,
metadata and reconstructions (section 3's own configuration); the linear map
is the closed-form round-half-up grid; the alpha-law levels grow as
(1+alpha)^(q/q_max); the bias-and-cut identities hold for every code of every
split; the sign-aware rule, the chunk-isolation-off reading and the uniform
comparator's half-step bound hold by brute force on tiny inputs."""
import numpy as np
import pytest

import lynx_synth as S
from oracle import variants as V

SPLITS = [(4, 4), (2, 4), (6, 2), (3, 3), (4, 2)]


@pytest.fixture(scope="module")
def xb():
    w = S.WORKLOADS[2]                     # Laplace with outlier channels (x10^U(1,2))
    x = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K)[:1, :2], 1, 2, 512)
    return x.reshape(2, 512, 128)


def _unpack(plane):
    lo = (plane & 15).astype(np.int32)
    hi = (plane >> 4).astype(np.int32)
    out = np.empty(plane.shape[:-1] + (128,), np.int32)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return out


def test_default_matches_main_oracle(orc, xb):
    q = orc.quantize(xb.reshape(1, 2, 512, 128))
    o = V.encode(xb)
    A = _unpack(q["anchor"]).reshape(2, 512, 128)
    A = np.where(A >= 8, A - 16, A)
    r = _unpack(q["residual"]).reshape(2, 512, 128)
    assert np.array_equal(o["anchor"], A) and np.array_equal(o["residual"], r)
    assert np.array_equal(o["page_meta"].view(np.uint32), q["page_meta"].reshape(2, 2, 2, 128).view(np.uint32))
    assert np.array_equal(o["chunk_meta"], q["chunk_meta"].reshape(2, 2, 8, 2, 128))
    assert np.array_equal(o["x_full"], orc.dequant(q, True).reshape(2, 512, 128))
    assert np.array_equal(o["x_anchor"], orc.dequant(q, False).reshape(2, 512, 128))


def test_linear_map_is_the_round_half_up_grid():
    v = V.Variant(alpha=0.0)
    qm = v.qmax
    assert np.array_equal(V.thresholds(v)[1:], np.float32((np.arange(1, qm + 1) - 0.5) / qm))
    w = np.random.default_rng(3).uniform(-1, 1, 20000).astype(np.float32)
    c = V._stage3(w, v)
    exact = np.floor(qm * np.abs(w.astype(np.float64)) + 0.5)
    far = np.abs(qm * np.abs(w.astype(np.float64)) + 0.5 - np.round(qm * np.abs(w) + 0.5)) > 1e-4
    q = np.abs(c)
    ok = np.where(w < 0, q == np.maximum(exact, 1), q == exact)
    assert np.all(ok[far])
    assert np.array_equal(V.levels(v), np.float16(np.arange(qm + 2) / qm).astype(np.float64))


@pytest.mark.parametrize("alpha", [15.0, 255.0, 1023.0])
def test_alpha_law_levels_grow_geometrically(alpha):
    v = V.Variant(alpha=alpha)
    lv = V.levels(v)
    assert lv[0] == 0.0 and np.all(np.diff(lv) > 0)
    k = np.arange(v.qmax // 2, v.qmax + 2)
    ratio = (lv[k] + 1 / alpha) / (lv[k - 1] + 1 / alpha)
    assert np.allclose(ratio, (1 + alpha) ** (1 / v.qmax), rtol=3e-3)
    thr = V.thresholds(v)
    mid = ((1 + alpha) ** ((np.arange(1, v.qmax + 1) - 0.5) / v.qmax) - 1) / alpha
    assert np.allclose(thr[1:], mid, rtol=1e-6)


@pytest.mark.parametrize("a,r", SPLITS)
@pytest.mark.parametrize("bias", [True, False])
def test_split_identities_every_code(a, r, bias):
    v = V.Variant(anchor_bits=a, residual_bits=r, bias=bias)
    c = np.arange(-v.qmax, v.qmax + 1)
    A, rr = V.split(c, v)
    b = v.bias_value
    assert b == ((1 << (r - 1)) - 1 if bias else 0)
    assert np.array_equal((A << r) + rr - b, c)
    assert rr.min() >= 0 and rr.max() <= (1 << r) - 1
    assert A.min() >= -(1 << (a - 1)) and A.max() <= (1 << (a - 1)) - 1
    d = c - (A << r)                               # the correction the residual carries
    if bias:
        assert d.min() >= -b and d.max() <= (1 << r) - 1 - b      # centred, signed
    else:
        assert d.min() >= 0                                        # one-sided
    assert np.abs(A << r).max() <= v.qmax + 1


def test_sign_aware_mapping():
    w = np.array([-1e-6, 1e-6, -0.0, 0.0, -0.5, 0.5], np.float32)
    on = V._stage3(w, V.Variant())
    off = V._stage3(w, V.Variant(sign_aware=False))
    assert list(on[:4]) == [-1, 0, 0, 0] and list(off[:4]) == [0, 0, 0, 0]
    assert on[4] == -on[5] and off[4] == -off[5]


def test_no_chunk_isolation_reading(xb):
    o = V.encode(xb, V.Variant(chunk_isolation=False))
    assert np.all(o["chunk_meta"] == 0x3800)                       # fp16 0.5
    x = (xb.astype(np.uint32) << 16).view(np.float32).reshape(2, 2, 256, 128)
    c = o["codes"].reshape(2, 2, 256, 128)
    imax, imin = x.argmax(axis=2), x.argmin(axis=2)
    top = np.take_along_axis(c, imax[:, :, None, :], axis=2)
    bot = np.take_along_axis(c, imin[:, :, None, :], axis=2)
    assert np.all(top == V.Variant().qmax) and np.all(bot == -V.Variant().qmax)


@pytest.mark.parametrize("C", [16, 32, 64])
def test_each_chunk_reaches_the_top_level(xb, C):
    v = V.Variant(chunk=C)
    o = V.encode(xb, v)
    assert o["chunk_meta"].shape == (2, 2, 256 // C, 2, 128)
    c = np.abs(o["codes"]).reshape(2, 2, 256 // C, C, 128).max(axis=3)
    s = o["chunk_meta"][:, :, :, 1, :].view(np.float16).astype(np.float64)
    assert np.all(c[s > 0] == v.qmax)


@pytest.mark.parametrize("bits", [4, 8])
def test_uniform_comparator_half_step(xb, bits):
    o = V.encode(xb, V.Variant(uniform_bits=bits))
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(2, 2, 256, 128)
    pm = o["page_meta"]
    step = pm[:, :, 1, :].astype(np.float64) / (2 ** bits - 1)
    e = np.abs(o["x_full"].reshape(2, 2, 256, 128) - x)
    assert np.all(e <= step[:, :, None, :] * (0.5 + 1e-5) + 1e-12)
    c = o["codes"].reshape(2, 2, 256, 128)
    assert c.min() == 0 and c.max() == 2 ** bits - 1


def test_page_norm_off_changes_little(xb):
    """Chunk isolation is affine-invariant, so without page normalisation the
    codes move only where the fp16 chunk mean and scale round differently:
    by one level almost everywhere they move at all."""
    a = V.encode(xb)["codes"]
    b = V.encode(xb, V.Variant(page_norm=False))
    assert np.all(b["page_meta"][:, :, 0] == 0) and np.all(b["page_meta"][:, :, 1] == 1)
    d = np.abs(a - b["codes"])
    assert (d == 0).mean() > 0.95 and (d <= 1).mean() > 0.995 and d.max() <= 4


def test_six_bit_split_range(xb):
    v = V.Variant(anchor_bits=2, residual_bits=4)
    o = V.encode(xb, v)
    assert v.qmax == 15 and np.abs(o["codes"]).max() == 15
    assert o["anchor"].min() >= -2 and o["anchor"].max() <= 1


def test_error_sums_and_orders(xb):
    o = V.encode(xb)
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(2, 2, 256, 128)
    assert np.allclose(o["err"][..., 0], (x * x).sum(axis=(2, 3)))
    assert np.allclose(o["err"][..., 2], ((o["x_full"].reshape(x.shape) - x) ** 2).sum(axis=(2, 3)))
    ea, ef = V.vnmse(o["err"])
    assert ef < ea                                  # the residual refines
    e4 = V.vnmse(V.encode(xb, V.Variant(uniform_bits=4))["err"])[0]
    e8 = V.vnmse(V.encode(xb, V.Variant(uniform_bits=8))["err"])[0]
    assert e8 < e4


@pytest.mark.parametrize("C", [16, 64])
def test_chunk_statistics_against_fp64(xb, C):
    o = V.encode(xb, V.Variant(chunk=C))
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(2, 2, 256, 128)
    pm = o["page_meta"].astype(np.float64)
    u = (x - pm[:, :, None, 0, :]) / pm[:, :, None, 1, :]
    uc = u.reshape(2, 2, 256 // C, C, 128)
    mu = o["chunk_meta"][:, :, :, 0, :].view(np.float16).astype(np.float64)
    s = o["chunk_meta"][:, :, :, 1, :].view(np.float16).astype(np.float64)
    ulp = np.spacing(np.abs(mu).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(mu - uc.mean(axis=3)) <= ulp * 0.5 + 1e-6)
    dev = np.abs(uc - mu[:, :, :, None, :]).max(axis=3)
    assert np.all(s >= dev * (1 - 1e-6)) and np.all(s <= dev * (1 + 2.0 ** -10) + 2.0 ** -24)


@pytest.mark.parametrize("bits", [4, 8])
def test_uniform_per_token_half_step(xb, bits):
    o = V.encode(xb, V.Variant(uniform_bits=bits, uniform_per_token=True))
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    step = (x.max(axis=-1) - x.min(axis=-1)) / (2 ** bits - 1)
    e = np.abs(o["x_full"] - x)
    assert np.all(e <= step[..., None] * (0.5 + 1e-5) + 1e-12)
    c = o["codes"]
    assert np.all(c.min(axis=-1) == 0) and np.all(c.max(axis=-1) == 2 ** bits - 1)
    # outlier channels widen every token's grid: per token is coarser here
    per_chan = V.vnmse(V.encode(xb, V.Variant(uniform_bits=bits))["err"])[1]
    assert V.vnmse(o["err"])[1] > per_chan


# ---- attention-output error (the measure of the section 5 figures) -------

def test_dense_attention_equals_paged_decode_over_the_reconstruction(orc, xb):
    """One decode step over the dense full reconstruction is the main
    oracle's paged decode attention over the same cache (identity page table,
    every request attending to all tokens): two independent codes."""
    H, T = 2, 512
    xk = xb.reshape(1, H, T, 128)
    xv = xb[::-1].copy().reshape(1, H, T, 128)
    k, v = orc.quantize(xk), orc.quantize(xv)
    q = S.WORKLOADS[2].queries_bf16(3, 4)
    sm = 1 / np.sqrt(128)
    table = np.tile(np.arange(T // 256, dtype=np.int32), (3, 1))
    ctx = np.full(3, T, np.int32)
    for full in (False, True):
        want = orc.decode_attn(q, k, v, 0, table, ctx, sm, full)
        Kd = V.encode(xk[0])["x_full" if full else "x_anchor"]
        Vd = V.encode(xv[0])["x_full" if full else "x_anchor"]
        got = V.dense_attn(q, Kd, Vd, sm)
        assert np.allclose(got, want, rtol=1e-10, atol=1e-12)


def test_dense_attention_brute_force_with_head_groups():
    """Pure-Python softmax on a tiny case with 4 query heads over 2 KV heads
    (query head h reads KV head h // 2)."""
    import math
    rng = np.random.default_rng(11)
    H, T, B, Hq = 2, 5, 2, 4
    k = rng.normal(size=(H, T, 128))
    v = rng.normal(size=(H, T, 128))
    q = S.f32_to_bf16_bits(rng.normal(size=(B, Hq, 128)).astype(np.float32))
    qf = S.bf16_bits_to_f32(q).astype(np.float64)
    sm = 0.3
    got = V.dense_attn(q, k, v, sm)
    for b in range(B):
        for h in range(Hq):
            g = h // 2
            s = [sm * sum(float(qf[b, h, i]) * float(k[g, t, i]) for i in range(128)) for t in range(T)]
            e = [math.exp(x) for x in s]
            z = sum(e)
            for i in range(0, 128, 17):
                want = sum(e[t] * float(v[g, t, i]) for t in range(T)) / z
                assert abs(got[b, h, i] - want) <= 1e-12 * (1 + abs(want))


def test_dense_attention_special_cases():
    rng = np.random.default_rng(12)
    v = rng.normal(size=(1, 7, 128))
    q = S.f32_to_bf16_bits(rng.normal(size=(2, 3, 128)).astype(np.float32))
    # one token: the output is its value row
    assert np.allclose(V.dense_attn(q, rng.normal(size=(1, 1, 128)), v[:, :1], 0.1), v[0, 0], rtol=0, atol=1e-15)
    # equal scores: the output is the mean of the values
    assert np.allclose(V.dense_attn(q, np.zeros((1, 7, 128)), v, 0.1), v[0].mean(axis=0), rtol=0, atol=1e-14)
    # a dominant key: the output is that key's value row
    k = np.zeros((1, 7, 128))
    k[0, 4] = 1e3 * np.sign(S.bf16_bits_to_f32(q[0, 0]))
    assert np.allclose(V.dense_attn(q[:1, :1], k, v, 1.0)[0, 0], v[0, 4], atol=1e-12)


def test_attention_vnmse_closed_forms():
    o = np.random.default_rng(13).normal(size=(3, 4, 128))
    assert V.attn_vnmse(o, o) == 0.0
    assert abs(V.attn_vnmse(1.1 * o, o) - 0.01) < 1e-12
    assert abs(V.attn_vnmse(np.zeros_like(o), o) - 1.0) < 1e-15
