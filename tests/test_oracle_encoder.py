"""Pins of the whole per-page encoder and the two decoders.

Lynx reading, section 3 "The quantizer": per 256-token page, per channel, page
min/range normalisation to [0,1]; chunks of C = 32 tokens centred by the local
mean and divided by the local max-abs; the alpha-law map; the +7 bias and the
4/4 cut. Section 4: the anchor stream alone is the draft cache; the residual
refines it to the full reconstruction.

Pins used here: brute-force code selection on small pages (argmin over all 127
levels in the log domain), metadata against fp64 statistics of the input,
exact invariances (power-of-two scaling, integer shifts, constant channels),
the half-step reconstruction bound, ragged pages, and the nibble layout.
"""
import numpy as np
import pytest

import lynx_synth as S

PAGE, CH, D = 256, 32, 128


def _x_f64(xb):
    return S.bf16_bits_to_f32(xb).astype(np.float64)


def _page(seed, n_out=4, scale=1.0, n=PAGE):
    w = S.Workload("t", seed, L=1, H=1, T=PAGE, n_outliers_fixed=n_out)
    sc = w.scales(S.S_K) * np.float32(scale)
    return S.laplace_bf16(w.key(S.S_K), sc, 1, 1, PAGE)


def _unpack(plane):
    lo = (plane & 15).astype(np.int64)
    hi = (plane >> 4).astype(np.int64)
    out = np.empty(plane.shape[:-1] + (plane.shape[-1] * 2,), np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _codes_from_planes(q):
    A = _unpack(q["anchor"])
    A = np.where(A >= 8, A - 16, A)
    r = _unpack(q["residual"])
    return A, r, 16 * A + r - 7


def _stage12_w(xb, q):
    """w of every element, recomputed in numpy fp32 from the stored metadata
    (mn, rng, mu, s), used only to feed the brute-force level selection."""
    x = S.bf16_bits_to_f32(xb)[0, 0]
    pm = q["page_meta"][0, 0]
    cm = q["chunk_meta"][0, 0].view(np.float16).astype(np.float32)
    P = x.shape[0] // PAGE
    w = np.zeros_like(x)
    for p in range(P):
        mn, rng = pm[p, 0], pm[p, 1]
        inv_r = np.where(rng > 0, np.float32(1) / np.where(rng > 0, rng, 1), 0).astype(np.float32)
        for j in range(8):
            sl = slice(p * PAGE + j * CH, p * PAGE + (j + 1) * CH)
            u = ((x[sl] - mn).astype(np.float32) * inv_r).astype(np.float32)
            v = (u - cm[p, j, 0]).astype(np.float32)
            s = cm[p, j, 1]
            inv_s = np.where(s > 0, np.float32(1) / np.where(s > 0, s, 1), 0).astype(np.float32)
            w[sl] = (v * inv_s).astype(np.float32)
    return w


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_brute_force_code_selection(orc, seed):
    xb = _page(seed)
    q = orc.quantize(xb)
    _, _, c = _codes_from_planes(q)
    w = _stage12_w(xb, q).astype(np.float64)
    a = orc.alpha()
    # argmin over the 127 levels of |F(|w|) - k/63| in the log domain, ties upward
    y = 63 * np.log1p(a * np.abs(w)) / np.log1p(a)
    k = np.arange(64)[None, None, :]
    dist = np.abs(y[..., None] - k)
    best = 63 - np.argmin(dist[..., ::-1], axis=-1)     # ties to the larger level
    want = np.where(w < 0, -np.maximum(best, 1), best)
    near_tie = np.abs(np.abs(y - np.floor(y)) - 0.5) < 1e-5
    mism = (c[0, 0] != want) & ~near_tie
    assert not mism.any(), np.argwhere(mism)[:5]


def test_metadata_against_fp64_statistics(orc):
    xb = _page(21, n_out=8)
    q = orc.quantize(xb)
    x = _x_f64(xb)[0, 0]
    pm = q["page_meta"][0, 0, 0].astype(np.float64)
    cm = q["chunk_meta"][0, 0, 0].view(np.float16).astype(np.float64)
    mn, rng = x.min(0), x.max(0) - x.min(0)
    assert np.array_equal(pm[0], mn)                               # page minimum, exact
    assert np.all(np.abs(pm[1] - rng) <= np.spacing(rng.astype(np.float32)))
    u = (x - mn) / rng
    for j in range(8):
        uj = u[j * CH:(j + 1) * CH]
        mean = uj.mean(0)
        ulp = np.spacing(np.abs(mean).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(cm[j, 0] - mean) <= 0.5 * ulp + 1e-6)      # fp16 nearest mean
        smax = np.abs(uj - cm[j, 0]).max(0)
        assert np.all(cm[j, 1] >= smax - 1e-6)                          # rounded up: covers max|v|
        sulp = np.spacing(cm[j, 1].astype(np.float16)).astype(np.float64)
        assert np.all(cm[j, 1] - smax <= sulp + 1e-6)                   # ... by at most one ulp


def test_power_of_two_scaling_and_integer_shift_are_exact_invariances(orc):
    xb = _page(31)
    q0 = orc.quantize(xb)
    # x * 4: codes and chunk metadata identical, page metadata scaled by 4
    x4 = S.f32_to_bf16_bits(S.bf16_bits_to_f32(xb) * np.float32(4))
    q4 = orc.quantize(x4)
    for k in ("anchor", "residual", "chunk_meta"):
        assert np.array_equal(q0[k], q4[k]), k
    assert np.array_equal(q4["page_meta"], q0["page_meta"] * 4)
    # integer-valued data shifted by an integer (both exact in bf16, |x| <= 256):
    # codes identical, page minimum shifted
    xr = np.clip(np.round(S.bf16_bits_to_f32(xb) * 8), -100, 100).astype(np.float32)
    xi = S.f32_to_bf16_bits(xr)
    xs = S.f32_to_bf16_bits(xr + np.float32(37))
    assert np.array_equal(S.bf16_bits_to_f32(xs), xr + 37)
    qi, qs = orc.quantize(xi), orc.quantize(xs)
    for k in ("anchor", "residual", "chunk_meta"):
        assert np.array_equal(qi[k], qs[k]), k
    assert np.array_equal(qs["page_meta"][..., 0, :], qi["page_meta"][..., 0, :] + 37)


def test_constant_channel_codes_zero_and_decodes_exactly(orc):
    xb = _page(41)
    xb[..., 5] = S.f32_to_bf16_bits(np.full(PAGE, 3.25, np.float32))
    q = orc.quantize(xb)
    A, r, c = _codes_from_planes(q)
    assert np.all(c[..., 5] == 0)
    assert q["page_meta"][0, 0, 0, 1, 5] == 0.0
    for full in (False, True):
        assert np.all(orc.dequant(q, full)[..., 5] == 3.25)


def test_reconstruction_within_half_a_log_step(orc):
    """|x - x_full| <= rng*s*((1+a)^(1/126) - 1)*(|w| + 1/a) (half a code step,
    section 3's log map), plus fp16 level rounding and fp32 slop; the anchor
    alone stays within 8.5 code steps."""
    a = orc.alpha()
    for seed in (51, 52):
        xb = _page(seed, n_out=6)
        q = orc.quantize(xb)
        x = _x_f64(xb)[0, 0]
        rng = q["page_meta"][0, 0, 0, 1].astype(np.float64)[None, :]
        s = np.repeat(q["chunk_meta"][0, 0, 0, :, 1].view(np.float16).astype(np.float64), CH, axis=0)
        scale = rng * s
        slop = 8 * 2.0 ** -24 * (np.abs(x) + np.abs(q["page_meta"][0, 0, 0, 0])[None, :] + rng)
        for full, steps in ((True, 0.5), (False, 8.5)):
            xh = orc.dequant(q, full)[0, 0]
            step = ((1 + a) ** (steps / 63) - 1) * (1 + 1 / a) + 2.0 ** -11 * 1.1
            assert np.all(np.abs(xh - x) <= scale * step + slop)


def test_full_beats_anchor_and_anchor_keeps_order_of_magnitude(orc):
    xb = _page(61)
    q = orc.quantize(xb)
    x = _x_f64(xb)
    ef = np.abs(orc.dequant(q, True) - x).mean()
    ea = np.abs(orc.dequant(q, False) - x).mean()
    assert ef < ea / 4


def test_residual_centre_gives_anchor_decode(orc):
    """Residual planes of 7 everywhere turn the full decode into the anchor decode."""
    q = orc.quantize(_page(71))
    q7 = dict(q)
    q7["residual"] = np.full_like(q["residual"], 0x77)
    assert np.array_equal(orc.dequant(q7, True), orc.dequant(q, False))


def test_nibble_layout_even_channel_low(orc):
    xb = _page(81)
    q = orc.quantize(xb)
    A, r, c = _codes_from_planes(q)
    # pick the element with the largest positive code in channel 2 and 3
    for d in (2, 3):
        t = int(np.argmax(c[0, 0, :, d]))
        byte = q["residual"][0, 0, t, d // 2]
        nib = (byte & 15) if d % 2 == 0 else (byte >> 4)
        assert nib == r[0, 0, t, d]
        # independent: the largest |x - mn| in a chunk with positive deviation has a large code
        assert c[0, 0, t, d] > 40


@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 100, 255])
def test_ragged_page(orc, n):
    w = S.Workload("t", 90 + n, L=1, H=2, T=2 * PAGE, n_outliers_fixed=3)
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, 2, 2 * PAGE)
    pv = np.array([PAGE, n], np.int32)
    q = orc.quantize(xb, pv)
    full = orc.quantize(xb)
    # the full first page is untouched by the ragged second one
    assert np.array_equal(q["anchor"][:, :, :PAGE], full["anchor"][:, :, :PAGE])
    # invalid rows carry code 0: anchor 0, residual 7
    assert np.all(q["anchor"][:, :, PAGE + n:] == 0)
    assert np.all(q["residual"][:, :, PAGE + n:] == 0x77)
    # the valid prefix encodes as a page of its own would (stats over valid rows only)
    if n:
        x = _x_f64(xb)[:, :, PAGE:PAGE + n]
        assert np.array_equal(q["page_meta"][:, :, 1, 0], x.min(2).astype(np.float32))
        nc = (n + CH - 1) // CH
        assert np.all(q["chunk_meta"][:, :, 1, nc:] == 0)           # empty chunks: mu = s = 0
    else:
        assert np.all(q["page_meta"][:, :, 1] == 0)
        assert np.all(q["chunk_meta"][:, :, 1] == 0)


def test_layout_of_multi_layer_tensor(orc):
    """[L,H,T,128] pages are independent: encoding a slice equals slicing the encoding."""
    w = S.Workload("t", 7, L=2, H=3, T=3 * PAGE, n_outliers_fixed=2)
    xb = S.laplace_bf16(w.key(S.S_V), w.scales(S.S_V), 2, 3, 3 * PAGE)
    q = orc.quantize(xb)
    sub = orc.quantize(np.ascontiguousarray(xb[1:2, 2:3, PAGE:2 * PAGE]))
    assert np.array_equal(q["anchor"][1:2, 2:3, PAGE:2 * PAGE], sub["anchor"])
    assert np.array_equal(q["residual"][1:2, 2:3, PAGE:2 * PAGE], sub["residual"])
    assert np.array_equal(q["page_meta"][1:2, 2:3, 1:2], sub["page_meta"])
    assert np.array_equal(q["chunk_meta"][1:2, 2:3, 1:2], sub["chunk_meta"])


def test_signed_zero_extremes_store_plus_zero(orc):
    """A page whose minimum (or maximum) is a zero stores +0 whether the data
    held +0 or -0, and the codes do not depend on the zero's sign."""
    xb = _page(91)
    xf = S.bf16_bits_to_f32(xb).copy()
    xf[0, 0, :, 7] = np.abs(xf[0, 0, :, 7])          # channel 7 >= 0, minimum at a zero
    xf[0, 0, 10, 7] = 0.0
    xf[0, 0, :, 9] = -np.abs(xf[0, 0, :, 9])         # channel 9 <= 0, maximum at a zero
    xf[0, 0, 20, 9] = 0.0
    a = S.f32_to_bf16_bits(xf)
    b = a.copy()
    b[0, 0, 10, 7] = 0x8000                            # -0 in place of +0
    b[0, 0, 20, 9] = 0x8000
    qa, qb = orc.quantize(a), orc.quantize(b)
    for k in ("anchor", "residual", "page_meta", "chunk_meta"):
        assert np.array_equal(qa[k].view(np.uint8), qb[k].view(np.uint8)), k
    assert qa["page_meta"][0, 0, 0, 0, 7].view(np.uint32) == 0       # +0 minimum
    assert qa["page_meta"][0, 0, 0, 1, 9] > 0


def test_ragged_chunk_metadata_against_fp64_statistics(orc):
    """A page with 77 valid tokens: chunk 2 holds 13 of them; its mean and scale
    are statistics of those 13 values only."""
    n = 77
    w = S.Workload("t", 95, L=1, H=1, T=PAGE, n_outliers_fixed=4)
    xb = S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K), 1, 1, PAGE)
    q = orc.quantize(xb, np.array([n], np.int32))
    x = _x_f64(xb)[0, 0, :n]
    mn, rng = x.min(0), x.max(0) - x.min(0)
    u = (x - mn) / rng
    cm = q["chunk_meta"][0, 0, 0].view(np.float16).astype(np.float64)
    for j in range(3):
        uj = u[j * CH:min((j + 1) * CH, n)]
        mean = uj.mean(0)
        ulp = np.spacing(np.abs(mean).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(cm[j, 0] - mean) <= 0.5 * ulp + 1e-6), j
        smax = np.abs(uj - cm[j, 0]).max(0)
        assert np.all(cm[j, 1] >= smax - 1e-6) and np.all(cm[j, 1] - smax <= np.spacing(
            cm[j, 1].astype(np.float16)).astype(np.float64) + 1e-6), j


def _special_page():
    """A page with channels whose statistics fp32 cannot carry, and the same page
    without them."""
    base = _page(97)
    xf = S.bf16_bits_to_f32(base).copy()
    xf[0, 0, :, 4] = np.abs(xf[0, 0, :, 4])
    xf[0, 0, 9, 4] = np.inf                             # infinite value: range inf
    xf[0, 0, :, 5] = 1.0
    xf[0, 0, 3, 5], xf[0, 0, 200, 5] = -3.0e38, 3.0e38  # finite values, range beyond fp32
    xf[0, 0, :, 6] = 0.0
    xf[0, 0, 17, 6] = 2.0 ** -130                       # subnormal range, 1/range overflows
    xf[0, 0, :, 8] = 0.0
    xf[0, 0, 40, 8] = 2.0 ** -126                       # smallest normal range: representable
    xb = S.f32_to_bf16_bits(xf)
    xb[0, 0, 5, 3] = 0x7FC1                             # a NaN (non-canonical payload)
    return base, xb


def test_unrepresentable_statistics_code_the_channel_as_constant(orc):
    """Reading for inputs the pages leave open: a NaN value stores min and range
    as the quiet NaN 0x7FC00000; a range (or reciprocal) that fp32 cannot carry
    codes every value of the channel as 0 with chunk mean and scale 0; other
    channels, and a tiny but representable range, are untouched."""
    base, xb = _special_page()
    q, qb = orc.quantize(xb), orc.quantize(base)
    A, r, c = _codes_from_planes(q)
    pm, cm = q["page_meta"][0, 0, 0], q["chunk_meta"][0, 0, 0]
    assert pm[0, 3].view(np.uint32) == 0x7FC00000 and pm[1, 3].view(np.uint32) == 0x7FC00000
    assert np.isinf(pm[1, 4]) and np.isfinite(pm[0, 4])
    assert np.isinf(pm[1, 5]) and pm[0, 5] == np.float32(S.bf16_bits_to_f32(xb)[0, 0, 3, 5])
    assert pm[0, 6] == 0.0 and pm[1, 6] == np.float32(2.0 ** -130)
    for ch in (3, 4, 5, 6):
        assert np.all(c[0, 0, :, ch] == 0), ch
        assert np.all(A[0, 0, :, ch] == 0) and np.all(r[0, 0, :, ch] == 7), ch
        assert np.all(cm[:, :, ch] == 0), ch
    # the smallest normal range is an ordinary channel: u = 1 at token 40, 0 elsewhere
    assert pm[1, 8] == np.float32(2.0 ** -126)
    assert c[0, 0, 40, 8] == 63 and np.count_nonzero(c[0, 0, :, 8]) >= 1
    others = [d for d in range(D) if d not in (3, 4, 5, 6, 8)]
    cb = _codes_from_planes(qb)[2]
    assert np.array_equal(c[..., others], cb[..., others])
    assert np.array_equal(q["page_meta"][..., others].view(np.uint32), qb["page_meta"][..., others].view(np.uint32))
