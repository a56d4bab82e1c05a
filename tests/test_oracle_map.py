"""Pins of stage 3 (alpha-law map, sign-aware mapping) and stage 4 (bias, cut).

Lynx reading, section 3: |w| goes through a logarithmic alpha-law map onto
127 levels; small negative values keep their sign through a sign-aware rule
(a negative w whose level rounds to 0 is coded -1); adding 7 before the 4-bit
shift rounds the anchor half down, so the residual is a signed correction
centred on the anchor; each code is cut into a 4-bit anchor and a 4-bit
residual.
"""
import numpy as np


def _F63(w, alpha):
    return 63.0 * np.log1p(alpha * np.abs(np.asarray(w, np.float64))) / np.log1p(alpha)


def _sweep_values(thr):
    """Every 101st fp32 in [0, 1] plus +-2048 ulps around each threshold."""
    top = int(np.float32(1.0).view(np.uint32))
    base = np.arange(0, top + 1, 101, dtype=np.uint32)
    near = [np.arange(int(t) - 2048, int(t) + 2048, dtype=np.uint32) for t in thr[1:].view(np.uint32)]
    extra = np.array([top, top + 1, top + 2], np.uint32)
    return np.unique(np.concatenate([base] + near + [extra])).view(np.float32)


def test_map_is_round_half_up_in_log_domain(orc):
    thr, _ = orc.tables()
    a = orc.alpha()
    w = _sweep_values(thr)
    got = orc.codes(w).astype(np.int64)
    y = _F63(w, a)
    want = np.minimum(np.floor(y + 0.5), 63).astype(np.int64)
    bad = got != want
    # disagreements may only sit within one fp32 rounding of a half-level crossing
    frac = np.abs(y[bad] - np.round(y[bad] - 0.5) - 0.5)
    assert np.all(frac < 1e-5), frac.max() if frac.size else 0
    assert bad.sum() <= 2 * 63
    assert got.min() == 0 and got.max() == 63


def test_map_saturates_and_boundaries(orc):
    thr, _ = orc.tables()
    c = orc.codes(np.array([0.0, 1.0, np.nextafter(np.float32(1), np.float32(2)), 1.5], np.float32))
    assert list(c) == [0, 63, 63, 63]
    # exactly at a threshold the code steps up (ties go up)
    for k in range(1, 64):
        t = thr[k]
        below = np.nextafter(t, np.float32(0))
        assert orc.codes(np.array([t], np.float32))[0] == k
        assert orc.codes(np.array([below], np.float32))[0] == k - 1


def test_sign_aware_mapping_keeps_small_negatives_negative(orc):
    thr, _ = orc.tables()
    lv = orc.level_values()
    t1 = thr[1]
    w = -np.linspace(np.float32(1e-12), t1, 1000, endpoint=False, dtype=np.float32)
    w = np.concatenate([w, [np.float32(-1e-30), -np.nextafter(t1, np.float32(0))]]).astype(np.float32)
    c = orc.codes(w)
    assert np.all(c == -1)
    # the decode of -1 is below the chunk mean: -Lv[1] < 0
    assert -lv[1] < 0
    # non-negative values below the first threshold give 0; -0 counts as non-negative
    z = np.array([0.0, -0.0, 1e-30, np.nextafter(t1, np.float32(0))], np.float32)
    assert np.all(orc.codes(z) == 0)
    # larger negatives mirror the positives
    pos = np.linspace(t1, 1.0, 5000, dtype=np.float32)
    assert np.array_equal(orc.codes(-pos), -orc.codes(pos))


def test_codes_span_127_levels(orc):
    w = np.linspace(-1, 1, 200001, dtype=np.float32)
    c = orc.codes(w)
    assert set(np.unique(c).tolist()) == set(range(-63, 64))


def test_split_enumerates_all_codes(orc):
    c = np.arange(-63, 64, dtype=np.int8)
    A, r = orc.split(c)
    A = A.astype(np.int64)
    r = r.astype(np.int64)
    assert np.array_equal(16 * A + r - 7, c.astype(np.int64))          # lossless cut
    assert A.min() == -4 and A.max() == 4                                # anchor fits 4 signed bits
    assert r.min() == 0 and r.max() == 15                                # residual fits 4 bits
    corr = r - 7                                                         # c - 16A
    assert corr.min() == -7 and corr.max() == 8                          # centred, signed
    # round-half-down of c/16: ties (c = 16A + 8) go to the lower anchor
    ci = c.astype(np.int64)
    assert np.array_equal(A, np.ceil((ci - 8) / 16).astype(np.int64))
    assert np.all(np.abs(ci - 16 * A) <= 8)
    # without the bias the residual would be one-sided: floor(c/16) leaves 0..15
    assert np.all((c.astype(np.int64) - 16 * np.floor(c / 16)) >= 0)
    assert abs(corr.mean()) < 1.0


def test_anchor_nibble_is_twos_complement(orc):
    c = np.arange(-63, 64, dtype=np.int8)
    A, r = orc.split(c)
    nib = (A.astype(np.int64) & 15)
    back = np.where(nib >= 8, nib - 16, nib)
    assert np.array_equal(back, A.astype(np.int64))
