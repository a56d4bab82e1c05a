"""Pins of the alpha-law thresholds and level values.

The page (Lynx reading, section 3 "Non-linear transform" / "The cut") fixes 127
levels and a reconstructed magnitude that scales as (1+alpha)^q; it leaves alpha
open (the oracle takes 255). These tests check the tables through the inverse
map ln(1 + alpha y)/ln(1 + alpha), which the oracle never evaluates, and against
the stored fixture written by tests/golden/make_golden.py.
"""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tables_alpha255.json")


def _F(y, alpha):
    return np.log1p(alpha * np.asarray(y, np.float64)) / np.log1p(alpha)


def test_alpha_is_the_stated_reading(orc):
    assert orc.alpha() == 255.0


def test_thresholds_sit_at_half_levels(orc):
    thr, _ = orc.tables()
    a = orc.alpha()
    k = np.arange(1, 64)
    t = thr[1:].astype(np.float64)
    # the fp32 threshold is the fp32 nearest to the crossing of 63 F(y) = k - 1/2
    y = 63.0 * _F(t, a)
    assert np.all(np.abs(y - (k - 0.5)) < 1e-5)
    up = np.nextafter(thr[1:], np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(thr[1:], np.float32(-np.inf)).astype(np.float64)
    # neighbours straddle the crossing or lie further from it
    assert np.all(np.abs(63 * _F(up, a) - (k - 0.5)) >= np.abs(y - (k - 0.5)) - 1e-12)
    assert np.all(np.abs(63 * _F(dn, a) - (k - 0.5)) >= np.abs(y - (k - 0.5)) - 1e-12)
    assert np.all(np.diff(t) > 0) and t[0] > 0 and t[-1] < 1


def test_levels_properties(orc):
    lv = orc.level_values()
    a = orc.alpha()
    assert lv[0] == 0.0
    assert lv[63] == 1.0                      # the top level reproduces max |w| = 1
    assert np.all(np.diff(lv) > 0)
    k = np.arange(65)
    # each level is the fp16 nearest to F^-1(k/63): its image under 63 F is k
    assert np.all(np.abs(63 * _F(lv, a) - k) < 0.02)
    # fp16 nearest: within half an fp16 ulp of the exact inverse
    exact = np.expm1(k / 63.0 * np.log1p(a)) / a
    ulp = np.spacing(exact.astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(lv - exact) <= 0.5 * ulp + 1e-18)


def test_anchor_magnitude_is_geometric(orc):
    """'reconstructed magnitude scales as (1+alpha)^q' for the anchor steps."""
    lv = orc.level_values()
    a = orc.alpha()
    ratio = (1 + a) ** (16 / 63)
    for A in range(0, 4):
        got = (lv[16 * (A + 1)] + 1 / a) / (lv[16 * A] + 1 / a)
        assert abs(got / ratio - 1) < 2.0 ** -10
    # one code step grows by (1+alpha)^(1/63)
    g = (lv[1:] + 1 / a) / (lv[:-1] + 1 / a)
    assert np.all(np.abs(g / (1 + a) ** (1 / 63) - 1) < 2e-3)


def test_tables_match_golden_fixture(orc):
    with open(GOLDEN) as f:
        g = json.load(f)
    thr, lv = orc.tables()
    assert [int(v) for v in thr.view(np.uint32)] == g["thr_f32_bits"]
    assert [int(v) for v in lv] == g["lv_f16_bits"]
    assert g["alpha"] == orc.alpha()
