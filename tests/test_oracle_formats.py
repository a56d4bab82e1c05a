"""Pins of the oracle's number-format helpers against numpy and brute force."""
import numpy as np


def _all_finite_f16():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16)
    keep = np.isfinite(v)
    return h[keep], v[keep].astype(np.float64)


def test_f16_nearest_matches_numpy(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.uniform(-9, 4, 3000),
        np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 0.5 + 2.0 ** -12, 1.0 + 2.0 ** -11]),
    ]).astype(np.float32)
    got = np.array([orc.f16_bits(float(v)) for v in x], np.uint16)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_round_up_is_smallest_f16_not_below(orc):
    bits, vals = _all_finite_f16()
    order = np.argsort(vals, kind="stable")
    sv = vals[order]
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(0, 1, 2000) * 10.0 ** rng.uniform(-8, 0, 2000),
                        sv[(sv > 0) & (sv < 2)][::37]]).astype(np.float32).astype(np.float64)
    for v in x:
        got = orc.f16_value(orc.f16_bits(v, round_up=True))
        i = np.searchsorted(sv, v, side="left")
        assert got == sv[i], (v, got, sv[i])
        assert got >= v


def test_f16_decode_matches_numpy(orc):
    bits, vals = _all_finite_f16()
    for b, v in zip(bits[::61], vals[::61]):
        assert orc.f16_value(int(b)) == v
