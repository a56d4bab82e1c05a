"""The encoder's reciprocal of a chunk scale (an fp16 value): the hardware
approximation r followed by one Newton step r + r (1 - s r), as two fused
multiply-adds, is the correctly rounded fp32 reciprocal. Checked here for every
positive finite fp16 value s and every starting point r within 2 ulp of the
correctly rounded 1/s, in exact rational arithmetic, so the claim does not
depend on how close the hardware approximation is within that bound."""
from fractions import Fraction

import numpy as np


def _rn32(x):
    """Nearest fp32 to the exact rational x (ties to even)."""
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - x), int(np.float32(c).view(np.uint32)) & 1))


def test_newton_step_gives_the_correctly_rounded_reciprocal():
    s_all = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    wrong = []
    for s in s_all:
        S = Fraction(float(s))
        want = _rn32(1 / S)
        for k in range(-2, 3):
            r = np.int32(want.view(np.int32) + k).view(np.float32)
            R = Fraction(float(r))
            e = _rn32(1 - S * R)                 # fma(-s, r, 1): one rounding
            got = _rn32(R + R * Fraction(float(e)))   # fma(r, e, r): one rounding
            if got != want:
                wrong.append((float(s), k))
    assert not wrong, wrong[:5]


def test_the_bound_is_tight_enough_to_matter():
    """A plain rounded product r * (2 - s r) in fp32 (two roundings, no fused
    step) is not always correct: the pin would catch a step written that way."""
    rng = np.random.default_rng(3)
    s_all = rng.choice(np.arange(1, 0x7C00, dtype=np.uint16), 4000, replace=False).view(np.float16).astype(np.float32)
    misses = 0
    for s in s_all:
        S = Fraction(float(s))
        want = _rn32(1 / S)
        r = np.int32(want.view(np.int32) + 1).view(np.float32)
        t = _rn32(2 - S * Fraction(float(r)))     # rounded, not fused
        got = _rn32(Fraction(float(r)) * Fraction(float(t)))
        misses += got != want
    assert misses > 0
