"""The variant oracle's pins catch plausible mistakes.

Each case loads a copy of oracle/variants.py with one planted mistake (a
wrong bias or level count, a shifted threshold, a wrong divisor or rounding,
a dropped rule, a wrong centre or axis, a wrong attention head group,
scale, normaliser or error ratio) and runs the pins of
tests/test_oracle_variants.py against it: at least one pin must fail. Nothing
here touches the real oracle or the GPU."""
import importlib.util
import os
import sys

import pytest

import test_oracle_variants as P

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "variants.py")

MUTANTS = {
    "bias 2^(r-1)": ("return (1 << (self.residual_bits - 1)) - 1 if self.bias else 0",
                     "return (1 << (self.residual_bits - 1)) if self.bias else 0"),
    "q_max off by one": ("return (1 << (self.anchor_bits + self.residual_bits - 2)) - 1",
                         "return (1 << (self.anchor_bits + self.residual_bits - 2))"),
    "linear threshold offset": ("            t = (k - 0.5) / qm\n", "            t = (k - 0.4) / qm\n"),
    "level exponent": ("t = (math.pow(1.0 + v.alpha, k / qm) - 1.0) / v.alpha",
                       "t = (math.pow(1.0 + v.alpha, k / (qm + 1)) - 1.0) / v.alpha"),
    "mean divisor": ("mean = (slots[:, :, 0] / f32(C)).astype(f32)", "mean = (slots[:, :, 0] / f32(C - 1)).astype(f32)"),
    "scale rounded to nearest": ("s_h = _f16_round_up(s.astype(f32))", "s_h = s.astype(f32).astype(np.float16)"),
    "sign-aware rule dropped": ("qn = np.maximum(q, 1) if v.sign_aware else q", "qn = q"),
    "no-isolation scale": ("w = ((uc - f32(0.5)) * f32(2.0)).astype(f32)", "w = ((uc - f32(0.5)) * f32(1.0)).astype(f32)"),
    "uniform rounds down": ("code = np.floor((t + f32(0.5)).astype(f32))", "code = np.floor(t)"),
    "anchor decode off centre": ("xa = _decode(mn, rng, mu_b, s_b, A << v.residual_bits, v)",
                                 "xa = _decode(mn, rng, mu_b, s_b, (A << v.residual_bits) + 1, v)"),
    "page minimum dropped": ("u = ((x - mn[:, None, :]) * inv[:, None, :]).astype(f32)",
                             "u = (x * inv[:, None, :]).astype(f32)"),
    "attention head group": ("        g = h // G\n", "        g = h % H\n"),
    "attention scale dropped": ("s = sm_scale * (q[:, h, :] @ K[g].T)", "s = (q[:, h, :] @ K[g].T)"),
    "attention normaliser": ("/ p.sum(axis=1, keepdims=True)", "/ T"),
    "attention vnmse denominator": ("return float((e * e).sum() / (o * o).sum())",
                                    "return float((e * e).sum() / np.abs(o).sum())"),
}


def _load(name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not found: {name}"
    spec = importlib.util.spec_from_loader(f"variants_mut_{abs(hash(name))}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod          # dataclasses resolve the module by name
    exec(compile(text.replace(old, new), SRC, "exec"), mod.__dict__)
    return mod


def _pins(orc, xb):
    return [
        lambda: P.test_split_identities_every_code(4, 4, True),
        lambda: P.test_split_identities_every_code(6, 2, True),
        lambda: P.test_sign_aware_mapping(),
        lambda: P.test_linear_map_is_the_round_half_up_grid(),
        lambda: P.test_alpha_law_levels_grow_geometrically(255.0),
        lambda: P.test_default_matches_main_oracle(orc, xb),
        lambda: P.test_no_chunk_isolation_reading(xb),
        lambda: P.test_chunk_statistics_against_fp64(xb, 16),
        lambda: P.test_uniform_comparator_half_step(xb, 4),
        lambda: P.test_six_bit_split_range(xb),
        lambda: P.test_dense_attention_equals_paged_decode_over_the_reconstruction(orc, xb),
        lambda: P.test_dense_attention_brute_force_with_head_groups(),
        lambda: P.test_dense_attention_special_cases(),
        lambda: P.test_attention_vnmse_closed_forms(),
    ]


@pytest.fixture(scope="module")
def xb():
    import lynx_synth as S
    w = S.WORKLOADS[2]                   # the same input as the pins' own fixture
    return S.laplace_bf16(w.key(S.S_K), w.scales(S.S_K)[:1, :2], 1, 2, 512).reshape(2, 512, 128)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(orc, xb, name, monkeypatch):
    old, new = MUTANTS[name]
    monkeypatch.setattr(P, "V", _load(name, old, new))
    caught = False
    for pin in _pins(orc, xb):
        try:
            pin()
        except Exception:                 # an assertion, or a crash the mistake causes
            caught = True
            break
    assert caught, f"no pin caught the mutant: {name}"


def test_unmutated_copy_passes(orc, xb, monkeypatch):
    text = open(SRC).read()
    monkeypatch.setattr(P, "V", _load("none", text[:40], text[:40]))
    for pin in _pins(orc, xb):
        pin()
