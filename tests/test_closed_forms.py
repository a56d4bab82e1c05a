"""Numbers the Lynx reading prints, checked against the workload definitions and
the oracle's comparator (tests/golden/page_facts.json holds them with sections)."""
import json
import math
import os

import numpy as np

import lynx_synth as S

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_worked_example_cache_size_is_23_5_gib():
    f = FACTS["worked_example"]
    w = S.WORKLOADS[3]
    assert (w.L, w.H, w.T, S.D) == (f["layers"], f["kv_heads"], f["context_tokens"], f["head_dim"])
    size = w.elements * f["bytes_per_value"]
    assert size == 25_232_932_864
    assert size / 2 ** 30 == f["stated_size_gb"]           # the page's "GB" is GiB
    t100 = size * 8 / 100e9
    t400 = size * 8 / 400e9
    assert abs(t100 - f["stated_transfer_s_at_100gbps"]) < 0.05    # roughly two seconds
    assert t400 > f["stated_lower_bound_s_at_400gbps"]             # more than half a second


def test_effective_bins_of_a_linear_grid_under_an_outlier(orc):
    """2^B * m_i / m: a channel 100x smaller than the one setting a shared 8-bit
    grid sees about 2.56 bins (log2 = 1.36 bits; the page rounds to ~1.5)."""
    f = FACTS["effective_bins"]
    n = 4096
    u = S.uniform01(3, 99, 2 * n)
    big = (u[:n] * 2 - 1) * f["outlier_ratio"]
    small = u[n:] * 2 - 1
    x = np.stack([big, small], 1).astype(np.float32)
    x[0] = [-f["outlier_ratio"], 0]
    x[1] = [f["outlier_ratio"], 0]
    xb = S.f32_to_bf16_bits(x)
    codes, _ = orc.uniform(xb, f["bits"], axis=None)
    used = len(np.unique(codes[:, 1]))
    expected = 2 ** f["bits"] * 2 / (2 * f["outlier_ratio"])
    assert abs(expected - 2.56) < 1e-12
    # a range of e grid steps touches ceil(e) or ceil(e) + 1 round-to-nearest bins
    assert used in (math.ceil(expected), math.ceil(expected) + 1)
    step = (2.0 * f["outlier_ratio"]) / (2 ** f["bits"] - 1)
    span = S.bf16_bits_to_f32(xb[:, 1]).max() - S.bf16_bits_to_f32(xb[:, 1]).min()
    assert abs(span / step - expected) < 0.05
    assert abs(math.log2(expected) - f["stated_effective_bits"]) < 0.2


def test_structural_constants(orc):
    q = FACTS["quantizer"]
    assert 2 ** 7 - 1 == q["levels"]
    w = np.linspace(-1, 1, 100001, dtype=np.float32)
    assert len(np.unique(orc.codes(w))) == q["levels"]
    A, r = orc.split(np.arange(-63, 64, dtype=np.int8))
    assert int(A.max() - A.min()) < 2 ** q["anchor_bits"]
    assert int(r.max()) < 2 ** q["residual_bits"]
    assert orc.PAGE == q["page_tokens"] and orc.CHUNK == q["chunk_tokens"]
