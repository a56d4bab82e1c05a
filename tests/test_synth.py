"""The seeded input generator: determinism, published SplitMix64 values,
distribution shape and outlier channel counts of each workload recipe."""
import numpy as np

import lynx_synth as S


def test_splitmix64_reference_values():
    # first outputs of SplitMix64 seeded with 0 (state advanced by the golden gamma)
    z, outs = 0, []
    for _ in range(3):
        outs.append(S.splitmix64_int(z))
        z = (z + S.GAMMA) & S.M64
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    arr = S.splitmix64(np.array([0, S.GAMMA, (2 * S.GAMMA) & S.M64], np.uint64))
    assert [int(v) for v in arr] == outs


def test_laplace_shape_and_determinism():
    sc = np.ones((1, 1, 128), np.float32)
    a = S.laplace_bf16(S.key(5, 1), sc, 1, 1, 4096)
    b = S.laplace_bf16(S.key(5, 1), sc, 1, 1, 4096)
    assert np.array_equal(a, b)
    x = S.bf16_bits_to_f32(a).astype(np.float64).ravel()
    assert abs(x.mean()) < 0.01
    assert abs(np.abs(x).mean() - 1.0) < 0.01          # E|X| = b = 1
    assert abs(x.var() - 2.0) < 0.05                    # Var = 2 b^2
    # sub-block generation agrees with slicing the full block
    c = S.laplace_bf16(S.key(5, 1), sc, 1, 1, 4096, t0=1000, t1=1100)
    assert np.array_equal(c[0, 0], a[0, 0, 1000:1100])


def test_outlier_channel_counts():
    for i, w in S.WORKLOADS.items():
        if w.L * w.H > 4096:
            continue
        s = w.scales(S.S_K)
        big = (s >= 9.99).sum(axis=-1) if w.base_log10 is None else (s >= 0.99 * 100 * 0.01).sum(-1)
        if w.base_log10 is None:
            assert np.all(big == w.n_outliers), i
    assert S.WORKLOADS[2].n_outliers == 4 and S.WORKLOADS[3].n_outliers == 3


def test_batched_layout_is_a_partition():
    w = S.WORKLOADS[4]
    ctx, pool, table = S.batched_layout(w)
    assert ctx.min() >= 4096 and ctx.max() <= 16384 and len(ctx) == 32
    used = np.concatenate([table[b, :(c + 255) // 256] for b, c in enumerate(ctx)])
    assert np.array_equal(np.sort(used), np.arange(pool))
    assert np.any(ctx % 256 != 0)                         # ragged last pages occur
