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
