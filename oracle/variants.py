"""Plain CPU oracle of the Lynx quantizer's variants and ablations (test
infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; it shares no code with the CUDA
library and imports nothing from it).

What it computes. "Lynx: the KV cache does not have to arrive whole"
(aigenapps reading of Han et al.), section 3 "The quantizer" fixes one
configuration: page normalisation, chunk isolation with C = 32, an alpha-law
map onto 2^7 - 1 = 127 levels with a sign-aware mapping, a +7 round-half-down
bias and a 4 + 4 bit cut. Section 7 "What the paper does not establish" names
what was never measured: other splits (INT6 and INT2 splits are future work),
a chunk-size sweep (the claim that smaller chunks reduce error), and a
stage-by-stage ablation (the bundle is worth 35x in vNMSE over uniform INT4,
but which stage earned it is unknown). This module encodes one page at a time
with every one of those knobs, plus the uniform comparator, and returns the
codes, the metadata and the squared errors of the anchor-only and the full
reconstruction.

Readings (where the pages leave a step open):
- a split (a, r) gives codes with 2^(a+r-1) - 1 levels (q_max = 2^(a+r-2) - 1
  per sign: 4 + 4 gives the page's 127); the bias is 2^(r-1) - 1 (the page's
  +7 at r = 4); anchor-only decoding takes the code 2^r A (the residual at its
  centre);
- no page normalisation: u = x (metadata min 0, range 1);
- no chunk isolation: the page's own centre, w = 2u - 1 (metadata mean 1/2,
  scale 1/2, so the decoder's formula is unchanged);
- no log map: the alpha -> 0 limit of the alpha-law map, a linear grid
  (thresholds (k - 1/2)/q_max, levels k/q_max);
- no bias: the cut is a plain floor (the residual is one-sided, which is what
  the page says the bias avoids), anchor-only decoding still takes 2^r A;
- no sign-aware mapping: c = -q for w < 0 (small negatives collapse to 0);
- uniform INTb comparator: per (page, channel) min and range (or per token,
  over its 128 channels), 2^b levels, code = floor((x - mn) * ((2^b - 1) /
  rng) + 1/2) with every step in fp32 (the integer decision is taken in the
  precision the GPU takes it), decoded in fp64;
- vNMSE: sum (x_hat - x)^2 / sum x^2 over the tensor; the section 5 figures
  are the vNMSE of the attention output, so ``dense_attn`` runs one decode
  step over a dense cache (the original values or a reconstruction) and
  ``attn_vnmse`` takes the same ratio over the outputs [batch, heads, 128].

The encoder follows the same numeric contract as the main oracle: fp32 with
round-to-nearest and no fused multiply-add, a stride-halving tree for the
chunk sum, fp16 chunk mean rounded to nearest and fp16 chunk scale rounded
up, a threshold count for the level. numpy float32 arithmetic is IEEE
round-to-nearest and never fused, so the arrays below carry it out as written.
Tables come from libm's pow in fp64 (math.pow), as the main oracle's do.

Parity status: every function is pinned by ``tests/test_oracle_variants.py``
(the default configuration against the main oracle's codes and metadata,
closed forms for the linear map, the split identities, brute force on tiny
inputs); none is "parity unpinned".
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

PAGE = 256
D = 128


@dataclass(frozen=True)
class Variant:
    """One configuration of the quantizer (defaults: the page's own)."""
    chunk: int = 32                 # C, tokens per chunk (16, 32 or 64)
    anchor_bits: int = 4            # a
    residual_bits: int = 4          # r
    alpha: float = 255.0            # alpha-law parameter; 0 selects the linear map
    page_norm: bool = True
    chunk_isolation: bool = True
    bias: bool = True
    sign_aware: bool = True
    uniform_bits: int = 0           # > 0: the uniform INTb comparator instead of the method
    uniform_per_token: bool = False # comparator grid per token (over its 128 channels), not per (page, channel)

    @property
    def qmax(self) -> int:
        return (1 << (self.anchor_bits + self.residual_bits - 2)) - 1

    @property
    def bias_value(self) -> int:
        return (1 << (self.residual_bits - 1)) - 1 if self.bias else 0


def thresholds(v: Variant) -> np.ndarray:
    """thr[k], k = 0..q_max, fp32 (thr[0] = 0): where the map crosses k - 1/2
    (section 3, "Non-linear transform"; rounding half up in the map's domain)."""
    qm = v.qmax
    thr = np.zeros(qm + 1, np.float32)
    for k in range(1, qm + 1):
        if v.alpha > 0:
            t = (math.pow(1.0 + v.alpha, (k - 0.5) / qm) - 1.0) / v.alpha
        else:
            t = (k - 0.5) / qm
        thr[k] = np.float32(t)
    return thr


def levels(v: Variant) -> np.ndarray:
    """Lv[k], k = 0..q_max + 1, the fp16-exact level values as float64 (the
    magnitude an anchor-only code 2^r A can reach is q_max + 1)."""
    qm = v.qmax
    out = np.zeros(qm + 2, np.float64)
    for k in range(qm + 2):
        if v.alpha > 0:
            t = (math.pow(1.0 + v.alpha, k / qm) - 1.0) / v.alpha
        else:
            t = k / qm
        out[k] = float(np.float16(t))
    return out


def _bf16_to_f32(x_bf16) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    return (x.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _f16_round_up(s: np.ndarray) -> np.ndarray:
    """fp16 of fp32 values rounded toward +infinity: nearest, then one step up
    where the nearest fell below."""
    h = s.astype(np.float16)
    low = h.astype(np.float32) < s
    return np.where(low, np.nextafter(h, np.float16(np.inf)), h)


def _stage1(x: np.ndarray, v: Variant):
    """Page normalisation per channel (section 3, "Page-level normalisation"):
    mn, rng, u = (x - mn) / rng in fp32. x: [P, 256, 128] float32."""
    f32 = np.float32
    if not v.page_norm:
        P = x.shape[0]
        return np.zeros((P, D), f32), np.ones((P, D), f32), x.copy()
    nan = np.isnan(x)
    mn = np.where(nan, f32(np.inf), x).min(axis=1) + f32(0.0)
    mx = np.where(nan, f32(-np.inf), x).max(axis=1) + f32(0.0)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        rng = (mx - mn).astype(f32)
        has_nan = nan.any(axis=1)
        mn = np.where(has_nan, f32(np.nan), mn)
        rng = np.where(has_nan | np.isnan(rng), f32(np.nan), rng)
        inv = np.where(rng > 0, f32(1.0) / np.where(rng > 0, rng, f32(1.0)), f32(0.0)).astype(f32)
        degenerate = ~(rng <= np.finfo(f32).max) | ~(inv <= np.finfo(f32).max)
        u = ((x - mn[:, None, :]) * inv[:, None, :]).astype(f32)
    u = np.where(degenerate[:, None, :], f32(0.0), u)
    return mn.astype(f32), rng.astype(f32), u


def _stage2(u: np.ndarray, v: Variant):
    """Chunk isolation (section 3, "Chunk-wise outlier isolation"): per C-token
    chunk, centre by the fp16 mean, divide by the fp16 max-abs rounded up.
    Returns (w [P, 256, 128] f32, mu bits, s bits [P, 256/C, 128] uint16)."""
    f32 = np.float32
    P = u.shape[0]
    C = v.chunk
    nch = PAGE // C
    uc = u.reshape(P, nch, C, D)
    if not v.chunk_isolation:
        half = np.float16(0.5)
        mu_h = np.full((P, nch, D), half, np.float16)
        s_h = np.full((P, nch, D), half, np.float16)
        w = ((uc - f32(0.5)) * f32(2.0)).astype(f32)
        return w.reshape(P, PAGE, D), mu_h.view(np.uint16), s_h.view(np.uint16)
    slots = uc.copy()
    h = C // 2
    while h >= 1:                                   # stride-halving tree
        slots[:, :, :h] = slots[:, :, :h] + slots[:, :, h:2 * h]
        h //= 2
    mean = (slots[:, :, 0] / f32(C)).astype(f32)
    mu_h = mean.astype(np.float16)
    vv = (uc - mu_h.astype(f32)[:, :, None, :]).astype(f32)
    s = np.where(np.isnan(vv), f32(0.0), np.abs(vv)).max(axis=2)
    s_h = _f16_round_up(s.astype(f32))
    sf = s_h.astype(f32)
    inv_s = np.where(sf > 0, f32(1.0) / np.where(sf > 0, sf, f32(1.0)), f32(0.0)).astype(f32)
    w = (vv * inv_s[:, :, None, :]).astype(f32)
    return w.reshape(P, PAGE, D), mu_h.view(np.uint16), s_h.view(np.uint16)


def _stage3(w: np.ndarray, v: Variant) -> np.ndarray:
    """Level count and sign-aware code (section 3, "Non-linear transform" and
    "Two details that look small"): q = #{k : |w| >= T_k}; c = q for w >= 0,
    -max(q, 1) (sign-aware) or -q for w < 0."""
    thr = thresholds(v)
    aw = np.abs(w)
    q = np.searchsorted(thr[1:], aw, side="right").astype(np.int32)
    q = np.where(np.isnan(aw), 0, q)
    neg = w < 0
    qn = np.maximum(q, 1) if v.sign_aware else q
    return np.where(neg, -qn, q).astype(np.int32)


def split(c: np.ndarray, v: Variant):
    """Bias and cut (section 3, "The cut"): b = c + bias, anchor A = floor(b / 2^r),
    residual r = b - 2^r A in [0, 2^r)."""
    b = np.asarray(c, dtype=np.int64) + v.bias_value
    A = np.floor_divide(b, 1 << v.residual_bits)
    return A.astype(np.int32), (b - (A << v.residual_bits)).astype(np.int32)


def _decode(mn, rng, mu_bits, s_bits, c, v: Variant) -> np.ndarray:
    """x_hat = mn + rng (mu + s sgn(c) Lv[|c|]) in fp64 (the main decoder's form)."""
    lv = levels(v)
    P = c.shape[0]
    nch = PAGE // v.chunk
    mu = mu_bits.view(np.float16).astype(np.float64)
    s = s_bits.view(np.float16).astype(np.float64)
    k = np.minimum(np.abs(c), v.qmax + 1)
    val = (mu[:, :, None, :] + s[:, :, None, :] * np.sign(c).reshape(P, nch, v.chunk, D)
           * lv[k].reshape(P, nch, v.chunk, D))
    return mn.astype(np.float64)[:, None, :] + rng.astype(np.float64)[:, None, :] * val.reshape(P, PAGE, D)


def _uniform(x: np.ndarray, v: Variant):
    """The uniform comparator: min-max grid of 2^b levels per (page, channel),
    or per token. Returns (mn, rng) of shape [P, 128] per (page, channel), or
    [P, 256, 1] per token."""
    f32 = np.float32
    if v.uniform_per_token:
        mn, rng, _ = _stage1(np.swapaxes(x, 1, 2), Variant())        # tokens as channels
        mn, rng = mn[:, :, None], rng[:, :, None]
    else:
        mn, rng, _ = _stage1(x, Variant())
        mn, rng = mn[:, None, :], rng[:, None, :]
    top = f32((1 << v.uniform_bits) - 1)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv_step = np.where(rng > 0, top / np.where(rng > 0, rng, f32(1.0)), f32(0.0)).astype(f32)
        t = ((x - mn) * inv_step).astype(f32)
        code = np.floor((t + f32(0.5)).astype(f32))
    code = np.clip(np.nan_to_num(code, nan=0.0), 0, float(top)).astype(np.int32)
    step = rng.astype(np.float64) / float(top)
    xh = mn.astype(np.float64) + code * step
    return mn, rng, code, xh


def encode(x_bf16, v: Variant = Variant()) -> dict:
    """Encode a [N, T, 128] bf16 tensor (uint16 bits; T a multiple of 256)
    page by page. Returns codes c [N, T, 128] int32 (uniform: grid codes),
    anchor A and residual r (method only), page_meta [N, P, 2, 128] f32,
    chunk_meta [N, P, 256/C, 2, 128] uint16 (method only), the anchor-only and
    full reconstructions [N, T, 128] float64 and err [N, P, 3] float64
    (sum x^2, sum (x_anchor - x)^2, sum (x_full - x)^2 per page)."""
    x = _bf16_to_f32(x_bf16)
    N, T, d = x.shape
    assert d == D and T % PAGE == 0
    P = T // PAGE
    xp = x.reshape(N * P, PAGE, D)
    out = {}
    if v.uniform_bits:
        mn, rng, code, xh = _uniform(xp, v)
        out["codes"] = code.reshape(N, T, D)
        xa = xf = xh
        if v.uniform_per_token:                     # no per-(page, channel) metadata
            mn, rng = np.zeros((N * P, D), np.float32), np.zeros((N * P, D), np.float32)
        else:
            mn, rng = mn[:, 0, :], rng[:, 0, :]
    else:
        assert v.chunk in (16, 32, 64) and 1 <= v.residual_bits <= 4 and 1 <= v.anchor_bits <= 6
        assert v.anchor_bits + v.residual_bits <= 8
        mn, rng, u = _stage1(xp, v)
        w, mu_b, s_b = _stage2(u, v)
        c = _stage3(w, v)
        A, r = split(c, v)
        out["codes"] = c.reshape(N, T, D)
        out["anchor"] = A.reshape(N, T, D)
        out["residual"] = r.reshape(N, T, D)
        out["chunk_meta"] = np.stack([mu_b, s_b], axis=2).reshape(N, P, PAGE // v.chunk, 2, D)
        xa = _decode(mn, rng, mu_b, s_b, A << v.residual_bits, v)
        xf = _decode(mn, rng, mu_b, s_b, c, v)
    out["page_meta"] = np.stack([mn, rng], axis=1).reshape(N, P, 2, D)
    x64 = xp.astype(np.float64)
    err = np.stack([(x64 * x64).sum(axis=(1, 2)), ((xa - x64) ** 2).sum(axis=(1, 2)),
                    ((xf - x64) ** 2).sum(axis=(1, 2))], axis=1)
    out["err"] = err.reshape(N, P, 3)
    out["x_anchor"] = xa.reshape(N, T, D)
    out["x_full"] = xf.reshape(N, T, D)
    return out


def vnmse(err: np.ndarray) -> tuple[float, float]:
    """(anchor-only, full) vNMSE of a tensor from its per-page error sums."""
    e = np.asarray(err, dtype=np.float64).reshape(-1, 3).sum(axis=0)
    return float(e[1] / e[0]), float(e[2] / e[0])


def dense_attn(q_bf16, k, v, sm_scale: float) -> np.ndarray:
    """fp64 decode attention of one query per (request, query head) over a
    dense cache shared by every request: q [B, Hq, 128] bf16 bits, k and v
    [H, T, 128] real values. out[b, h] = softmax(sm_scale K_g q) V_g with
    g = h // (Hq / H), the textbook definition (max subtracted before exp)."""
    q = _bf16_to_f32(q_bf16).astype(np.float64)
    B, Hq, d = q.shape
    K = np.asarray(k, dtype=np.float64)
    Vv = np.asarray(v, dtype=np.float64)
    H, T, _ = K.shape
    assert d == D and Hq % H == 0 and T > 0
    G = Hq // H
    out = np.empty((B, Hq, D), np.float64)
    for h in range(Hq):
        g = h // G
        s = sm_scale * (q[:, h, :] @ K[g].T)              # [B, T]
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h, :] = (p @ Vv[g]) / p.sum(axis=1, keepdims=True)
    return out


def attn_vnmse(out_hat, out_ref) -> float:
    """vNMSE of an attention output against the reference output."""
    o = np.asarray(out_ref, dtype=np.float64)
    e = np.asarray(out_hat, dtype=np.float64) - o
    return float((e * e).sum() / (o * o).sum())
