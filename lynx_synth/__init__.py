"""Seeded synthetic KV inputs, shared by the CUDA path's tests/bench and the oracle.

This module holds none of the quantizer's arithmetic. It turns a counter-based
hash into bf16 values drawn from a Laplace law with per-channel scales and a
few outlier channels, the data shape the Lynx reading describes ("Not all bits
are equal": a few channels up to 100x larger, the rest Laplacian-like).

Generator (identical on the host, here, and on the GPU, ``synth.cu``):
  splitmix64(z)    Vigna's SplitMix64 finaliser (public domain definition)
  key(seed, s)     splitmix64(splitmix64(seed) ^ s)          one key per stream
  bits(i)          splitmix64(key + i)                        i = linear index
  magnitude        E[(bits >> 47) & 0xFFFF], E[k] = fp32(-ln(1 - (k + 1/2)/65536))
                   (the Exp(1) quantile at the bucket centre)
  sign             bit 63
  value            bf16_rn(fp32(sign * magnitude) * scale[channel])
Only integer operations, one table lookup and one fp32 multiply are involved,
so both implementations give the same bytes.

Index conventions: a tensor is [L, H, T, 128]; i = ((l*H + h)*T + t)*128 + d;
scales are [L, H, 128].
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

D = 128
PAGE = 256

# stream ids
S_K, S_V, S_Q = 1, 2, 3
S_SCALE, S_OUTLIER_RANK, S_OUTLIER_FACTOR = 10, 11, 12
S_CTX, S_PERM, S_ORDER = 20, 21, 22


def splitmix64_int(z: int) -> int:
    z = (z + GAMMA) & M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def splitmix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def key(seed: int, stream: int) -> int:
    return splitmix64_int(splitmix64_int(seed & M64) ^ (stream & M64))


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n doubles in [0, 1) from the counter hash (53 high bits)."""
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        h = splitmix64(np.uint64(key(seed, stream)) + idx)
    return (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_EXP_TABLE = None


def exp_table() -> np.ndarray:
    """65536 fp32 Exp(1) quantiles at bucket centres."""
    global _EXP_TABLE
    if _EXP_TABLE is None:
        k = np.arange(65536, dtype=np.float64)
        _EXP_TABLE = (-np.log1p(-(k + 0.5) / 65536.0)).astype(np.float32)
    return _EXP_TABLE


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 to bf16 (nearest-even), returned as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def laplace_bf16(k: int, scales: np.ndarray, L: int, H: int, T: int,
                 layers=None, heads=None, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """bf16 bits of x[l, h, t0:t1, :] for the listed layers/heads of a [L,H,T,128] tensor."""
    layers = range(L) if layers is None else list(layers)
    heads = range(H) if heads is None else list(heads)
    t1 = T if t1 is None else t1
    table = exp_table()
    out = np.empty((len(layers), len(heads), t1 - t0, D), np.uint16)
    tt = np.arange(t0, t1, dtype=np.uint64)[:, None]
    dd = np.arange(D, dtype=np.uint64)[None, :]
    for a, l in enumerate(layers):
        for b, h in enumerate(heads):
            base = np.uint64(((l * H + h) * T) * D)
            with np.errstate(over="ignore"):
                bits = splitmix64(np.uint64(k) + base + tt * np.uint64(D) + dd)
            mag = table[((bits >> np.uint64(47)) & np.uint64(0xFFFF)).astype(np.int64)]
            neg = (bits >> np.uint64(63)).astype(bool)
            val = np.where(neg, -mag, mag).astype(np.float32)
            val = (val * scales[l, h][None, :].astype(np.float32)).astype(np.float32)
            out[a, b] = f32_to_bf16_bits(val)
    return out


def channel_scales(seed: int, tensor_stream: int, L: int, H: int, *, base_log10=None,
                   n_outliers: int = 0, factor_log10=(2.0, 2.0)) -> np.ndarray:
    """[L,H,128] fp32 per-channel scales: a base (1, or 10^U(lo,hi)) times an
    outlier factor 10^U(f_lo, f_hi) on exactly n_outliers channels per (l, h),
    chosen without replacement by ranking channels on a hash."""
    n = L * H * D
    s = np.ones(n, np.float64)
    if base_log10 is not None:
        lo, hi = base_log10
        s *= 10.0 ** (lo + (hi - lo) * uniform01(seed, tensor_stream * 100 + S_SCALE, n))
    s = s.reshape(L, H, D)
    if n_outliers:
        rank = uniform01(seed, tensor_stream * 100 + S_OUTLIER_RANK, n).reshape(L, H, D)
        fac = uniform01(seed, tensor_stream * 100 + S_OUTLIER_FACTOR, n).reshape(L, H, D)
        flo, fhi = factor_log10
        pick = np.argsort(rank, axis=-1, kind="stable")[..., :n_outliers]
        f = 10.0 ** (flo + (fhi - flo) * fac)
        mask = np.zeros((L, H, D), bool)
        np.put_along_axis(mask, pick, True, axis=-1)
        s = np.where(mask, s * f, s)
    return s.astype(np.float32)


# ---------------------------------------------------------------------------
# workloads (shapes and recipes of the five synthetic configurations)
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    seed: int
    L: int
    H: int
    T: int
    Hq: int = 0
    B: int = 0
    base_log10: tuple | None = None
    outlier_frac: float = 0.0
    n_outliers_fixed: int | None = None
    factor_log10: tuple = (2.0, 2.0)
    ctx_range: tuple | None = None      # seeded uniform context lengths
    shared_context: bool = False        # every request's page table aliases one context
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_outliers(self) -> int:
        if self.n_outliers_fixed is not None:
            return self.n_outliers_fixed
        return int(math.floor(self.outlier_frac * D + 0.5))

    @property
    def pages(self) -> int:
        return self.T // PAGE

    @property
    def elements(self) -> int:
        """K + V elements of the whole cache."""
        return 2 * self.L * self.H * self.T * D

    def scales(self, tensor_stream: int) -> np.ndarray:
        return channel_scales(self.seed, tensor_stream, self.L, self.H, base_log10=self.base_log10,
                              n_outliers=self.n_outliers, factor_log10=self.factor_log10)

    def key(self, tensor_stream: int) -> int:
        return key(self.seed, tensor_stream)

    def queries_bf16(self, B: int | None = None, Hq: int | None = None, step: int = 0) -> np.ndarray:
        B = self.B if B is None else B
        Hq = self.Hq if Hq is None else Hq
        ones = np.ones((1, B * Hq, D), np.float32)
        q = laplace_bf16(key(self.seed, S_Q * 1000 + step), ones, 1, B * Hq, 1)
        return q.reshape(B, Hq, D)

    def ctx_lens(self) -> np.ndarray:
        if self.ctx_range is None:
            return np.full(self.B, self.T, np.int32)
        lo, hi = self.ctx_range
        u = uniform01(self.seed, S_CTX, self.B)
        return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


WORKLOADS = {
    1: Workload("one_page", 1001, L=1, H=1, T=256, Hq=1, B=1, n_outliers_fixed=4,
                factor_log10=(2.0, 2.0),
                notes="one page, Laplace(0,1), 4 outlier channels x100, one query"),
    2: Workload("qwen3_235b_like_layer_32k", 1002, L=1, H=4, T=32768, Hq=64, B=1,
                outlier_frac=0.03, factor_log10=(1.0, 2.0),
                notes="4 KV heads, 32K tokens, 3% outlier channels x10^U(1,2), 64 q heads"),
    3: Workload("full_cache_94L_128k", 1003, L=94, H=4, T=131072, Hq=64, B=1,
                base_log10=(-2.0, 0.0), outlier_frac=0.02, factor_log10=(2.0, 2.0),
                notes="94 layers x 4 KV heads x 128K tokens, channel scales 10^U(-2,0), "
                      "2% outlier channels x100"),
    4: Workload("batched_decode_32req", 1004, L=1, H=8, T=0, Hq=64, B=32,
                outlier_frac=0.03, factor_log10=(1.0, 2.0), ctx_range=(4096, 16384),
                notes="32 requests, ctx U[4K,16K], 8 KV heads, 64 q heads, permuted pages"),
    5: Workload("progressive_arrival_8L_64k", 1005, L=8, H=8, T=65536, Hq=64, B=8,
                outlier_frac=0.03, factor_log10=(1.0, 2.0), shared_context=True,
                notes="8 layers x 8 KV heads x 64K, residual layers arrive in seeded order, "
                      "8 requests share one context"),
}


def batched_layout(w: Workload):
    """Context lengths, the page pool size and a seeded random page table for a
    batched workload: request b owns ceil(ctx_b/256) physical pages drawn from a
    seeded permutation of the pool."""
    ctx = w.ctx_lens()
    need = [(int(c) + PAGE - 1) // PAGE for c in ctx]
    pool = int(sum(need))
    max_pages = max(need)
    perm = np.argsort(uniform01(w.seed, S_PERM, pool), kind="stable").astype(np.int32)
    table = np.zeros((w.B, max_pages), np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[o:o + n]
        o += n
    return ctx, pool, table


def arrival_order(w: Workload) -> np.ndarray:
    return np.argsort(uniform01(w.seed, S_ORDER, w.L), kind="stable").astype(np.int32)


# ---------------------------------------------------------------------------
# GPU implementation of the same generator (liblynx_synth.so)
# ---------------------------------------------------------------------------

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_LIB = os.path.join(_HERE, "liblynx_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                               "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise RuntimeError(f"{_LIB} is not built; run __graft_entry__.build()")
            lib = ctypes.CDLL(_LIB)
            lib.synth_fill_laplace_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                                    ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_int64, ctypes.c_void_p]
            lib.synth_fill_laplace_bf16.restype = ctypes.c_int
            _lib = lib
    return _lib


class DeviceGenerator:
    """Fills device tensors with the generator above (torch owns the memory)."""

    def __init__(self, device="cuda"):
        import torch
        self.torch = torch
        self.device = device
        self.table = torch.from_numpy(exp_table()).to(device)

    def fill(self, out, k: int, scales: np.ndarray, stream=None):
        """out: uint8/int16/bfloat16 device tensor viewed as [L,H,T,128]; scales [L,H,128]."""
        torch = self.torch
        L, H = scales.shape[0], scales.shape[1]
        n = out.numel() if out.element_size() == 2 else out.numel() // 2
        T = n // (L * H * D)
        assert L * H * T * D == n
        sc = torch.from_numpy(np.ascontiguousarray(scales, np.float32)).to(self.device)
        st = stream if stream is not None else torch.cuda.current_stream()
        rc = _load().synth_fill_laplace_bf16(ctypes.c_void_p(out.data_ptr()), ctypes.c_uint64(k),
                                             ctypes.c_void_p(sc.data_ptr()),
                                             ctypes.c_void_p(self.table.data_ptr()),
                                             L * H, T, D, ctypes.c_void_p(st.cuda_stream))
        if rc:
            raise RuntimeError(f"synth_fill_laplace_bf16 failed ({rc})")
        st.synchronize()
        del sc
        return out
