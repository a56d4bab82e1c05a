"""Plain CPU oracle of the Lynx progressive KV quantizer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library
(``progressive_kv_cache_gb300``) and imports nothing from it; the CUDA path
never calls back into it.

The arithmetic lives in ``lynx_oracle.c`` (plain C, fp32 where the encoder's
numeric contract fixes fp32, fp64 for decoding and attention). This module
compiles it with gcc on first use and wraps it for numpy arrays.

Source of every step: "Lynx: the KV cache does not have to arrive whole"
(aigenapps reading of Han et al.), section 3 "The quantizer" (four stages and
the 4+4 cut) and section 4 "Speculation at the communication boundary"
(anchor-only draft cache, refinement to the full reconstruction). Decode
attention is the textbook softmax(q K^T) V over the reconstructed cache, in
fp64 ("KV-cache quantization" explainer, aicassindra, "Middle row").

Parity status of each function: every function here is pinned by tests under
``tests/test_oracle_*.py`` (closed forms, exhaustive enumeration, brute force
on tiny inputs, library routines); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lynx_oracle.c")
_LIB = os.path.join(_HERE, "liblynx_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE = 256
CHUNK = 32
D = 128
NCHUNK = PAGE // CHUNK


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, no FP contraction, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_f16_from_double.argtypes = [dbl, i32]
            lib.orc_f16_from_double.restype = ctypes.c_uint16
            lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_double.restype = dbl
            lib.orc_alpha.restype = dbl
            lib.orc_tables.argtypes = [P, P]
            lib.orc_codes.argtypes = [P, i64, P]
            lib.orc_split.argtypes = [P, i64, P, P]
            lib.orc_quantize.argtypes = [P, i32, i32, i32, P, P, P, P, P]
            lib.orc_quantize.restype = i32
            lib.orc_dequant.argtypes = [P, P, P, P, i32, i32, i32, i32, P]
            lib.orc_dequant.restype = i32
            lib.orc_decode_attn.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                            P, P, i32, dbl, i32, P, P]
            lib.orc_decode_attn.restype = i32
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().orc_num_threads()


def alpha() -> float:
    return _load().orc_alpha()


def f16_bits(x: float, round_up: bool = False) -> int:
    """binary16 bits of x, nearest-even or rounded toward +infinity."""
    return int(_load().orc_f16_from_double(float(x), 1 if round_up else 0))


def f16_value(bits: int) -> float:
    return float(_load().orc_f16_to_double(int(bits)))


def tables():
    """(thr[64] float32 with thr[0] = 0, lv[65] uint16 fp16 bits)."""
    thr = np.zeros(64, np.float32)
    lv = np.zeros(65, np.uint16)
    _load().orc_tables(_p(thr), _p(lv))
    return thr, lv


def level_values() -> np.ndarray:
    """Lv[0..64] as float64 (exact fp16 values)."""
    _, lv = tables()
    return lv.view(np.float16).astype(np.float64)


def codes(w) -> np.ndarray:
    """Sign-aware alpha-law code (-63..63) of each fp32 value w."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(w.shape, np.int8)
    _load().orc_codes(_p(w), w.size, _p(out))
    return out


def split(c) -> tuple[np.ndarray, np.ndarray]:
    """(+7 bias, 4-bit cut) of codes: anchor A in -4..4 and residual r in 0..15."""
    c = np.ascontiguousarray(c, dtype=np.int8)
    A = np.empty(c.shape, np.int8)
    r = np.empty(c.shape, np.uint8)
    _load().orc_split(_p(c), c.size, _p(A), _p(r))
    return A, r


class Quantized(dict):
    """anchor, residual: [L,H,T,64] u8; page_meta: [L,H,P,2,128] f32;
    chunk_meta: [L,H,P,8,2,128] u16 (fp16 bits)."""


def quantize(x_bf16, page_valid=None) -> Quantized:
    """Encode a [L,H,T,128] bf16 tensor (given as uint16 bits) page by page."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    L, H, T, d = x.shape
    assert d == D and T % PAGE == 0
    P = T // PAGE
    pv = None if page_valid is None else np.ascontiguousarray(page_valid, dtype=np.int32)
    assert pv is None or pv.shape == (P,)
    q = Quantized(
        anchor=np.empty((L, H, T, D // 2), np.uint8),
        residual=np.empty((L, H, T, D // 2), np.uint8),
        page_meta=np.empty((L, H, P, 2, D), np.float32),
        chunk_meta=np.empty((L, H, P, NCHUNK, 2, D), np.uint16),
    )
    rc = _load().orc_quantize(_p(x), L, H, T, _p(pv), _p(q["anchor"]), _p(q["residual"]),
                              _p(q["page_meta"]), _p(q["chunk_meta"]))
    if rc:
        raise ValueError("orc_quantize rejected its arguments")
    return q


def dequant(q: Quantized, full: bool) -> np.ndarray:
    """fp64 reconstruction: anchor-only (full=False) or anchor+residual."""
    a = q["anchor"]
    L, H, T, _ = a.shape
    out = np.empty((L, H, T, D), np.float64)
    rc = _load().orc_dequant(_p(a), _p(q["residual"]) if full else None, _p(q["page_meta"]),
                             _p(q["chunk_meta"]), L, H, T, 1 if full else 0, _p(out))
    if rc:
        raise ValueError("orc_dequant rejected its arguments")
    return out


def decode_attn(q_bf16, k: Quantized, v: Quantized, layer: int, page_table, ctx_lens,
                sm_scale: float, full: bool, want_scores: bool = False):
    """fp64 decode attention of one layer. Returns out [B,Hq,128] (and scores)."""
    qb = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    B, Hq, d = qb.shape
    assert d == D
    L, H, T, _ = k["anchor"].shape
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    max_pages = pt.shape[1]
    out = np.empty((B, Hq, D), np.float64)
    sc = np.empty((B, Hq, max_pages * PAGE), np.float64) if want_scores else None
    rc = _load().orc_decode_attn(
        _p(qb), B, Hq, _p(k["anchor"]), _p(k["residual"]), _p(k["page_meta"]), _p(k["chunk_meta"]),
        _p(v["anchor"]), _p(v["residual"]), _p(v["page_meta"]), _p(v["chunk_meta"]),
        L, H, T, layer, _p(pt), _p(cl), max_pages, float(sm_scale), 1 if full else 0,
        _p(out), _p(sc))
    if rc:
        raise ValueError("orc_decode_attn rejected its arguments")
    return (out, sc) if want_scores else out


def verify_attn(q_bf16, k: Quantized, v: Quantized, layer: int, page_table, ctx_lens, sm_scale: float,
                full: bool):
    """fp64 verify attention of one layer for a block of T_q draft positions
    per request, causal within the block (the Lynx reading, section 4: the
    drafted positions are checked against the refined cache). The last T_q
    tokens of each context are the drafted ones, so position i of request b is
    exactly one decode step over the first ctx_b - T_q + i + 1 tokens (none
    when that count is not positive). Returns out [B, T_q, Hq, 128]."""
    qb = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    B, Tq, Hq, d = qb.shape
    assert d == D
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    out = np.empty((B, Tq, Hq, D), np.float64)
    for i in range(Tq):
        n = np.maximum(cl - Tq + i + 1, 0).astype(np.int32)
        out[:, i] = decode_attn(qb[:, i], k, v, layer, page_table, n, sm_scale, full)
    return out


def uniform(x_bf16, bits: int, axis=None):
    """The plain linear grid that the Lynx reading argues against ("Not all bits
    are equal"): min/max over `axis` (None = the whole array, -1 = per token),
    2^bits levels, round half up. Returns (codes, fp64 reconstruction)."""
    x = (np.asarray(x_bf16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    x = x.astype(np.float64)
    mn = x.min(axis=axis, keepdims=axis is not None)
    mx = x.max(axis=axis, keepdims=axis is not None)
    step = (mx - mn) / (2.0 ** bits - 1.0)
    safe = np.where(step > 0, step, 1.0)
    c = np.where(step > 0, np.floor((x - mn) / safe + 0.5), 0.0)
    return c.astype(np.int64), mn + c * step
