"""Lynx progressive KV quantizer on GB300: Python binding of liblynx.so.

This module only marshals arguments: torch tensors are passed to the C ABI
(include/lynx.h) as raw device pointers together with the current CUDA stream.
Every step of the encoder, the decoders and the decode attention runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing the
module without a built library raises.

Method: "Lynx: the KV cache does not have to arrive whole" (aigenapps reading
of Han et al.), sections 3 ("The quantizer") and 4 ("Speculation at the
communication boundary").
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblynx.so")

PAGE = 256
CHUNK = 32
HEAD_DIM = 128
NCHUNK = PAGE // CHUNK

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = range(7)
OUT_BF16, OUT_F32 = 0, 1
MODE_ANCHOR, MODE_FULL = 0, 1
DEVERR_PAGE, DEVERR_CTX = 1, 2


class LynxError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().lynx_status_string(status).decode()} (status {status})")


class LynxQKV(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("tokens", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("anchor", ctypes.c_void_p), ("residual", ctypes.c_void_p),
                ("page_meta", ctypes.c_void_p), ("chunk_meta", ctypes.c_void_p)]


class LynxVariant(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int32), ("anchor_bits", ctypes.c_int32), ("residual_bits", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("flags", ctypes.c_uint32), ("uniform_bits", ctypes.c_int32)]


VAR_NO_PAGE_NORM, VAR_NO_CHUNK_ISOLATION, VAR_NO_BIAS, VAR_NO_SIGN_AWARE, VAR_UNIFORM_PER_TOKEN = 1, 2, 4, 8, 16

_lock = threading.Lock()
_L = None


def _lib():
    global _L
    with _lock:
        if _L is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m progressive_kv_cache_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.lynx_status_string.argtypes = [ctypes.c_int]
            L.lynx_status_string.restype = ctypes.c_char_p
            L.lynx_quantize_pages.argtypes = [vp, vp, ctypes.POINTER(LynxQKV), vp]
            L.lynx_quantize_append.argtypes = [vp, vp, vp, i32, ctypes.POINTER(LynxQKV), vp, vp]
            L.lynx_dequant_anchor.argtypes = [ctypes.POINTER(LynxQKV), vp, ctypes.c_int, vp]
            L.lynx_refine_residual.argtypes = [ctypes.POINTER(LynxQKV), vp, ctypes.c_int, vp]
            L.lynx_decode_attn_workspace.argtypes = [i32, i32, i32]
            L.lynx_decode_attn_workspace.restype = ctypes.c_size_t
            L.lynx_decode_attn.argtypes = [vp, ctypes.POINTER(LynxQKV), ctypes.POINTER(LynxQKV), i32, vp, vp,
                                           i32, i32, i32, ctypes.c_float, ctypes.c_int, vp, vp, vp,
                                           ctypes.c_size_t, vp, vp]
            L.lynx_decode_attn_noalloc.argtypes = [vp, ctypes.POINTER(LynxQKV), ctypes.POINTER(LynxQKV), i32,
                                                   vp, vp, i32, i32, i32, ctypes.c_float, ctypes.c_int, vp, vp,
                                                   vp, vp]
            L.lynx_decode_attn_noalloc.restype = ctypes.c_int
            L.lynx_verify_attn_workspace.argtypes = [i32, i32, i32, i32]
            L.lynx_verify_attn_workspace.restype = ctypes.c_size_t
            L.lynx_verify_attn.argtypes = [vp, ctypes.POINTER(LynxQKV), ctypes.POINTER(LynxQKV), i32, vp, vp, i32,
                                           i32, i32, i32, ctypes.c_float, ctypes.c_int, vp, vp, ctypes.c_size_t,
                                           vp, vp]
            L.lynx_host_tables.argtypes = [vp, vp]
            L.lynx_host_tables.restype = None
            L.lynx_level_codes.argtypes = [vp, i64, vp, vp]
            L.lynx_quantize_variant.argtypes = [vp, i32, i32, ctypes.POINTER(LynxVariant), vp, vp, vp, vp, vp, vp,
                                                vp, vp, vp]
            L.lynx_dense_attn.argtypes = [vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp, vp]
            for f in ("lynx_quantize_pages", "lynx_quantize_append", "lynx_dequant_anchor", "lynx_refine_residual",
                      "lynx_decode_attn", "lynx_verify_attn", "lynx_level_codes", "lynx_quantize_variant",
                      "lynx_dense_attn"):
                getattr(L, f).restype = ctypes.c_int
            _L = L
    return _L


def library():
    """The loaded ctypes handle of liblynx.so."""
    return _lib()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != OK:
        raise LynxError(status, what)


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class QuantizedKV:
    """Planes and metadata of one quantized tensor (K or V), owned by torch.

    anchor, residual: uint8 [L, H, T, 64]; page_meta: float32 [L, H, P, 2, 128];
    chunk_meta: int16 [L, H, P, 8, 2, 128] (fp16 bits)."""

    def __init__(self, anchor, residual, page_meta, chunk_meta):
        self.anchor, self.residual, self.page_meta, self.chunk_meta = anchor, residual, page_meta, chunk_meta

    @classmethod
    def empty(cls, layers, kv_heads, tokens, device="cuda", residual=True):
        if tokens % PAGE:
            raise ValueError("tokens must be a multiple of 256")
        P = tokens // PAGE
        dev = torch.device(device)
        return cls(torch.empty((layers, kv_heads, tokens, HEAD_DIM // 2), dtype=torch.uint8, device=dev),
                   torch.empty((layers, kv_heads, tokens, HEAD_DIM // 2), dtype=torch.uint8, device=dev)
                   if residual else None,
                   torch.empty((layers, kv_heads, P, 2, HEAD_DIM), dtype=torch.float32, device=dev),
                   torch.empty((layers, kv_heads, P, NCHUNK, 2, HEAD_DIM), dtype=torch.int16, device=dev))

    @property
    def shape(self):
        L, H, T, _ = self.anchor.shape
        return L, H, T

    def layers(self, l0, l1):
        """A view of layers [l0, l1) (shares memory)."""
        return QuantizedKV(self.anchor[l0:l1], None if self.residual is None else self.residual[l0:l1],
                           self.page_meta[l0:l1], self.chunk_meta[l0:l1])

    def without_residual(self):
        return QuantizedKV(self.anchor, None, self.page_meta, self.chunk_meta)

    def desc(self) -> LynxQKV:
        L, H, T = self.shape
        return LynxQKV(L, H, T, HEAD_DIM, self.anchor.data_ptr(),
                       None if self.residual is None else self.residual.data_ptr(),
                       self.page_meta.data_ptr(), self.chunk_meta.data_ptr())

    def nbytes(self):
        n = self.anchor.numel() + self.page_meta.numel() * 4 + self.chunk_meta.numel() * 2
        return n + (self.residual.numel() if self.residual is not None else 0)


def quantize_pages(x, out: QuantizedKV, page_valid=None, stream=None):
    """lynx_quantize_pages: encode bf16 x [L, H, T, 128] into `out`."""
    _dev(x, torch.bfloat16, "x")
    if page_valid is not None:
        _dev(page_valid, torch.int32, "page_valid")
    d = out.desc()
    _check(_lib().lynx_quantize_pages(_ptr(x), _ptr(page_valid), ctypes.byref(d), _stream(stream)),
           "lynx_quantize_pages")
    return out


def quantize_append(tail, phys_page, valid, out: QuantizedKV, dev_err=None, stream=None):
    """lynx_quantize_append: re-encode bf16 tails [n, L, H, 256, 128] into
    physical pages phys_page[n] of every layer and KV head of `out`."""
    _dev(tail, torch.bfloat16, "tail")
    _dev(phys_page, torch.int32, "phys_page")
    _dev(valid, torch.int32, "valid")
    if dev_err is not None:
        _dev(dev_err, torch.int32, "dev_err")
    n = phys_page.numel()
    L, H, _ = out.shape
    if valid.numel() != n or tuple(tail.shape) != (n, L, H, PAGE, HEAD_DIM):
        raise ValueError("tail must be [n, L, H, 256, 128] with n = len(phys_page) = len(valid)")
    d = out.desc()
    _check(_lib().lynx_quantize_append(_ptr(tail), _ptr(phys_page), _ptr(valid), n, ctypes.byref(d),
                                       _ptr(dev_err), _stream(stream)), "lynx_quantize_append")
    return out


def _dense_dtype(t):
    if t.dtype == torch.bfloat16:
        return OUT_BF16
    if t.dtype == torch.float32:
        return OUT_F32
    raise TypeError("dense cache must be bfloat16 or float32")


def dequant_anchor(q: QuantizedKV, out, stream=None):
    """lynx_dequant_anchor: anchor-only reconstruction into out [L, H, T, 128]."""
    if not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA tensor")
    d = q.desc()
    _check(_lib().lynx_dequant_anchor(ctypes.byref(d), _ptr(out), _dense_dtype(out), _stream(stream)),
           "lynx_dequant_anchor")
    return out


def refine_residual(q: QuantizedKV, inout, stream=None):
    """lynx_refine_residual: overwrite the dense cache with the full reconstruction."""
    if not inout.is_cuda or not inout.is_contiguous():
        raise ValueError("inout must be a contiguous CUDA tensor")
    d = q.desc()
    _check(_lib().lynx_refine_residual(ctypes.byref(d), _ptr(inout), _dense_dtype(inout), _stream(stream)),
           "lynx_refine_residual")
    return inout


def decode_attn_workspace(batch, q_heads, max_pages) -> int:
    return int(_lib().lynx_decode_attn_workspace(batch, q_heads, max_pages))


def decode_attn(q, k: QuantizedKV, v: QuantizedKV, layer, page_table, ctx_lens, sm_scale, mode,
                out=None, scores=None, workspace=None, dev_err=None, stream=None):
    """lynx_decode_attn: one decode step of attention over layer `layer`.

    q: bf16 [B, Hq, 128]; page_table: int32 [B, max_pages]; ctx_lens: int32 [B].
    Returns out (float32 [B, Hq, 128])."""
    _dev(q, torch.bfloat16, "q")
    _dev(page_table, torch.int32, "page_table")
    _dev(ctx_lens, torch.int32, "ctx_lens")
    B, Hq, _ = q.shape
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = decode_attn_workspace(B, Hq, max_pages)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    kd, vd = k.desc(), v.desc()
    _check(_lib().lynx_decode_attn(_ptr(q), ctypes.byref(kd), ctypes.byref(vd), layer, _ptr(page_table),
                                   _ptr(ctx_lens), B, Hq, max_pages, float(sm_scale), int(mode), _ptr(out),
                                   _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(dev_err), _stream(stream)),
           "lynx_decode_attn")
    return out


def verify_attn_workspace(batch, draft, q_heads, max_pages):
    return int(_lib().lynx_verify_attn_workspace(batch, draft, q_heads, max_pages))


def verify_attn(q, k: QuantizedKV, v: QuantizedKV, layer, page_table, ctx_lens, sm_scale, mode, out=None,
                workspace=None, dev_err=None, stream=None):
    """lynx_verify_attn: attention of a block of draft positions per request,
    causal within the block. q: bfloat16 [B, T_q, Hq, 128]; returns float32
    [B, T_q, Hq, 128]."""
    _dev(q, torch.bfloat16, "q")
    _dev(page_table, torch.int32, "page_table")
    _dev(ctx_lens, torch.int32, "ctx_lens")
    B, Tq, Hq, _ = q.shape
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty((B, Tq, Hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = verify_attn_workspace(B, Tq, Hq, max_pages)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    kd, vd = k.desc(), v.desc()
    _check(_lib().lynx_verify_attn(_ptr(q), ctypes.byref(kd), ctypes.byref(vd), layer, _ptr(page_table),
                                   _ptr(ctx_lens), B, Tq, Hq, max_pages, float(sm_scale), int(mode), _ptr(out),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                   _stream(stream)),
           "lynx_verify_attn")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def decode_attn_noalloc(q, k: QuantizedKV, v: QuantizedKV, layer, page_table, ctx_lens, sm_scale, mode,
                        out=None, scores=None, dev_err=None, stream=None):
    """lynx_decode_attn_noalloc: decode attention for callers that cannot
    allocate device memory. Its split-K scratch is a fixed 16 MiB array inside
    the library, shared by every call on the device (serialise calls)."""
    _dev(q, torch.bfloat16, "q")
    _dev(page_table, torch.int32, "page_table")
    _dev(ctx_lens, torch.int32, "ctx_lens")
    B, Hq, _ = q.shape
    if out is None:
        out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    kd, vd = k.desc(), v.desc()
    _check(_lib().lynx_decode_attn_noalloc(_ptr(q), ctypes.byref(kd), ctypes.byref(vd), layer, _ptr(page_table),
                                           _ptr(ctx_lens), B, Hq, page_table.shape[1], float(sm_scale), int(mode),
                                           _ptr(out), _ptr(scores), _ptr(dev_err), _stream(stream)),
           "lynx_decode_attn_noalloc")
    return out


def host_tables():
    """(thr float32[64], lv uint16[65]) exactly as the kernels use them (host call)."""
    import numpy as np
    thr = np.zeros(64, np.float32)
    lv = np.zeros(65, np.uint16)
    _lib().lynx_host_tables(thr.ctypes.data_as(ctypes.c_void_p), lv.ctypes.data_as(ctypes.c_void_p))
    return thr, lv


def level_codes(w, stream=None):
    """Stage-3 codes of a float32 CUDA tensor, through the encoder's code path."""
    _dev(w, torch.float32, "w")
    codes = torch.empty(w.shape, dtype=torch.int8, device=w.device)
    _check(_lib().lynx_level_codes(_ptr(w), w.numel(), _ptr(codes), _stream(stream)), "lynx_level_codes")
    return codes


def quantize_variant(x, chunk=32, anchor_bits=4, residual_bits=4, alpha=255.0, flags=0, uniform_bits=0,
                     codes=False, planes=False, meta=False, recon=False, stream=None):
    """lynx_quantize_variant: encode x (bfloat16 [..., tokens, 128], tokens a
    multiple of 256) with one variant of the quantizer in a single pass.
    Returns a dict with "err" (float64 [n, pages, 3]: sum x^2, anchor-only and
    full squared errors per page) and, on request, "codes" (int16), "anchor"
    (int8) / "residual" (uint8), "page_meta" / "chunk_meta" and (recon=True)
    the fp32 reconstructions "x_anchor" / "x_full" ([n, tokens, 128])."""
    _dev(x, torch.bfloat16, "x")
    if x.dim() < 2 or x.shape[-1] != HEAD_DIM:
        raise ValueError("x must be [..., tokens, 128]")
    T = x.shape[-2]
    n = x.numel() // (T * HEAD_DIM)
    P = T // 256
    dev = x.device
    v = LynxVariant(chunk, anchor_bits, residual_bits, alpha, flags, uniform_bits)
    out = {"err": torch.empty((n, P, 3), dtype=torch.float64, device=dev)}
    if codes:
        out["codes"] = torch.empty((n, T, HEAD_DIM), dtype=torch.int16, device=dev)
    if planes and not uniform_bits:
        out["anchor"] = torch.empty((n, T, HEAD_DIM), dtype=torch.int8, device=dev)
        out["residual"] = torch.empty((n, T, HEAD_DIM), dtype=torch.uint8, device=dev)
    if meta:
        out["page_meta"] = torch.empty((n, P, 2, HEAD_DIM), dtype=torch.float32, device=dev)
        if not uniform_bits:
            out["chunk_meta"] = torch.empty((n, P, 256 // chunk, 2, HEAD_DIM), dtype=torch.int16, device=dev)
    if recon:
        out["x_anchor"] = torch.empty((n, T, HEAD_DIM), dtype=torch.float32, device=dev)
        out["x_full"] = torch.empty((n, T, HEAD_DIM), dtype=torch.float32, device=dev)
    _check(_lib().lynx_quantize_variant(_ptr(x), n, T, ctypes.byref(v), _ptr(out.get("codes")),
                                        _ptr(out.get("anchor")), _ptr(out.get("residual")),
                                        _ptr(out.get("page_meta")), _ptr(out.get("chunk_meta")), _ptr(out["err"]),
                                        _ptr(out.get("x_anchor")), _ptr(out.get("x_full")), _stream(stream)),
           "lynx_quantize_variant")
    return out


def dense_attn(q, k, v, sm_scale=None, stream=None):
    """lynx_dense_attn: decode attention over a dense fp32 cache (a quality
    study tool). q: bfloat16 [batch, q_heads, 128]; k, v: float32
    [kv_heads, tokens, 128], shared by every request. Returns float32
    [batch, q_heads, 128]."""
    _dev(q, torch.bfloat16, "q")
    _dev(k, torch.float32, "k")
    _dev(v, torch.float32, "v")
    if q.dim() != 3 or k.dim() != 3 or q.shape[-1] != HEAD_DIM or k.shape != v.shape or k.shape[-1] != HEAD_DIM:
        raise ValueError("q must be [batch, q_heads, 128], k and v [kv_heads, tokens, 128]")
    B, Hq = q.shape[0], q.shape[1]
    H, T = k.shape[0], k.shape[1]
    scale = HEAD_DIM ** -0.5 if sm_scale is None else sm_scale
    out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    _check(_lib().lynx_dense_attn(_ptr(q), _ptr(k), _ptr(v), B, Hq, H, T, scale, _ptr(out), _stream(stream)),
           "lynx_dense_attn")
    return out

