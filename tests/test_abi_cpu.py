"""The C ABI without a GPU: the library loads, exports every declared symbol,
builds the same tables as the oracle, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lynx.h")


@pytest.fixture(scope="module")
def lx():
    from progressive_kv_cache_gb300 import build
    build.build()
    import progressive_kv_cache_gb300 as lx
    return lx


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lynx_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lx):
    names = _declared()
    assert {"lynx_quantize_pages", "lynx_dequant_anchor", "lynx_refine_residual", "lynx_decode_attn",
            "lynx_decode_attn_workspace", "lynx_status_string"} <= set(names)
    lib = lx.library()
    for n in names:
        assert hasattr(lib, n), n


def test_noalloc_scratch_size_matches_the_header(lx):
    """The binding's copy of the no-alloc scratch size is the header's."""
    src = open(HEADER).read()
    m = re.search(r"#define\s+LYNX_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", src)
    assert m, "LYNX_NOALLOC_SCRATCH_BYTES not found"
    assert lx.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_status_strings(lx):
    lib = lx.library()
    seen = set()
    for s in range(7):
        txt = lib.lynx_status_string(s).decode()
        assert txt and txt not in seen
        seen.add(txt)
    assert lib.lynx_status_string(99).decode() == "unknown status"


def test_host_tables_equal_the_oracles(lx, orc):
    thr, lv = lx.host_tables()
    othr, olv = orc.tables()
    assert np.array_equal(thr.view(np.uint32), othr.view(np.uint32))
    assert np.array_equal(lv, olv)


def _qkv(lx, L=1, H=1, T=256, base=0x10000, residual=True):
    return lx.LynxQKV(L, H, T, 128, base, base + 0x100000 if residual else None, base + 0x200000,
                      base + 0x300000)


def _q(lx, d, x=0x400000, pv=None):
    lib = lx.library()
    return lib.lynx_quantize_pages(ctypes.c_void_p(x), None if pv is None else ctypes.c_void_p(pv),
                                   ctypes.byref(d), None)


def test_quantize_rejects_bad_arguments(lx):
    assert _q(lx, _qkv(lx), x=0) == lx.ERR_NULL
    assert _q(lx, _qkv(lx, residual=False)) == lx.ERR_NULL
    assert _q(lx, _qkv(lx, T=300)) == lx.ERR_SHAPE
    d = _qkv(lx)
    d.head_dim = 64
    assert _q(lx, d) == lx.ERR_SHAPE
    assert _q(lx, _qkv(lx, L=-1)) == lx.ERR_SHAPE
    assert _q(lx, _qkv(lx), x=0x400008) == lx.ERR_ALIGN
    assert _q(lx, _qkv(lx, base=0x10004)) == lx.ERR_ALIGN
    assert _q(lx, _qkv(lx), pv=0x500002) == lx.ERR_ALIGN
    # 2^23 pages: more rows than 32-bit tile coordinates address (refused
    # before anything reaches a device)
    assert _q(lx, _qkv(lx, L=1024, H=32, T=65536)) == lx.ERR_UNSUPPORTED


def test_dequant_and_refine_reject_bad_arguments(lx):
    lib = lx.library()
    d = _qkv(lx)
    assert lib.lynx_dequant_anchor(ctypes.byref(d), None, 0, None) == lx.ERR_NULL
    assert lib.lynx_dequant_anchor(ctypes.byref(d), ctypes.c_void_p(0x400004), 0, None) == lx.ERR_ALIGN
    assert lib.lynx_dequant_anchor(ctypes.byref(d), ctypes.c_void_p(0x400000), 7, None) == lx.ERR_UNSUPPORTED
    d2 = _qkv(lx, residual=False)
    assert lib.lynx_refine_residual(ctypes.byref(d2), ctypes.c_void_p(0x400000), 0, None) == lx.ERR_NULL
    assert lib.lynx_dequant_anchor(None, ctypes.c_void_p(0x400000), 0, None) == lx.ERR_NULL


def _attn(lx, k, v, layer=0, B=1, Hq=4, maxp=1, mode=0, q=0x600000, pt=0x700000, ctx=0x700100,
          out=0x800000, ws=0x900000, wsb=1 << 30):
    lib = lx.library()
    return lib.lynx_decode_attn(ctypes.c_void_p(q) if q else None, ctypes.byref(k), ctypes.byref(v), layer,
                                ctypes.c_void_p(pt) if pt else None, ctypes.c_void_p(ctx), B, Hq, maxp, 0.1,
                                mode, ctypes.c_void_p(out), None, ctypes.c_void_p(ws) if ws else None, wsb,
                                None, None)


def test_decode_attn_rejects_bad_arguments(lx):
    k, v = _qkv(lx, H=2), _qkv(lx, H=2, base=0x20000000)
    assert _attn(lx, k, v, q=0) == lx.ERR_NULL
    assert _attn(lx, k, v, pt=0) == lx.ERR_NULL
    assert _attn(lx, k, v, layer=1) == lx.ERR_SHAPE
    assert _attn(lx, k, v, Hq=3) == lx.ERR_SHAPE                 # not a multiple of kv_heads
    assert _attn(lx, k, v, Hq=2 * 33) == lx.ERR_UNSUPPORTED       # group of 33
    assert _attn(lx, k, v, maxp=0) == lx.ERR_SHAPE
    assert _attn(lx, k, _qkv(lx, H=1, base=0x20000000)) == lx.ERR_SHAPE
    assert _attn(lx, k, v, out=0x800004) == lx.ERR_ALIGN
    assert _attn(lx, k, v, pt=0x700002) == lx.ERR_ALIGN
    ka, va = _qkv(lx, H=2, residual=False), _qkv(lx, H=2, base=0x20000000, residual=False)
    assert _attn(lx, ka, va, mode=1) == lx.ERR_NULL              # full mode needs residuals
    assert _attn(lx, ka, va, mode=5) == lx.ERR_UNSUPPORTED
    assert _attn(lx, k, v, B=0) == lx.OK                          # nothing to do, no launch


def test_workspace_query(lx):
    lib = lx.library()
    assert lib.lynx_decode_attn_workspace(0, 64, 10) == 0
    assert lib.lynx_decode_attn_workspace(1, 64, 0) == 0
    a = lib.lynx_decode_attn_workspace(1, 64, 512)
    b = lib.lynx_decode_attn_workspace(2, 64, 512)
    assert a > 0 and b > 0 and a % 16 == 0


def test_level_codes_rejects_bad_arguments(lx):
    lib = lx.library()
    assert lib.lynx_level_codes(None, 10, None, None) == lx.ERR_NULL
    assert lib.lynx_level_codes(None, -1, None, None) == lx.ERR_SHAPE
    assert lib.lynx_level_codes(None, 0, None, None) == lx.OK


def test_quantize_append_rejects_bad_arguments(lx):
    lib = lx.library()

    def call(d, tail=0x400000, pp=0x500000, va=0x500100, n=2, err=None):
        return lib.lynx_quantize_append(ctypes.c_void_p(tail) if tail else None,
                                        ctypes.c_void_p(pp) if pp else None,
                                        ctypes.c_void_p(va) if va else None, n, ctypes.byref(d),
                                        ctypes.c_void_p(err) if err else None, None)

    assert call(_qkv(lx), tail=0) == lx.ERR_NULL
    assert call(_qkv(lx), pp=0) == lx.ERR_NULL
    assert call(_qkv(lx), va=0) == lx.ERR_NULL
    assert call(_qkv(lx, residual=False)) == lx.ERR_NULL
    assert call(_qkv(lx), n=-1) == lx.ERR_SHAPE
    assert call(_qkv(lx, T=300)) == lx.ERR_SHAPE
    assert call(_qkv(lx), tail=0x400008) == lx.ERR_ALIGN
    assert call(_qkv(lx), pp=0x500002) == lx.ERR_ALIGN
    assert call(_qkv(lx), err=0x600001) == lx.ERR_ALIGN
    assert call(_qkv(lx), n=0) == lx.OK                       # nothing to do, no launch


def test_verify_attn_rejects_bad_arguments(lx):
    lib = lx.library()
    k, v = _qkv(lx, H=2), _qkv(lx, H=2, base=0x20000000)

    def call(k=k, v=v, layer=0, B=1, Tq=4, Hq=4, maxp=1, mode=1, q=0x600000, out=0x800000, ws=0x900000,
             wsb=1 << 30):
        return lib.lynx_verify_attn(ctypes.c_void_p(q) if q else None, ctypes.byref(k), ctypes.byref(v), layer,
                                    ctypes.c_void_p(0x700000), ctypes.c_void_p(0x700100), B, Tq, Hq, maxp, 0.1,
                                    mode, ctypes.c_void_p(out) if out else None,
                                    ctypes.c_void_p(ws) if ws else None, wsb, None, None)

    assert call(q=0) == lx.ERR_NULL
    assert call(out=0) == lx.ERR_NULL
    assert call(Tq=0) == lx.ERR_SHAPE
    assert call(Tq=65) == lx.ERR_SHAPE
    assert call(Hq=3) == lx.ERR_SHAPE
    assert call(layer=2) == lx.ERR_SHAPE
    assert call(out=0x800004) == lx.ERR_ALIGN
    assert call(mode=7) == lx.ERR_UNSUPPORTED
    assert call(k=_qkv(lx, H=2, residual=False)) == lx.ERR_NULL     # full mode needs residuals
    assert call(B=0) == lx.OK
    assert lib.lynx_verify_attn_workspace(1, 0, 64, 8) == 0
    assert lib.lynx_verify_attn_workspace(1, 65, 64, 8) == 0
    assert lib.lynx_verify_attn_workspace(2, 64, 64, 512) % 16 == 0


def test_quantize_variant_rejects_bad_arguments(lx):
    lib = lx.library()

    def call(n=1, T=256, x=0x400000, err=0x500000, codes=None, xf=None, **kw):
        v = lx.LynxVariant(kw.get("chunk", 32), kw.get("a", 4), kw.get("r", 4), kw.get("alpha", 255.0),
                           kw.get("flags", 0), kw.get("ub", 0))
        return lib.lynx_quantize_variant(ctypes.c_void_p(x) if x else None, n, T, ctypes.byref(v),
                                         ctypes.c_void_p(codes) if codes else None, None, None, None, None,
                                         ctypes.c_void_p(err) if err else None, None,
                                         ctypes.c_void_p(xf) if xf else None, None)

    assert lib.lynx_quantize_variant(None, 1, 256, None, None, None, None, None, None, None, None, None,
                                     None) == lx.ERR_NULL
    assert call(x=0) == lx.ERR_NULL
    assert call(T=300) == lx.ERR_SHAPE
    assert call(n=-1) == lx.ERR_SHAPE
    assert call(chunk=8) == lx.ERR_UNSUPPORTED
    assert call(a=7) == lx.ERR_UNSUPPORTED
    assert call(r=5) == lx.ERR_UNSUPPORTED
    assert call(a=6, r=4) == lx.ERR_UNSUPPORTED              # more than 8 bits
    assert call(alpha=-1.0) == lx.ERR_UNSUPPORTED
    assert call(alpha=float("nan")) == lx.ERR_UNSUPPORTED
    assert call(flags=16) == lx.ERR_UNSUPPORTED
    assert call(ub=9) == lx.ERR_UNSUPPORTED
    assert call(x=0x400008) == lx.ERR_ALIGN
    assert call(codes=0x600002) == lx.ERR_ALIGN
    assert call(xf=0x700004) == lx.ERR_ALIGN
    assert call(n=0) == lx.OK                                 # nothing to do, no launch
    assert call(T=0) == lx.OK


def test_dense_attn_rejects_bad_arguments(lx):
    lib = lx.library()
    q, k, v, o = (ctypes.c_void_p(a) for a in (0x400000, 0x500000, 0x600000, 0x700000))

    def call(B=1, Hq=8, H=2, T=64, q=q, k=k, v=v, o=o):
        return lib.lynx_dense_attn(q, k, v, B, Hq, H, T, 0.088, o, None)

    assert call(B=-1) == lx.ERR_SHAPE
    assert call(T=-1) == lx.ERR_SHAPE
    assert call(Hq=6, H=4) == lx.ERR_SHAPE                   # query heads not a multiple of KV heads
    assert call(H=0) == lx.ERR_SHAPE
    assert call(T=0) == lx.ERR_SHAPE
    assert call(T=49153) == lx.ERR_SHAPE                     # scores no longer fit in shared memory
    assert call(k=None) == lx.ERR_NULL
    assert call(o=None) == lx.ERR_NULL
    assert call(k=ctypes.c_void_p(0x500008)) == lx.ERR_ALIGN
    assert call(q=ctypes.c_void_p(0x400001)) == lx.ERR_ALIGN
    assert call(B=0) == lx.OK                                # nothing to do, no launch
    assert call(Hq=0, q=None) == lx.OK


def test_stage3_integer_index_scheme(lx, orc):
    """The encoder's stage-3 lookup, emulated from the library's thresholds:
    16 buckets per octave of |w| + 2^-13 hold at most one threshold T*, and
    bits 31-30 of bits(w) + (2^30 - bits(T*)) (0 when a bucket holds none) are
    2 sign(w) + (|w| >= T*), the index of the stored code among the four an
    entry carries. The result is compared with the oracle's direct count of
    thresholds, near every threshold (both signs, 64 fp32 steps each side),
    at every bucket edge, and on a dense uniform sample of [-1, 1]."""
    thr, _ = lx.host_tables()
    thr = np.asarray(thr, np.float32)
    off = np.float32(2.0 ** -13)
    base = (127 - 13) << 4

    def bucket(a):
        return ((np.asarray(a, np.float32) + off).view(np.uint32) >> 19).astype(np.int64) - base

    tb = bucket(thr[1:])
    nb = 14 * 16
    assert tb.min() >= 0 and tb.max() < nb
    assert len(np.unique(tb)) == len(tb)       # at most one threshold per bucket
    q0 = np.searchsorted(np.sort(tb), np.arange(nb), side="left")   # thresholds in lower buckets
    k_add = np.zeros(nb, np.uint64)
    k_add[tb] = (1 << 30) - thr[1:].view(np.uint32).astype(np.uint64)
    q1 = np.minimum(q0 + 1, 63)
    entry = np.stack([q0, q1, -np.maximum(q0, 1), -np.maximum(q1, 1)], axis=1)

    near = (thr[1:].view(np.int32)[:, None] + np.arange(-64, 65)[None, :]).ravel().view(np.float32)
    edges = ((np.arange(nb, dtype=np.uint32) + base) << 19).view(np.float32) - off
    edges = np.concatenate([edges, np.nextafter(edges, np.float32(0)), np.nextafter(edges, np.float32(2))])
    edges = edges[(edges >= 0) & (edges <= 1)]
    rng = np.random.default_rng(7)
    mag = np.concatenate([near, edges, rng.random(1 << 20, dtype=np.float32), np.float32([0.0, 1.0])])
    w = np.concatenate([mag, -mag[mag > 0]]).astype(np.float32)

    b = bucket(np.abs(w))
    assert b.min() >= 0 and b.max() < nb
    t = (w.view(np.uint32).astype(np.uint64) + k_add[b]) & 0xFFFFFFFF
    got = entry[b, (t >> 30).astype(np.int64)]
    assert np.array_equal(got, orc.codes(w).astype(np.int64))
