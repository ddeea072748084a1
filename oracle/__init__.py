"""fp64 CPU oracle for cartridge attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never routes through it.

The arithmetic lives in ``cart_oracle.c`` (plain loops in fp64, OpenMP over
independent (batch, head) problems); this module only compiles it with gcc and
marshals numpy arrays into it.  See that file's header for what is computed
and which passage of the Cartridges guide each part follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cart_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcart_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libcart_oracle.so`` (gcc, -O2,
    OpenMP when available; never -ffast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("n", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("p", ctypes.c_int),
                ("frozen_prefix", ctypes.c_int), ("scale", ctypes.c_double),
                ("theta", ctypes.c_double), ("window", ctypes.c_int)]


_D = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.cart_oracle_fwd.restype = ctypes.c_int
            L.cart_oracle_fwd.argtypes = [ctypes.POINTER(_Geom)] + [_D] * 7 + [ctypes.c_int] * 4
            L.cart_oracle_bwd.restype = ctypes.c_int
            L.cart_oracle_bwd.argtypes = [ctypes.POINTER(_Geom)] + [_D] * 11 + [ctypes.c_int] * 4
            L.cart_oracle_decode.restype = ctypes.c_int
            L.cart_oracle_decode.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_double] * 2
                                             + [_D] * 7 + [ctypes.c_int,
                                                           ctypes.POINTER(ctypes.c_int), _D,
                                                           ctypes.c_int])
            L.cart_oracle_rope.restype = None
            L.cart_oracle_rope.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double, ctypes.c_int]
            L.cart_oracle_write_to_cache.restype = None
            L.cart_oracle_write_to_cache.argtypes = [
                ctypes.POINTER(ctypes.c_float), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_uint16), ctypes.c_longlong, ctypes.c_int]
            L.cart_oracle_num_threads.restype = ctypes.c_int
            _lib = L
        return _lib


def num_threads() -> int:
    return int(lib().cart_oracle_num_threads())


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _geom(B, n, Hq, Hkv, d, p, frozen_prefix, scale, theta, window=0) -> _Geom:
    return _Geom(B, n, Hq, Hkv, d, p, frozen_prefix, float(scale), float(theta), int(window))


def fwd(q, k, v, kc, vc, *, p=None, frozen_prefix=1, scale=None, theta=1.0e6,
        heads=None, rows=None, window=0):
    """Forward of cartridge attention.

    q ``[B, n, Hq, d]``, k/v ``[B, n, Hkv, d]``, kc/vc ``[p, Hkv, d]`` (any
    float arrays; read as fp64).  Returns ``(o [B, n, Hq, d], lse [B, Hq, n])``.
    ``heads=(lo, hi)`` / ``rows=(lo, hi)`` restrict which outputs are computed
    (the rest are NaN).  ``window`` W > 0 is a sliding window (Cartridges
    guide, "gemma4 (measured)": a cartridge is visible to a local-SWA query
    exactly as a real prefix, within the window): the query at position P
    sees keys at positions P - W + 1 .. P, cartridge row j at position j."""
    q, k, v, kc, vc = (_f64(t) for t in (q, k, v, kc, vc))
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    if p is None:
        p = kc.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if kc.size == 0:
        kc = np.zeros((1, Hkv, d))
        vc = np.zeros((1, Hkv, d))
    o = np.full((B, n, Hq, d), np.nan)
    lse = np.full((B, Hq, n), np.nan)
    h_lo, h_hi = heads if heads is not None else (0, Hq)
    i_lo, i_hi = rows if rows is not None else (0, n)
    # the forward does not depend on which rows are frozen
    g = _geom(B, n, Hq, Hkv, d, p, min(frozen_prefix, p), scale, theta, window)
    rc = lib().cart_oracle_fwd(ctypes.byref(g), _ptr(q), _ptr(k), _ptr(v), _ptr(kc),
                               _ptr(vc), _ptr(o), _ptr(lse), h_lo, h_hi, i_lo, i_hi)
    if rc != 0:
        raise ValueError(f"cart_oracle_fwd failed ({rc})")
    return o, lse


def bwd(q, k, v, kc, vc, dout, *, p=None, frozen_prefix=1, scale=None, theta=1.0e6,
        kv_heads=None, rows=None, frozen_rows=(), window=0):
    """Gradients of ``sum(dout * o)``: returns ``dq, dk, dv, dkc, dvc`` (fp64),
    dkc/dvc summed over the batch with rows ``< frozen_prefix`` exactly 0.
    ``frozen_rows`` lists further frozen cartridge rows (a composed
    cartridge: parts concatenated along the rows, each keeping its own sink
    row); a frozen row is a constant of the loss, so its gradient is 0.
    ``kv_heads=(lo, hi)`` restricts the work to those kv heads and the query
    heads reading them (other entries are NaN).  ``rows=(lo, hi)`` counts only
    those query rows of the loss: dq outside them is NaN and dk/dv/dkc/dvc
    hold those rows' contributions (exact for keys no other row sees)."""
    q, k, v, kc, vc, dout = (_f64(t) for t in (q, k, v, kc, vc, dout))
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    if p is None:
        p = kc.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    pc = max(p, 1)
    if kc.size == 0:
        kc = np.zeros((1, Hkv, d))
        vc = np.zeros((1, Hkv, d))
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    dkc = np.full((pc, Hkv, d), np.nan)
    dvc = np.full((pc, Hkv, d), np.nan)
    lo, hi = kv_heads if kv_heads is not None else (0, Hkv)
    i_lo, i_hi = rows if rows is not None else (0, n)
    g = _geom(B, n, Hq, Hkv, d, p, frozen_prefix, scale, theta, window)
    rc = lib().cart_oracle_bwd(ctypes.byref(g), _ptr(q), _ptr(k), _ptr(v), _ptr(kc),
                               _ptr(vc), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(dkc), _ptr(dvc), lo, hi, i_lo, i_hi)
    if rc != 0:
        raise ValueError(f"cart_oracle_bwd failed ({rc})")
    for j in frozen_rows:
        if not 0 <= j < p:
            raise ValueError("frozen row outside the cartridge")
        dkc[j] = 0.0
        dvc[j] = 0.0
    return dq, dk, dv, dkc[:p], dvc[:p]


def _segments(cu_seqlens, total):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must rise from 0 to the packed token count")
    return [(int(a), int(b)) for a, b in zip(cu[:-1], cu[1:])]


def fwd_packed(q, k, v, kc, vc, cu_seqlens, *, p=None, frozen_prefix=1, scale=None,
               theta=1.0e6, window=0, heads=None):
    """Packed segments (Cartridges guide, "Deliberate divergences from the
    reference", packing bullet; "Batched self-study (measured)", packed
    training step): the group's sequences lie back to back along ONE token
    axis, q ``[T, Hq, d]``, k/v ``[T, Hkv, d]``, segment s holding tokens
    ``cu_seqlens[s] .. cu_seqlens[s+1] - 1``.  RoPE restarts per segment
    (its token i sits at position p + i) and attention runs per segment
    behind the one shared cartridge, so each segment is exactly a
    single-sequence call of ``fwd``.  Returns ``(o [T, Hq, d], lse [Hq, T])``
    (``heads`` restricts the computed heads as in ``fwd``)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    o = np.zeros((T, Hq, d))
    lse = np.zeros((Hq, T))
    for a, b in _segments(cu_seqlens, T):
        if b == a:
            continue
        o_s, lse_s = fwd(q[None, a:b], k[None, a:b], v[None, a:b], kc, vc, p=p,
                         frozen_prefix=frozen_prefix, scale=scale, theta=theta, window=window,
                         heads=heads)
        o[a:b] = o_s[0]
        lse[:, a:b] = lse_s[0]
    return o, lse


def bwd_packed(q, k, v, kc, vc, dout, cu_seqlens, *, p=None, frozen_prefix=1, scale=None,
               theta=1.0e6, frozen_rows=(), window=0, kv_heads=None):
    """Gradients of ``sum(dout * o)`` for packed segments (layouts of
    ``fwd_packed``): each segment's dq/dk/dv are those of its own
    single-sequence problem, and the cartridge gradient is their sum over
    the segments (one shared cartridge), frozen rows exactly 0."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T = q.shape[0]
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    kc64 = _f64(kc)
    dkc = np.zeros(kc64.shape)
    dvc = np.zeros(kc64.shape)
    for a, b in _segments(cu_seqlens, T):
        if b == a:
            continue
        g = bwd(q[None, a:b], k[None, a:b], v[None, a:b], kc, vc, dout[None, a:b], p=p,
                frozen_prefix=frozen_prefix, scale=scale, theta=theta, frozen_rows=frozen_rows,
                window=window, kv_heads=kv_heads)
        dq[a:b], dk[a:b], dv[a:b] = g[0][0], g[1][0], g[2][0]
        dkc += g[3]
        dvc += g[4]
    return dq, dk, dv, dkc, dvc


def decode(q, k_new, v_new, kc, vc, k_cache, v_cache, lens, *, scale=None, theta=1.0e6,
           window=0):
    """One decode step behind a shared cartridge.  Returns
    ``(o [B, Hq, d], k_cache', v_cache')`` where the caches have the new
    token's rotated key / value written at row ``lens[b]``."""
    q, k_new, v_new, kc, vc = (_f64(t) for t in (q, k_new, v_new, kc, vc))
    kcache = _f64(k_cache).copy()
    vcache = _f64(v_cache).copy()
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    p = kc.shape[0]
    rows = kcache.shape[1]
    lens = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if kc.size == 0:
        kc = np.zeros((1, Hkv, d))
        vc = np.zeros((1, Hkv, d))
    o = np.full((B, Hq, d), np.nan)
    rc = lib().cart_oracle_decode(B, Hq, Hkv, d, p, float(scale), float(theta), _ptr(q),
                                  _ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(kcache),
                                  _ptr(vcache), rows,
                                  lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _ptr(o),
                                  int(window))
    if rc != 0:
        raise ValueError(f"cart_oracle_decode failed ({rc})")
    return o, kcache, vcache


def decode_span(q, k_new, v_new, kc, vc, k_cache, v_cache, lens, *, scale=None, theta=1.0e6,
                window=0):
    """Span verify (Cartridges guide, "Batched self-study (measured)", the
    --spec-b bullet): ``span`` new tokens per conversation in one step
    (q ``[B, span, Hq, d]``, k_new / v_new ``[B, span, Hkv, d]``).  Token t
    sits at position p + lens[b] + t, its rotated key / value go to private
    row lens[b] + t, and query t sees the cartridge and private rows
    0 .. lens[b] + t -- the end-aligned causal mask over the span, i.e. the
    span's single-token steps taken in order.  Returns
    ``(o [B, span, Hq, d], k_cache', v_cache')``."""
    q, k_new, v_new = _f64(q), _f64(k_new), _f64(v_new)
    span = q.shape[1]
    kcache, vcache = _f64(k_cache).copy(), _f64(v_cache).copy()
    lens = np.asarray(lens, dtype=np.int64)
    o = np.empty(q.shape)
    for t in range(span):
        o[:, t], kcache, vcache = decode(q[:, t], k_new[:, t], v_new[:, t], kc, vc, kcache,
                                         vcache, lens + t, scale=scale, theta=theta,
                                         window=window)
    return o, kcache, vcache


def rope(x, pos0, *, theta=1.0e6, inverse=False):
    """Rotate ``x [rows, H, d]`` row r at position ``pos0 + r``."""
    x = _f64(x)
    rows, H, d = x.shape
    out = np.empty_like(x)
    lib().cart_oracle_rope(_ptr(x), _ptr(out), rows, H, d, float(pos0), float(theta),
                           1 if inverse else 0)
    return out


def write_to_cache(src_f32, dst_u16, dst_row0=0):
    """f32 ``[p, Hkv, d]`` -> bf16 bit patterns written into ``dst_u16``
    (``[rows, Hkv, d]`` uint16, modified in place) from row ``dst_row0``."""
    src = np.ascontiguousarray(np.asarray(src_f32, dtype=np.float32))
    p, Hkv, d = src.shape
    assert dst_u16.dtype == np.uint16 and dst_u16.flags.c_contiguous
    assert dst_u16.shape[1:] == (Hkv, d) and dst_row0 + p <= dst_u16.shape[0]
    lib().cart_oracle_write_to_cache(src.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), p,
                                     Hkv, d,
                                     dst_u16.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                     Hkv * d, dst_row0)
    return dst_u16
