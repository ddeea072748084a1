"""Thin ctypes binding of ``libcartattn.so`` (see ``include/cartattn.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory (outputs and workspaces are
allocated with ``torch.empty`` on the inputs' device) and the current stream.
If the library has not been built, every call raises -- there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build

CART_BF16 = 0
CART_F32 = 1

STATUS = {0: "ok", -1: "bad geometry", -2: "null or misaligned pointer", -3: "unsupported dtype",
          -4: "workspace too small", -5: "CUDA error", -6: "device is not sm_103",
          -7: "a kernel gave up waiting"}

_lock = threading.Lock()
_lib = None


class CartError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


class _Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("n", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("p", ctypes.c_int),
                ("frozen_prefix", ctypes.c_int), ("scale", ctypes.c_float),
                ("rope_theta", ctypes.c_double), ("window", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the in-tree library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m trained_kv_prefix_gb300.build` "
                    "(there is no non-CUDA implementation of this path)")
            L = ctypes.CDLL(path)
            vp, sz, i, f, d = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float, ctypes.c_double
            G = ctypes.POINTER(_Geom)
            L.cart_write_to_cache.argtypes = [vp, vp, i, i, i, vp, vp, ctypes.c_longlong, i, i, vp]
            L.cart_attn_fwd_workspace_size.argtypes = [G, i, i]
            L.cart_attn_fwd_workspace_size.restype = sz
            L.cart_attn_fwd.argtypes = [G, i, i, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.cart_attn_bwd_workspace_size.argtypes = [G, i, i]
            L.cart_attn_bwd_workspace_size.restype = sz
            L.cart_attn_bwd.argtypes = [G, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        i, vp, sz, vp]
            L.cart_attn_bwd_parts.argtypes = [G, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, vp, ctypes.POINTER(ctypes.c_int), i, i, vp,
                                              sz, vp]
            L.cart_attn_bwd_reuse_workspace_size.argtypes = [G, i, i]
            L.cart_attn_bwd_reuse_workspace_size.restype = sz
            L.cart_attn_bwd_reuse.argtypes = [G, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, vp, i, vp, sz, vp, sz, vp]
            L.cart_attn_decode_workspace_size.argtypes = [i, i, i, i, i, i]
            L.cart_attn_decode_workspace_size.restype = sz
            L.cart_attn_decode.argtypes = [i, i, i, i, i, f, d, vp, vp, vp, vp, vp, vp, vp, i, vp,
                                           vp, vp, sz, vp]
            L.cart_attn_decode_span_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.cart_attn_decode_span_workspace_size.restype = sz
            L.cart_attn_decode_span.argtypes = [i, i, i, i, i, i, i, f, d, vp, vp, vp, vp, vp, vp,
                                                vp, i, vp, vp, vp, sz, vp]
            L.cart_attn_fwd_packed_workspace_size.argtypes = [G, i, i, i]
            L.cart_attn_fwd_packed_workspace_size.restype = sz
            L.cart_attn_fwd_packed.argtypes = [G, i, vp, i, i, vp, vp, vp, vp, vp, vp, vp, vp,
                                               sz, vp]
            L.cart_attn_bwd_packed_workspace_size.argtypes = [G, i, i, i]
            L.cart_attn_bwd_packed_workspace_size.restype = sz
            L.cart_attn_bwd_packed.argtypes = [G, i, vp, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                               vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int), i, i,
                                               vp, sz, vp]
            L.cart_status_string.argtypes = [i]
            L.cart_status_string.restype = ctypes.c_char_p
            L.cart_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
            L.cart_trace_enable.argtypes = [i]
            L.cart_release.argtypes = []
            L.cart_release.restype = ctypes.c_int
            L.cart_trace_count.argtypes = []
            L.cart_trace_get.argtypes = [i, ctypes.c_char_p, i, ctypes.POINTER(ctypes.c_float)]
            for name in ("cart_write_to_cache", "cart_attn_fwd", "cart_attn_bwd", "cart_attn_bwd_parts",
                         "cart_attn_bwd_reuse",
                         "cart_attn_fwd_packed", "cart_attn_bwd_packed",
                         "cart_attn_decode", "cart_attn_decode_span", "cart_device_status",
                         "cart_trace_enable",
                         "cart_trace_count", "cart_trace_get"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
        return _lib


EXPORTS = ("cart_write_to_cache", "cart_attn_fwd_workspace_size", "cart_attn_fwd",
           "cart_attn_bwd_workspace_size", "cart_attn_bwd", "cart_attn_bwd_parts",
           "cart_attn_bwd_reuse_workspace_size", "cart_attn_bwd_reuse",
           "cart_attn_decode_workspace_size",
           "cart_attn_decode", "cart_status_string", "cart_device_status", "cart_trace_enable",
           "cart_trace_count", "cart_trace_get", "cart_attn_decode_noalloc",
           "cart_attn_decode_span_workspace_size", "cart_attn_decode_span",
           "cart_attn_fwd_packed_workspace_size", "cart_attn_fwd_packed",
           "cart_attn_bwd_packed_workspace_size", "cart_attn_bwd_packed", "cart_release")


def _check(fn: str, rc: int):
    if rc != 0:
        raise CartError(fn, rc)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CART_BF16
    if t.dtype == torch.float32:
        return CART_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def geom(B, n, Hq, Hkv, d, p, frozen_prefix=1, scale=None, theta=1.0e6, window=0) -> _Geom:
    """Training geometry; ``window`` > 0 is a sliding window in keys (the
    query at position P sees keys P - window + 1 .. P), 0 none."""
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return _Geom(B, n, Hq, Hkv, d, p, frozen_prefix, float(scale), float(theta), int(window))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ calls ----
def cart_write_to_cache(kc: torch.Tensor, vc: torch.Tensor, k_dst: torch.Tensor,
                        v_dst: torch.Tensor, dst_row0: int = 0, stream=None):
    """Write f32 cartridge rows ``[p, Hkv, d]`` into ``k_dst``/``v_dst``
    (``[rows, Hkv, d]`` bf16 or f32) starting at row ``dst_row0``."""
    p, Hkv, d = kc.shape
    row_stride = k_dst.stride(0)
    rc = lib().cart_write_to_cache(_ptr(kc), _ptr(vc), p, Hkv, d, _ptr(k_dst), _ptr(v_dst),
                                   row_stride, dst_row0, _dt(k_dst), _stream(stream, kc.device))
    _check("cart_write_to_cache", rc)
    return k_dst, v_dst


def fwd_workspace_size(g: _Geom, in_dtype: int, cart_dtype: int) -> int:
    return int(lib().cart_attn_fwd_workspace_size(ctypes.byref(g), in_dtype, cart_dtype))


def bwd_workspace_size(g: _Geom, in_dtype: int, cart_dtype: int) -> int:
    return int(lib().cart_attn_bwd_workspace_size(ctypes.byref(g), in_dtype, cart_dtype))


def cart_attn_fwd(q, k, v, kc, vc, *, frozen_prefix=1, scale=None, theta=1.0e6, o=None, lse=None,
                  workspace=None, stream=None, window=0):
    """Training forward.  q ``[B, n, Hq, d]``, k/v ``[B, n, Hkv, d]`` (not
    rotated), kc/vc ``[p, Hkv, d]`` (bf16 shadow or f32 leaves).  Returns
    ``(o, lse)`` with o like q and lse ``[B, Hq, n]`` f32.  ``window`` > 0:
    sliding window in keys over the concatenated sequence (see ``geom``)."""
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    p = kc.shape[0]
    g = geom(B, n, Hq, Hkv, d, p, min(frozen_prefix, p), scale, theta, window)
    dt, cd = _dt(q), _dt(kc)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, n), dtype=torch.float32, device=q.device)
    ws = _workspace(fwd_workspace_size(g, dt, cd), q.device, workspace)
    rc = lib().cart_attn_fwd(ctypes.byref(g), dt, cd, _ptr(q), _ptr(k), _ptr(v), _ptr(kc),
                             _ptr(vc), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                             _stream(stream, q.device))
    _check("cart_attn_fwd", rc)
    return o, lse


def cart_attn_bwd(q, k, v, kc, vc, o, lse, dout, *, frozen_prefix=1, scale=None, theta=1.0e6,
                  accumulate=False, dq=None, dk=None, dv=None, dkc=None, dvc=None,
                  workspace=None, stream=None, frozen_rows=None, window=0,
                  fwd_workspace=None):
    """Backward.  Returns ``(dq, dk, dv, dkc, dvc)``; dkc/dvc are f32
    ``[p, Hkv, d]`` summed over the batch, rows < frozen_prefix and the rows
    listed in ``frozen_rows`` (a composed cartridge's part sinks) exactly 0.
    ``window`` must match the forward's.  ``fwd_workspace``: the workspace
    the forward of these inputs used (cart_attn_bwd_reuse: its rotated
    queries and keys are read instead of recomputed); not with
    ``frozen_rows``."""
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    p = kc.shape[0]
    g = geom(B, n, Hq, Hkv, d, p, frozen_prefix, scale, theta, window)
    dt, cd = _dt(q), _dt(kc)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dkc is None:
        dkc = (torch.zeros if accumulate else torch.empty)((max(p, 1), Hkv, d),
                                                           dtype=torch.float32, device=q.device)
    if dvc is None:
        dvc = (torch.zeros if accumulate else torch.empty)((max(p, 1), Hkv, d),
                                                           dtype=torch.float32, device=q.device)
    if fwd_workspace is not None:
        if frozen_rows is not None:
            raise ValueError("fwd_workspace does not combine with frozen_rows")
        ws = _workspace(int(lib().cart_attn_bwd_reuse_workspace_size(ctypes.byref(g), dt, cd)),
                        q.device, workspace)
        rc = lib().cart_attn_bwd_reuse(ctypes.byref(g), dt, cd, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(kc), _ptr(vc), _ptr(o), _ptr(lse), _ptr(dout),
                                       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkc), _ptr(dvc),
                                       1 if accumulate else 0, _ptr(fwd_workspace),
                                       fwd_workspace.numel(), _ptr(ws), ws.numel(),
                                       _stream(stream, q.device))
        _check("cart_attn_bwd_reuse", rc)
        return dq, dk, dv, dkc[:p], dvc[:p]
    ws = _workspace(bwd_workspace_size(g, dt, cd), q.device, workspace)
    if frozen_rows is None:
        rc = lib().cart_attn_bwd(ctypes.byref(g), dt, cd, _ptr(q), _ptr(k), _ptr(v), _ptr(kc),
                                 _ptr(vc), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(dkc), _ptr(dvc), 1 if accumulate else 0, _ptr(ws),
                                 ws.numel(), _stream(stream, q.device))
        _check("cart_attn_bwd", rc)
    else:
        rows = list(frozen_rows)
        arr = (ctypes.c_int * max(len(rows), 1))(*rows)
        rc = lib().cart_attn_bwd_parts(ctypes.byref(g), dt, cd, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(kc), _ptr(vc), _ptr(o), _ptr(lse), _ptr(dout),
                                       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkc), _ptr(dvc), arr,
                                       len(rows), 1 if accumulate else 0, _ptr(ws), ws.numel(),
                                       _stream(stream, q.device))
        _check("cart_attn_bwd_parts", rc)
    return dq, dk, dv, dkc[:p], dvc[:p]


def bwd_reuse_workspace_size(g: _Geom, in_dtype: int, cart_dtype: int) -> int:
    return int(lib().cart_attn_bwd_reuse_workspace_size(ctypes.byref(g), in_dtype, cart_dtype))


def fwd_packed_workspace_size(g: _Geom, total: int, in_dtype: int, cart_dtype: int) -> int:
    return int(lib().cart_attn_fwd_packed_workspace_size(ctypes.byref(g), total, in_dtype,
                                                         cart_dtype))


def bwd_packed_workspace_size(g: _Geom, total: int, in_dtype: int, cart_dtype: int) -> int:
    return int(lib().cart_attn_bwd_packed_workspace_size(ctypes.byref(g), total, in_dtype,
                                                         cart_dtype))


def _packing(cu_seqlens, max_seqlen, q):
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != q.device:
        raise TypeError("cu_seqlens must be int32 on the tensors' device")
    return cu_seqlens.numel() - 1, int(max_seqlen), q.shape[0]


def cart_attn_fwd_packed(q, k, v, kc, vc, cu_seqlens, max_seqlen, *, frozen_prefix=1,
                         scale=None, theta=1.0e6, o=None, lse=None, workspace=None, stream=None,
                         window=0):
    """Training forward on packed segments.  q ``[T, Hq, d]``, k/v
    ``[T, Hkv, d]`` (not rotated), segment s = tokens cu_seqlens[s] ..
    cu_seqlens[s+1]-1 (int32 on the device), none longer than max_seqlen.
    Returns ``(o [T, Hq, d], lse [Hq, T] f32)``."""
    S, n, T = _packing(cu_seqlens, max_seqlen, q)
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    p = kc.shape[0]
    g = geom(S, n, Hq, Hkv, d, p, min(frozen_prefix, p), scale, theta, window)
    dt, cd = _dt(q), _dt(kc)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    ws = _workspace(fwd_packed_workspace_size(g, T, dt, cd), q.device, workspace)
    rc = lib().cart_attn_fwd_packed(ctypes.byref(g), T, _ptr(cu_seqlens), dt, cd, _ptr(q),
                                    _ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(o), _ptr(lse),
                                    _ptr(ws), ws.numel(), _stream(stream, q.device))
    _check("cart_attn_fwd_packed", rc)
    return o, lse


def cart_attn_bwd_packed(q, k, v, kc, vc, o, lse, dout, cu_seqlens, max_seqlen, *,
                         frozen_prefix=1, scale=None, theta=1.0e6, accumulate=False, dq=None,
                         dk=None, dv=None, dkc=None, dvc=None, workspace=None, stream=None,
                         frozen_rows=(), window=0):
    """Backward on packed segments (layouts of cart_attn_fwd_packed).
    Returns ``(dq, dk, dv, dkc, dvc)``; dkc/dvc f32 ``[p, Hkv, d]`` summed
    over the segments, frozen rows exactly 0."""
    S, n, T = _packing(cu_seqlens, max_seqlen, q)
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    p = kc.shape[0]
    g = geom(S, n, Hq, Hkv, d, p, frozen_prefix, scale, theta, window)
    dt, cd = _dt(q), _dt(kc)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dkc is None:
        dkc = (torch.zeros if accumulate else torch.empty)((max(p, 1), Hkv, d),
                                                           dtype=torch.float32, device=q.device)
    if dvc is None:
        dvc = (torch.zeros if accumulate else torch.empty)((max(p, 1), Hkv, d),
                                                           dtype=torch.float32, device=q.device)
    ws = _workspace(bwd_packed_workspace_size(g, T, dt, cd), q.device, workspace)
    rows = list(frozen_rows)
    arr = (ctypes.c_int * max(len(rows), 1))(*rows)
    rc = lib().cart_attn_bwd_packed(ctypes.byref(g), T, _ptr(cu_seqlens), dt, cd, _ptr(q),
                                    _ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(o), _ptr(lse),
                                    _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkc),
                                    _ptr(dvc), arr, len(rows), 1 if accumulate else 0, _ptr(ws),
                                    ws.numel(), _stream(stream, q.device))
    _check("cart_attn_bwd_packed", rc)
    return dq, dk, dv, dkc[:p], dvc[:p]


def decode_workspace_size(B, Hq, Hkv, d, p, rows) -> int:
    return int(lib().cart_attn_decode_workspace_size(B, Hq, Hkv, d, p, rows))


def cart_attn_decode(q, k_new, v_new, kc, vc, k_cache, v_cache, lens, *, scale=None, theta=1.0e6,
                     o=None, workspace=None, stream=None):
    """One decode step.  q ``[B, Hq, d]``, k_new/v_new ``[B, Hkv, d]`` (bf16,
    not rotated), kc/vc ``[p, Hkv, d]`` bf16 shared cartridge, caches
    ``[B, rows, Hkv, d]`` bf16 (modified: row lens[b] receives the new token),
    lens ``[B]`` int32 on the device.  Returns o ``[B, Hq, d]`` bf16."""
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    p = kc.shape[0]
    rows = k_cache.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if lens.dtype != torch.int32:
        raise TypeError("lens must be int32")
    if o is None:
        o = torch.empty_like(q)
    ws = _workspace(decode_workspace_size(B, Hq, Hkv, d, p, rows), q.device, workspace)
    rc = lib().cart_attn_decode(B, Hq, Hkv, d, p, float(scale), float(theta), _ptr(q),
                                _ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(k_cache),
                                _ptr(v_cache), rows, _ptr(lens), _ptr(o), _ptr(ws), ws.numel(),
                                _stream(stream, q.device))
    _check("cart_attn_decode", rc)
    return o


def decode_span_workspace_size(B, span, Hq, Hkv, d, p, rows) -> int:
    return int(lib().cart_attn_decode_span_workspace_size(B, span, Hq, Hkv, d, p, rows))


def cart_attn_decode_span(q, k_new, v_new, kc, vc, k_cache, v_cache, lens, *, scale=None,
                          theta=1.0e6, o=None, workspace=None, stream=None, window=0):
    """Span verify: ``span`` new tokens per conversation in one step.  q
    ``[B, span, Hq, d]``, k_new/v_new ``[B, span, Hkv, d]`` (bf16, not
    rotated); the caches receive the span's rows lens[b] .. lens[b]+span-1.
    Returns o ``[B, span, Hq, d]`` bf16.  ``window`` > 0: token t sees the
    keys at positions p + lens[b] + t - window + 1 .. p + lens[b] + t."""
    B, span, Hq, d = q.shape
    Hkv = k_new.shape[2]
    p = kc.shape[0]
    rows = k_cache.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if lens.dtype != torch.int32:
        raise TypeError("lens must be int32")
    if o is None:
        o = torch.empty_like(q)
    ws = _workspace(decode_span_workspace_size(B, span, Hq, Hkv, d, p, rows), q.device, workspace)
    rc = lib().cart_attn_decode_span(B, span, int(window), Hq, Hkv, d, p, float(scale),
                                     float(theta), _ptr(q),
                                     _ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc),
                                     _ptr(k_cache), _ptr(v_cache), rows, _ptr(lens), _ptr(o),
                                     _ptr(ws), ws.numel(), _stream(stream, q.device))
    _check("cart_attn_decode_span", rc)
    return o


def release() -> None:
    """Destroy this device's helper stream and events (recreated on use)."""
    _check("cart_release", lib().cart_release())


def device_status(clear: bool = True) -> int:
    """Bits set by kernels whose bounded waits gave up (0 = none)."""
    bits = ctypes.c_uint(0)
    rc = lib().cart_device_status(ctypes.byref(bits), 1 if clear else 0)
    if rc not in (0, -7):
        raise CartError("cart_device_status", rc)
    return int(bits.value)


def trace_enable(on: bool = True):
    """Start (clearing earlier records) or stop recording per-launch events."""
    lib().cart_trace_enable(1 if on else 0)


def trace_read(with_times: bool = True):
    """List of (kernel name, device ms or None) for the recorded launches."""
    L = lib()
    out = []
    buf = ctypes.create_string_buffer(32)
    for i in range(L.cart_trace_count()):
        ms = ctypes.c_float(-1.0)
        rc = L.cart_trace_get(i, buf, 32, ctypes.byref(ms) if with_times else None)
        if rc != 0 and with_times:
            raise CartError("cart_trace_get", rc)
        out.append((buf.value.decode(), float(ms.value) if with_times else None))
    return out
