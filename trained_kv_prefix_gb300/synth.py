"""Seeded synthetic inputs for cartridge attention.

This module only draws random numbers and casts them to the storage dtype.
It holds none of the method's arithmetic (no RoPE, no softmax, no masks), so
both the CUDA path and the CPU oracle can take their inputs from here.

Workloads (shapes follow the Cartridges guide, "Semantics": a cartridge is a
per-layer ``[p, kv_head, d]`` key/value pair, real tokens follow it):

* ``tiny``       1 layer, Hq=4, Hkv=2, d=64, p=16 (row 0 frozen), n=32, all f32.
* ``equiv``      Hq=32, Hkv=8, d=128: 512 prefix tokens become the cartridge,
                 256 continuation tokens attend behind it (bf16).
* ``selfstudy``  B=4, Hq=32, Hkv=8, d=128, p=2048, n=1024, bf16 Q/K/V with f32
                 cartridge leaf rows.
* ``decode``     64 conversations behind one p=4096 cartridge, 0..1024 private
                 tokens each, q_seq=1 (bf16).
* ``longctx``    B=1, Hq=64, Hkv=8, d=128, p=8192, n=4096 (bf16, f32 leaves).

Values: ``std * N(0, 1)`` drawn in fp64 by ``numpy.random.default_rng(seed)``
and rounded to nearest-even into the storage dtype.  Both sides read the
stored (rounded) values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ROPE_THETA = 1.0e6


@dataclass(frozen=True)
class TrainShape:
    name: str
    B: int
    n: int
    Hq: int
    Hkv: int
    d: int
    p: int
    frozen_prefix: int = 1
    dtype: str = "bf16"          # Q/K/V/dO storage
    cart_dtype: str = "f32"      # cartridge leaf storage
    seed: int = 0
    qkv_std: float = 0.5
    do_std: float = 1.0e-2
    theta: float = ROPE_THETA

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def pairs_per_head(self) -> int:
        """Visible (query, key) pairs of one (batch, head): every query sees
        all p cartridge rows and is causal over the real tokens."""
        return self.n * self.p + self.n * (self.n + 1) // 2

    def fwd_flops(self) -> float:
        return 4.0 * self.d * self.Hq * self.B * self.pairs_per_head()

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    p: int
    max_private: int
    seed: int = 3
    std: float = 0.5
    theta: float = ROPE_THETA
    fixed_len: tuple = field(default=())

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def cache_rows(self) -> int:
        return self.max_private + 1


TINY = TrainShape("tiny", B=1, n=32, Hq=4, Hkv=2, d=64, p=16, dtype="f32",
                  cart_dtype="f32", seed=0, qkv_std=0.5, do_std=1.0)
EQUIV_P, EQUIV_N = 512, 256
EQUIV = TrainShape("equiv", B=1, n=EQUIV_N, Hq=32, Hkv=8, d=128, p=EQUIV_P,
                   frozen_prefix=1, dtype="bf16", cart_dtype="bf16", seed=1,
                   qkv_std=1.0, do_std=1.0e-2)
SELFSTUDY = TrainShape("selfstudy", B=4, n=1024, Hq=32, Hkv=8, d=128, p=2048,
                       seed=2, qkv_std=0.5, do_std=1.0e-2)
DECODE = DecodeShape("decode", B=64, Hq=32, Hkv=8, d=128, p=4096,
                     max_private=1024, seed=3)
LONGCTX = TrainShape("longctx", B=1, n=4096, Hq=64, Hkv=8, d=128, p=8192,
                     seed=4, qkv_std=0.5, do_std=1.0e-2)

TRAIN_SHAPES = {s.name: s for s in (TINY, EQUIV, SELFSTUDY, LONGCTX)}

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def _draw(rng: np.random.Generator, shape, std: float, dtype: str) -> torch.Tensor:
    x = rng.standard_normal(size=shape) * std
    # fp64 -> storage dtype, round-to-nearest-even (torch cast).
    return torch.from_numpy(x).to(_TORCH_DTYPE[dtype]).contiguous()


def train_inputs(s: TrainShape, seed: int | None = None) -> dict:
    """Q, K, V, dO as ``[B, n, H, d]``; cartridge Kc, Vc as ``[p, Hkv, d]``.

    All tensors live on the CPU; callers move them where they need them."""
    rng = np.random.default_rng(s.seed if seed is None else seed)
    q = _draw(rng, (s.B, s.n, s.Hq, s.d), s.qkv_std, s.dtype)
    k = _draw(rng, (s.B, s.n, s.Hkv, s.d), s.qkv_std, s.dtype)
    v = _draw(rng, (s.B, s.n, s.Hkv, s.d), s.qkv_std, s.dtype)
    kc = _draw(rng, (s.p, s.Hkv, s.d), s.qkv_std, s.cart_dtype)
    vc = _draw(rng, (s.p, s.Hkv, s.d), s.qkv_std, s.cart_dtype)
    do = _draw(rng, (s.B, s.n, s.Hq, s.d), s.do_std, s.dtype)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, do=do)


def packed_lengths(n_max: int, segments: int, seed: int) -> np.ndarray:
    """Segment lengths of a packed group: conversations of uneven length,
    ``U{1..n_max}`` (the longest set to n_max, so the grid bound is met)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, n_max + 1, size=segments)
    lens[int(rng.integers(0, segments))] = n_max
    return lens.astype(np.int32)


def packed_inputs(s: TrainShape, lens, seed: int | None = None) -> dict:
    """Packed segments of the given lengths (the shape's B and n are not
    used): Q, dO ``[T, Hq, d]``, K, V ``[T, Hkv, d]``, cartridge ``[p, Hkv,
    d]``, the int32 table ``cu_seqlens [S + 1]`` and ``max_seqlen``; values
    drawn as in :func:`train_inputs`."""
    lens = np.asarray(lens, dtype=np.int64)
    T = int(lens.sum())
    rng = np.random.default_rng(s.seed if seed is None else seed)
    q = _draw(rng, (T, s.Hq, s.d), s.qkv_std, s.dtype)
    k = _draw(rng, (T, s.Hkv, s.d), s.qkv_std, s.dtype)
    v = _draw(rng, (T, s.Hkv, s.d), s.qkv_std, s.dtype)
    kc = _draw(rng, (s.p, s.Hkv, s.d), s.qkv_std, s.cart_dtype)
    vc = _draw(rng, (s.p, s.Hkv, s.d), s.qkv_std, s.cart_dtype)
    do = _draw(rng, (T, s.Hq, s.d), s.do_std, s.dtype)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, do=do, cu=cu, max_seqlen=int(lens.max(initial=1)))


def token_kv(total: int, Hkv: int, d: int, seed: int, std: float = 1.0):
    """Raw (un-rotated) per-token K and V for a sequence of ``total`` tokens,
    ``[total, Hkv, d]`` fp64 numpy arrays, plus queries for the same tokens at
    the head count chosen by the caller via :func:`token_q`."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal(size=(total, Hkv, d)) * std
    v = rng.standard_normal(size=(total, Hkv, d)) * std
    return k, v, rng


def token_q(rng: np.random.Generator, n: int, Hq: int, d: int, std: float = 1.0):
    return rng.standard_normal(size=(n, Hq, d)) * std


def to_storage(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(_TORCH_DTYPE[dtype]).contiguous()


def decode_inputs(s: DecodeShape, seed: int | None = None) -> dict:
    """Shared cartridge ``[p, Hkv, d]``, private caches ``[B, rows, Hkv, d]``
    (rows = max_private + 1, so the new token always has a slot), lengths
    ``L_b ~ U{0..max_private}`` (int32), query ``[B, Hq, d]`` and the new
    token's K/V ``[B, Hkv, d]``.  All bf16 except the lengths."""
    rng = np.random.default_rng(s.seed if seed is None else seed)
    if s.fixed_len:
        lens = np.asarray(s.fixed_len, dtype=np.int32)
        assert lens.shape == (s.B,)
    else:
        lens = rng.integers(0, s.max_private + 1, size=s.B).astype(np.int32)
    kc = _draw(rng, (s.p, s.Hkv, s.d), s.std, "bf16")
    vc = _draw(rng, (s.p, s.Hkv, s.d), s.std, "bf16")
    k_cache = _draw(rng, (s.B, s.cache_rows, s.Hkv, s.d), s.std, "bf16")
    v_cache = _draw(rng, (s.B, s.cache_rows, s.Hkv, s.d), s.std, "bf16")
    q = _draw(rng, (s.B, s.Hq, s.d), s.std, "bf16")
    k_new = _draw(rng, (s.B, s.Hkv, s.d), s.std, "bf16")
    v_new = _draw(rng, (s.B, s.Hkv, s.d), s.std, "bf16")
    return dict(q=q, k_new=k_new, v_new=v_new, kc=kc, vc=vc,
                k_cache=k_cache, v_cache=v_cache,
                lens=torch.from_numpy(lens))


def decode_span_inputs(s: DecodeShape, span: int, seed: int | None = None) -> dict:
    """As decode_inputs for ``span`` new tokens per conversation: query
    ``[B, span, Hq, d]``, new K/V ``[B, span, Hkv, d]``, lengths
    ``L_b ~ U{0..rows - span}`` (or ``s.fixed_len``) so the span fits."""
    rng = np.random.default_rng(s.seed if seed is None else seed)
    if s.fixed_len:
        lens = np.asarray(s.fixed_len, dtype=np.int32)
        assert lens.shape == (s.B,) and (lens + span <= s.cache_rows).all()
    else:
        lens = rng.integers(0, s.cache_rows - span + 1, size=s.B).astype(np.int32)
    kc = _draw(rng, (s.p, s.Hkv, s.d), s.std, "bf16")
    vc = _draw(rng, (s.p, s.Hkv, s.d), s.std, "bf16")
    k_cache = _draw(rng, (s.B, s.cache_rows, s.Hkv, s.d), s.std, "bf16")
    v_cache = _draw(rng, (s.B, s.cache_rows, s.Hkv, s.d), s.std, "bf16")
    q = _draw(rng, (s.B, span, s.Hq, s.d), s.std, "bf16")
    k_new = _draw(rng, (s.B, span, s.Hkv, s.d), s.std, "bf16")
    v_new = _draw(rng, (s.B, span, s.Hkv, s.d), s.std, "bf16")
    return dict(q=q, k_new=k_new, v_new=v_new, kc=kc, vc=vc,
                k_cache=k_cache, v_cache=v_cache,
                lens=torch.from_numpy(lens))


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a stored tensor to an fp64 numpy array."""
    return t.detach().cpu().to(torch.float64).contiguous().numpy()
