"""A second, independent formulation of cartridge attention built from library
routines, used only to pin the oracle (never the CUDA path directly).

* RoPE is written as a complex multiplication: the pair (x_j, x_{j+d/2}) is the
  complex number x_j + i x_{j+d/2}, rotated by exp(i * pos * theta^(-2j/d)).
  (Rotate-half pairing, Qwen-style; angle per pair as in the oracle's reading.)
* Attention is ``torch.nn.functional.scaled_dot_product_attention`` in fp64
  with an explicit boolean mask matrix built from the end-aligned rule
  ``key j visible from query i  <=>  j <= i + (kv_seq - q_seq)``
  (Cartridges guide, "Semantics", attention bullet).
* GQA expands kv heads with ``repeat_interleave`` (contiguous groups).
* Gradients come from autograd through all of the above.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def rope_complex(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """x ``[..., L, d]`` (fp64), pos ``[L]`` -> rotated copy (differentiable)."""
    d = x.shape[-1]
    h = d // 2
    j = torch.arange(h, dtype=torch.float64)
    inv_freq = theta ** (-2.0 * j / d)
    ang = pos.to(torch.float64)[:, None] * inv_freq[None, :]          # [L, h]
    rot = torch.polar(torch.ones_like(ang), ang)                       # e^{i ang}
    z = torch.complex(x[..., :h], x[..., h:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def end_aligned_mask(q_seq: int, kv_seq: int, window: int = 0) -> torch.Tensor:
    """Key j visible from query i; with a sliding window W > 0 also
    i + (kv_seq - q_seq) - j < W (the W most recent keys, counting itself)."""
    i = torch.arange(q_seq)[:, None]
    j = torch.arange(kv_seq)[None, :]
    vis = j <= i + (kv_seq - q_seq)
    if window > 0:
        vis = vis & (i + (kv_seq - q_seq) - j < window)
    return vis


def cartridge_attention(q, k, v, kc, vc, *, theta=1.0e6, scale=None, window=0):
    """All inputs torch fp64 in the oracle's layouts:
    q ``[B, n, Hq, d]``, k/v ``[B, n, Hkv, d]``, kc/vc ``[p, Hkv, d]``.
    Returns (o ``[B, n, Hq, d]``, lse ``[B, Hq, n]``)."""
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    p = kc.shape[0]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    pos = torch.arange(p, p + n)
    qh = rope_complex(q.permute(0, 2, 1, 3), pos, theta)              # [B, Hq, n, d]
    kh = rope_complex(k.permute(0, 2, 1, 3), pos, theta)              # [B, Hkv, n, d]
    vh = v.permute(0, 2, 1, 3)
    kcb = kc.permute(1, 0, 2).unsqueeze(0).expand(B, Hkv, p, d)
    vcb = vc.permute(1, 0, 2).unsqueeze(0).expand(B, Hkv, p, d)
    K = torch.cat([kcb, kh], dim=2).repeat_interleave(G, dim=1)       # [B, Hq, kv, d]
    V = torch.cat([vcb, vh], dim=2).repeat_interleave(G, dim=1)
    mask = end_aligned_mask(n, p + n, window)
    o = F.scaled_dot_product_attention(qh, K, V, attn_mask=mask, scale=scale)
    logits = torch.matmul(qh, K.transpose(-1, -2)) * scale
    lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    return o.permute(0, 2, 1, 3), lse


def cartridge_grads(q, k, v, kc, vc, dout, *, frozen_prefix=1, theta=1.0e6, scale=None,
                    window=0):
    """Autograd gradients of sum(dout * o).  Frozen rows are held constant (the
    sink rows are not leaves), so their gradient is reported as exactly 0."""
    q = q.clone().requires_grad_(True)
    k = k.clone().requires_grad_(True)
    v = v.clone().requires_grad_(True)
    kt = kc[frozen_prefix:].clone().requires_grad_(True)
    vt = vc[frozen_prefix:].clone().requires_grad_(True)
    kcat = torch.cat([kc[:frozen_prefix], kt], dim=0)
    vcat = torch.cat([vc[:frozen_prefix], vt], dim=0)
    o, _ = cartridge_attention(q, k, v, kcat, vcat, theta=theta, scale=scale, window=window)
    (o * dout).sum().backward()
    dkc = torch.zeros_like(kc)
    dvc = torch.zeros_like(vc)
    dkc[frozen_prefix:] = kt.grad
    dvc[frozen_prefix:] = vt.grad
    return q.grad, k.grad, v.grad, dkc, dvc


def packed_attention(q, k, v, kc, vc, cu_seqlens, *, theta=1.0e6, scale=None, window=0):
    """Packed segments as ONE attention over the packed token axis: q
    ``[T, Hq, d]``, k/v ``[T, Hkv, d]``, keys = the p cartridge rows then all
    T tokens.  The mask is block diagonal over the segments: token i of
    segment s sees every cartridge row and the tokens 0..i of segment s;
    RoPE positions restart at p in every segment.  Returns (o ``[T, Hq, d]``,
    lse ``[Hq, T]``)."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    p = kc.shape[0]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    cu = [int(x) for x in cu_seqlens]
    seg = torch.zeros(T, dtype=torch.long)
    local = torch.zeros(T, dtype=torch.long)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        seg[a:b] = s
        local[a:b] = torch.arange(b - a)
    pos = p + local
    qh = rope_complex(q.permute(1, 0, 2), pos, theta)                  # [Hq, T, d]
    kh = rope_complex(k.permute(1, 0, 2), pos, theta)                  # [Hkv, T, d]
    K = torch.cat([kc.permute(1, 0, 2), kh], dim=1).repeat_interleave(G, dim=0)
    V = torch.cat([vc.permute(1, 0, 2), v.permute(1, 0, 2)], dim=1).repeat_interleave(G, dim=0)
    same = seg[:, None] == seg[None, :]
    causal = local[None, :] <= local[:, None]
    mask = torch.cat([torch.ones(T, p, dtype=torch.bool), same & causal], dim=1)  # [T, p + T]
    if window > 0:  # positions: cartridge row j at j, token i of a segment at p + i
        kpos = torch.cat([torch.arange(p), pos])
        mask = mask & (pos[:, None] - kpos[None, :] < window)
    o = F.scaled_dot_product_attention(qh, K, V, attn_mask=mask, scale=scale)
    logits = torch.matmul(qh, K.transpose(-1, -2)) * scale
    lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    return o.permute(1, 0, 2), lse


def packed_grads(q, k, v, kc, vc, dout, cu_seqlens, *, frozen_prefix=1, theta=1.0e6,
                 scale=None, window=0):
    """Autograd gradients of sum(dout * o) through ``packed_attention``, the
    sink rows held constant (gradient reported as exactly 0)."""
    q = q.clone().requires_grad_(True)
    k = k.clone().requires_grad_(True)
    v = v.clone().requires_grad_(True)
    kt = kc[frozen_prefix:].clone().requires_grad_(True)
    vt = vc[frozen_prefix:].clone().requires_grad_(True)
    o, _ = packed_attention(q, k, v, torch.cat([kc[:frozen_prefix], kt]),
                            torch.cat([vc[:frozen_prefix], vt]), cu_seqlens, theta=theta,
                            scale=scale, window=window)
    (o * dout).sum().backward()
    dkc = torch.zeros_like(kc)
    dvc = torch.zeros_like(vc)
    dkc[frozen_prefix:] = kt.grad
    dvc[frozen_prefix:] = vt.grad
    return q.grad, k.grad, v.grad, dkc, dvc
