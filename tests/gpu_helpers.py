"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
on seeded inputs and compare with the fp64 oracle.

Tolerances (stated for cartridge attention with bf16 operands and f32
accumulation):
  forward output   max-abs 1e-2 and relative-L2 5e-3
  dQ, dK, dV, dKc, dVc   relative-L2 1e-2
  frozen cartridge rows  exactly 0.0
  log-sum-exp      max-abs 2e-2 (a by-product the backward consumes; the
                   logits carry bf16 rounding of q and k, ~2^-9 relative, on
                   values of magnitude <~ 4, so a few 1e-3 is expected)
relL2(x, y) = ||x - y||_2 / ||y||_2 over the whole tensor, y the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from trained_kv_prefix_gb300 import cartattn, synth

FWD_MAXABS = 1e-2
FWD_RELL2 = 5e-3
GRAD_RELL2 = 1e-2
LSE_MAXABS = 2e-2


def rel_l2(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = np.linalg.norm(y.ravel())
    return float(np.linalg.norm((x - y).ravel()) / (den if den > 0 else 1.0))


def max_abs(x, y) -> float:
    return float(np.abs(np.asarray(x, np.float64) - np.asarray(y, np.float64)).max())


def to_gpu(d: dict) -> dict:
    return {k: v.cuda() for k, v in d.items()}


def run_train_gpu(s: synth.TrainShape, inp: dict, *, bwd=True, frozen_prefix=None, accumulate=False,
                  dkc0=None, dvc0=None, frozen_rows=None, window=0):
    fp = s.frozen_prefix if frozen_prefix is None else frozen_prefix
    g = to_gpu(inp)
    o, lse = cartattn.cart_attn_fwd(g["q"], g["k"], g["v"], g["kc"], g["vc"], frozen_prefix=fp,
                                    theta=s.theta, window=window)
    out = dict(o=o, lse=lse)
    if bwd:
        dkc = dkc0.clone().cuda() if dkc0 is not None else None
        dvc = dvc0.clone().cuda() if dvc0 is not None else None
        dq, dk, dv, dkc, dvc = cartattn.cart_attn_bwd(
            g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse, g["do"], frozen_prefix=fp,
            theta=s.theta, accumulate=accumulate, dkc=dkc, dvc=dvc, frozen_rows=frozen_rows,
            window=window)
        out.update(dq=dq, dk=dk, dv=dv, dkc=dkc, dvc=dvc)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0, "a kernel reported a timeout"
    return {k: synth.f64(v) for k, v in out.items()}


def oracle_train(s: synth.TrainShape, inp: dict, *, bwd=True, frozen_prefix=None, heads=None,
                 rows=None, kv_heads=None, bwd_rows=None, frozen_rows=(), window=0):
    fp = s.frozen_prefix if frozen_prefix is None else frozen_prefix
    a = {k: synth.f64(v) for k, v in inp.items()}
    o, lse = oracle.fwd(a["q"], a["k"], a["v"], a["kc"], a["vc"], frozen_prefix=fp,
                        theta=s.theta, heads=heads, rows=rows, window=window)
    ref = dict(o=o, lse=lse)
    if bwd:
        dq, dk, dv, dkc, dvc = oracle.bwd(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["do"],
                                          frozen_prefix=fp, theta=s.theta, kv_heads=kv_heads,
                                          rows=bwd_rows, frozen_rows=frozen_rows, window=window)
        ref.update(dq=dq, dk=dk, dv=dv, dkc=dkc, dvc=dvc)
    return ref


def check_fwd(got, ref, sl=(Ellipsis,), lse_sl=(Ellipsis,)):
    o, r = got["o"][sl], ref["o"][sl]
    assert not np.isnan(r).any()
    assert max_abs(o, r) <= FWD_MAXABS, max_abs(o, r)
    assert rel_l2(o, r) <= FWD_RELL2, rel_l2(o, r)
    assert max_abs(got["lse"][lse_sl], ref["lse"][lse_sl]) <= LSE_MAXABS


def check_grads(got, ref, frozen, names=("dq", "dk", "dv", "dkc", "dvc"), sls=None):
    sls = sls or {}
    for nme in names:
        sl = sls.get(nme, (Ellipsis,))
        x, y = got[nme][sl], ref[nme][sl]
        if nme in ("dkc", "dvc"):
            assert (got[nme][:frozen] == 0.0).all(), f"{nme}: frozen rows not exactly zero"
            if y.shape[0] > frozen and np.linalg.norm(y[frozen:]) > 0:
                assert rel_l2(x[frozen:], y[frozen:]) <= GRAD_RELL2, (nme, rel_l2(x[frozen:], y[frozen:]))
            continue
        assert not np.isnan(y).any(), nme
        assert rel_l2(x, y) <= GRAD_RELL2, (nme, rel_l2(x, y))


def oracle_group_parallel(s: synth.TrainShape, inp: dict, g: int, *, chunk_rows: int = 128,
                          workers: int | None = None):
    """fp64 oracle for every output of kv-head group ``g`` (its G query heads,
    every query row), the cartridge gradient of that group included.

    The group is an independent problem with Hq = G and Hkv = 1 (query head h
    reads kv head h // G), so its inputs are sliced out and the loss
    sum(dout * o) is split into query-row ranges run on host threads: o, lse
    and dq of a row come from the range holding it, and the key, value and
    cartridge gradients are the sums of the ranges' contributions (the loss
    is a sum over query rows).  The oracle's C code runs without the GIL.
    Returns arrays shaped like the full problem's outputs restricted to the
    group (heads g*G .. g*G + G - 1, kv head g)."""
    import concurrent.futures as cf
    import os

    G = s.Hq // s.Hkv
    hs = slice(g * G, (g + 1) * G)
    a = {k: synth.f64(v) for k, v in inp.items()}
    q, do = np.ascontiguousarray(a["q"][:, :, hs]), np.ascontiguousarray(a["do"][:, :, hs])
    k, v = np.ascontiguousarray(a["k"][:, :, g:g + 1]), np.ascontiguousarray(a["v"][:, :, g:g + 1])
    kc, vc = np.ascontiguousarray(a["kc"][:, g:g + 1]), np.ascontiguousarray(a["vc"][:, g:g + 1])
    ranges = [(lo, min(lo + chunk_rows, s.n)) for lo in range(0, s.n, chunk_rows)]

    def one(rg):
        o, lse = oracle.fwd(q, k, v, kc, vc, frozen_prefix=s.frozen_prefix, theta=s.theta,
                            rows=rg)
        grads = oracle.bwd(q, k, v, kc, vc, do, frozen_prefix=s.frozen_prefix, theta=s.theta,
                           rows=rg)
        return rg, o, lse, grads

    ref = dict(o=np.empty(q.shape), lse=np.empty((s.B, G, s.n)), dq=np.empty(q.shape),
               dk=np.zeros(k.shape), dv=np.zeros(v.shape), dkc=np.zeros(kc.shape),
               dvc=np.zeros(vc.shape))
    with cf.ThreadPoolExecutor(max_workers=workers or os.cpu_count()) as ex:
        for (lo, hi), o, lse, (dq, dk, dv, dkc, dvc) in ex.map(one, ranges):
            ref["o"][:, lo:hi] = o[:, lo:hi]
            ref["lse"][:, :, lo:hi] = lse[:, :, lo:hi]
            ref["dq"][:, lo:hi] = dq[:, lo:hi]
            ref["dk"] += dk
            ref["dv"] += dv
            ref["dkc"] += dkc
            ref["dvc"] += dvc
    return ref
