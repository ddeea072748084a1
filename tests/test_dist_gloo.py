"""Data-parallel host path on CPU with gloo, world size 2: sharding the packed
batch across ranks and all-reducing the cartridge gradients reproduces the
single-process gradient of the whole batch (packed == sequential); the
max-over-ranks timing reduction and the conversation sharding are exact."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        import oracle
        from trained_kv_prefix_gb300 import dist as cdist
        assert cdist.init_from_env("gloo")
        rng = np.random.default_rng(3)
        B, n, Hq, Hkv, d, p = 4, 6, 4, 2, 8, 5
        P = {k: rng.standard_normal(s) * 0.5 for k, s in dict(
            q=(B, n, Hq, d), k=(B, n, Hkv, d), v=(B, n, Hkv, d), kc=(p, Hkv, d), vc=(p, Hkv, d),
            do=(B, n, Hq, d)).items()}
        lo, hi = cdist.shard(B, rank, world)
        sl = slice(lo, hi)
        _, _, _, dkc, dvc = oracle.bwd(P["q"][sl], P["k"][sl], P["v"][sl], P["kc"], P["vc"],
                                       P["do"][sl])
        tk, tv = torch.from_numpy(dkc.copy()), torch.from_numpy(dvc.copy())
        cdist.allreduce_cartridge_grads(tk, tv)
        mx = cdist.max_over_ranks([float(rank), 10.0 - rank], "cpu")
        cdist.barrier()
        if rank == 0:
            _, _, _, fk, fv = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
            q.put(("ok", float(np.abs(tk.numpy() - fk).max()), float(np.abs(tv.numpy() - fv).max()),
                   bool((tk.numpy()[0] == 0).all()), mx))
        import torch.distributed as tdist
        tdist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put(("err", repr(e)))


def test_shard_covers_everything_once():
    from trained_kv_prefix_gb300 import dist as cdist
    for total in (1, 7, 64):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                lo, hi = cdist.shard(total, r, world)
                seen.extend(range(lo, hi))
            assert seen == list(range(total))


def test_two_rank_cartridge_gradient_allreduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("gloo worker did not finish")
    res = q.get(timeout=5)
    assert res[0] == "ok", res
    _, ek, ev, frozen_zero, mx = res
    assert ek < 1e-12 and ev < 1e-12
    assert frozen_zero
    assert mx == [1.0, 10.0]
