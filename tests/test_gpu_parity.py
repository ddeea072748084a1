"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
seeded inputs.  Small geometries span several 128-row tiles with ragged tails
and cover the degenerate cases (p = 0, sink-only cartridge, n = 1, MHA,
G = 8, f32 inputs); the full workloads are checked on sampled outputs or
properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
from tests import gpu_helpers as gh
from trained_kv_prefix_gb300 import cartattn, synth

pytestmark = pytest.mark.gpu


def _shape(name, B, n, Hq, Hkv, d, p, dtype="bf16", cart="f32", frozen=1, seed=100, do_std=1.0):
    return synth.TrainShape(name, B=B, n=n, Hq=Hq, Hkv=Hkv, d=d, p=p, frozen_prefix=frozen,
                            dtype=dtype, cart_dtype=cart, seed=seed, qkv_std=0.5, do_std=do_std)


SMALL = [
    synth.TINY,
    _shape("p0", 2, 200, 8, 2, 128, 0, frozen=0, seed=101),
    _shape("sink_only", 1, 130, 4, 2, 128, 1, seed=102),
    _shape("mha_ragged_p", 2, 70, 2, 2, 128, 130, seed=103),
    _shape("g8_d64", 1, 257, 8, 1, 64, 300, seed=104),
    _shape("n1", 3, 1, 4, 2, 128, 256, seed=105),
    _shape("multi_tile", 1, 384, 8, 2, 128, 513, seed=106),
    _shape("bf16_cart", 2, 160, 4, 1, 128, 200, cart="bf16", seed=107),
    _shape("f32_d128", 1, 150, 4, 2, 128, 140, dtype="f32", seed=108),
    _shape("frozen3", 1, 100, 4, 2, 64, 40, frozen=3, seed=109),
    # an odd group (3 heads per kv head): the forward pairs query tiles of
    # one head instead of one tile of two heads; ragged n, 3 query tiles
    _shape("g3_odd_tiles", 2, 300, 6, 2, 128, 140, seed=113),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from trained_kv_prefix_gb300 import build
    build.build()
    cartattn.device_status(clear=True)


@pytest.mark.parametrize("s", SMALL, ids=[s.name for s in SMALL])
def test_train_parity_small(s):
    inp = synth.train_inputs(s)
    got = gh.run_train_gpu(s, inp)
    ref = gh.oracle_train(s, inp)
    gh.check_fwd(got, ref)
    gh.check_grads(got, ref, s.frozen_prefix)


def test_bwd_accumulate_mode():
    s = _shape("acc", 1, 96, 4, 2, 64, 70, seed=110)
    inp = synth.train_inputs(s)
    rng = np.random.default_rng(5)
    dkc0 = torch.from_numpy(rng.standard_normal((s.p, s.Hkv, s.d))).float()
    dvc0 = torch.from_numpy(rng.standard_normal((s.p, s.Hkv, s.d))).float()
    got = gh.run_train_gpu(s, inp, accumulate=True, dkc0=dkc0, dvc0=dvc0)
    ref = gh.oracle_train(s, inp)
    ref["dkc"] = ref["dkc"] + dkc0.double().numpy()
    ref["dvc"] = ref["dvc"] + dvc0.double().numpy()
    ref["dkc"][: s.frozen_prefix] = 0.0
    ref["dvc"][: s.frozen_prefix] = 0.0
    gh.check_grads(got, ref, s.frozen_prefix, names=("dkc", "dvc"))


@pytest.mark.parametrize("accumulate", [False, True])
def test_bwd_composed_cartridge_parts(accumulate):
    """Three parts concatenated along the rows (rows 0, 130 and 300 are their
    sinks; 130 and 300 sit inside tiles, 300 in the ragged last tile): the
    listed sinks get exactly 0.0 in both modes, every other row matches the
    oracle."""
    s = _shape("parts", 2, 140, 8, 2, 128, 333, seed=112)
    sinks = (130, 300)
    inp = synth.train_inputs(s)
    kw = {}
    if accumulate:
        rng = np.random.default_rng(6)
        kw = dict(accumulate=True,
                  dkc0=torch.from_numpy(rng.standard_normal((s.p, s.Hkv, s.d))).float(),
                  dvc0=torch.from_numpy(rng.standard_normal((s.p, s.Hkv, s.d))).float())
    got = gh.run_train_gpu(s, inp, frozen_rows=sinks, **kw)
    ref = gh.oracle_train(s, inp, frozen_rows=sinks)
    if accumulate:
        ref["dkc"] = ref["dkc"] + kw["dkc0"].double().numpy()
        ref["dvc"] = ref["dvc"] + kw["dvc0"].double().numpy()
    frozen = [0, *sinks]
    for nme in ("dkc", "dvc"):
        assert (got[nme][frozen] == 0.0).all(), f"{nme}: a part's sink is not exactly zero"
        ref[nme][frozen] = 0.0
    gh.check_fwd(got, ref)
    gh.check_grads(got, ref, 1)


PACKED = [
    # (shape: heads, d, p, dtypes; B and n unused), segment lengths, max_seqlen
    (_shape("packed_ragged", 0, 0, 8, 2, 128, 300, seed=120), (130, 1, 0, 257, 64), 257),
    (_shape("packed_g8_d64", 0, 0, 8, 1, 64, 129, seed=121), (200, 77, 128), 256),
    (_shape("packed_p0", 0, 0, 4, 2, 128, 0, frozen=0, seed=122), (40, 300, 129), 300),
    (_shape("packed_f32", 0, 0, 4, 2, 128, 140, dtype="f32", seed=123), (100, 33, 150), 150),
    (_shape("packed_bf16_cart", 0, 0, 4, 1, 128, 200, cart="bf16", seed=124), (1, 384, 2), 384),
]


def _run_packed(s, inp, max_seqlen, **kw):
    g = gh.to_gpu({k: v for k, v in inp.items() if k != "max_seqlen"})
    o, lse = cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], g["cu"],
                                           max_seqlen, frozen_prefix=s.frozen_prefix,
                                           theta=s.theta)
    dq, dk, dv, dkc, dvc = cartattn.cart_attn_bwd_packed(
        g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse, g["do"], g["cu"], max_seqlen,
        frozen_prefix=s.frozen_prefix, theta=s.theta, **kw)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    out = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dkc=dkc, dvc=dvc)
    return {k: synth.f64(v) for k, v in out.items()}


@pytest.mark.parametrize("case", PACKED, ids=[c[0].name for c in PACKED])
def test_packed_parity(case):
    """Packed segments (ragged, empty, one-token, exactly one tile, a bound
    above the longest) against the oracle's per-segment definition."""
    s, lens, max_seqlen = case
    inp = synth.packed_inputs(s, lens)
    got = _run_packed(s, inp, max_seqlen)
    a = {k: synth.f64(v) for k, v in inp.items() if k not in ("cu", "max_seqlen")}
    cu = inp["cu"].numpy()
    o, lse = oracle.fwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], cu,
                               frozen_prefix=s.frozen_prefix, theta=s.theta)
    ref = dict(o=o, lse=lse)
    ref.update(zip(("dq", "dk", "dv", "dkc", "dvc"),
                   oracle.bwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["do"], cu,
                                     frozen_prefix=s.frozen_prefix, theta=s.theta)))
    gh.check_fwd(got, ref)
    gh.check_grads(got, ref, s.frozen_prefix)


def test_packed_bad_table_sets_status_bit():
    """A segment table that breaks its rules (falling, a segment longer than
    the bound, not ending at the token count) is reported in device status
    bit 6; the kernels clamp it, so every access stays inside the tensors."""
    s = _shape("packed_bad", 0, 0, 4, 2, 128, 130, seed=126)
    inp = synth.packed_inputs(s, (40, 60, 28))
    g = gh.to_gpu({k: v for k, v in inp.items() if k != "max_seqlen"})
    cartattn.device_status(clear=True)
    for bad in ((0, 50, 30, 128), (0, 100, 110, 128), (0, 40, 100, 127)):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        o, lse = cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], cu, 64)
        cartattn.cart_attn_bwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse, g["do"],
                                      cu, 64)
        torch.cuda.synchronize()
        assert cartattn.device_status(clear=True) == 1 << 6, bad
    # a good table afterwards: no bit
    cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], g["cu"], 60)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0


def test_packed_equal_segments_match_the_batch_bitwise():
    """Equal-length packed segments run the same tiles as the [B, n] batch:
    every output is bit for bit the batched call's (the ragged tails read the
    next segment's rows instead of zeros, which the masks remove exactly)."""
    s = _shape("packed_vs_batch", 3, 200, 8, 2, 128, 257, seed=125)
    inp = synth.train_inputs(s)
    batch = gh.run_train_gpu(s, inp)
    T = s.B * s.n
    flat = {k: inp[k].reshape(T, *inp[k].shape[2:]) for k in ("q", "k", "v", "do")}
    flat.update(kc=inp["kc"], vc=inp["vc"], cu=torch.arange(0, T + 1, s.n, dtype=torch.int32))
    got = _run_packed(s, flat, s.n)
    for k in ("o", "dq", "dk", "dv"):
        np.testing.assert_array_equal(got[k], batch[k].reshape(T, *batch[k].shape[2:]), err_msg=k)
    np.testing.assert_array_equal(got["lse"], batch["lse"].transpose(1, 0, 2).reshape(s.Hq, T))
    np.testing.assert_array_equal(got["dkc"], batch["dkc"])
    np.testing.assert_array_equal(got["dvc"], batch["dvc"])


WINDOWS = [
    # (shape, window): p = 333, n = 300 -> query positions 333..632
    (_shape("win1", 1, 300, 8, 2, 128, 333, seed=130), 1),          # itself only
    (_shape("win100", 2, 300, 8, 2, 128, 333, seed=131), 100),      # real keys only
    (_shape("win450", 1, 300, 8, 2, 128, 333, seed=132), 450),      # cuts the cartridge
    (_shape("win700_d64", 1, 300, 4, 1, 64, 333, seed=133), 700),   # cuts it for late rows
    (_shape("win200_ragged", 2, 130, 4, 2, 128, 70, seed=134), 200),  # sink cut for late rows
]


@pytest.mark.parametrize("case", WINDOWS, ids=[c[0].name for c in WINDOWS])
def test_window_parity(case):
    """Sliding window over the concatenated sequence (cartridge row j at
    position j): the window cuts through the cartridge and its sink; rows no
    query reaches get exactly zero gradient."""
    s, window = case
    inp = synth.train_inputs(s)
    got = gh.run_train_gpu(s, inp, window=window)
    ref = gh.oracle_train(s, inp, window=window)
    gh.check_fwd(got, ref)
    gh.check_grads(got, ref, s.frozen_prefix)
    unseen = max(0, s.p - window + 1)  # cartridge rows before the first query's window
    for nme in ("dkc", "dvc"):
        assert (got[nme][:unseen] == 0.0).all(), nme


def test_window_wider_than_the_sequence_is_bitwise_no_window():
    s = _shape("win_wide", 2, 200, 8, 2, 128, 257, seed=135)
    inp = synth.train_inputs(s)
    a = gh.run_train_gpu(s, inp)
    b = gh.run_train_gpu(s, inp, window=s.p + s.n)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


REUSE_CASES = [
    # (name, B, n, Hq, Hkv, d, p, dtype, cart dtype, window)
    ("reuse_bf16", 2, 300, 8, 2, 128, 200, "bf16", "f32", 0),
    ("reuse_bf16_cartbf16", 1, 257, 4, 1, 64, 129, "bf16", "bf16", 0),
    ("reuse_f32", 1, 130, 4, 2, 64, 64, "f32", "f32", 0),
    ("reuse_window", 2, 200, 8, 2, 128, 150, "bf16", "f32", 96),
]


@pytest.mark.parametrize("case", REUSE_CASES, ids=[c[0] for c in REUSE_CASES])
def test_bwd_reusing_the_forward_workspace_is_bitwise_bwd(case):
    """cart_attn_bwd_reuse reads the forward's rotated Q / K, table and bf16
    copies: its gradients equal cart_attn_bwd's bit for bit, and the oracle's
    at the gradient tolerance."""
    name, B, n, Hq, Hkv, d, p, dt, cdt, window = case
    s = synth.TrainShape(name, B=B, n=n, Hq=Hq, Hkv=Hkv, d=d, p=p, dtype=dt, cart_dtype=cdt,
                         seed=151, qkv_std=0.5, do_std=1.0)
    inp = synth.train_inputs(s)
    g = gh.to_gpu(inp)
    geom = cartattn.geom(B, n, Hq, Hkv, d, p, s.frozen_prefix, None, s.theta, window)
    ws_f = torch.empty(cartattn.fwd_workspace_size(geom, cartattn._dt(g["q"]),
                                                   cartattn._dt(g["kc"])),
                       dtype=torch.uint8, device="cuda")
    o, lse = cartattn.cart_attn_fwd(g["q"], g["k"], g["v"], g["kc"], g["vc"], theta=s.theta,
                                    window=window, workspace=ws_f)
    plain = cartattn.cart_attn_bwd(g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse, g["do"],
                                   theta=s.theta, window=window)
    reuse = cartattn.cart_attn_bwd(g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse, g["do"],
                                   theta=s.theta, window=window, fwd_workspace=ws_f)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    for nme, x, y in zip(("dq", "dk", "dv", "dkc", "dvc"), plain, reuse):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), nme
    got = {k: synth.f64(v) for k, v in zip(("dq", "dk", "dv", "dkc", "dvc"), reuse)}
    ref = gh.oracle_train(s, inp, window=window)
    gh.check_grads(got, ref, s.frozen_prefix)


def test_packed_window_parity():
    s = _shape("packed_win", 0, 0, 8, 2, 128, 300, seed=136)
    lens, window = (130, 1, 0, 257, 64), 180
    inp = synth.packed_inputs(s, lens)
    g = gh.to_gpu({k: v for k, v in inp.items() if k != "max_seqlen"})
    o, lse = cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], g["cu"], 257,
                                           window=window)
    grads = cartattn.cart_attn_bwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse,
                                          g["do"], g["cu"], 257, window=window)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    got = {k: synth.f64(v) for k, v in zip(("o", "lse", "dq", "dk", "dv", "dkc", "dvc"),
                                           (o, lse, *grads))}
    a = {k: synth.f64(v) for k, v in inp.items() if k not in ("cu", "max_seqlen")}
    cu = inp["cu"].numpy()
    ref = dict(zip(("o", "lse"), oracle.fwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], cu,
                                                   window=window)))
    ref.update(zip(("dq", "dk", "dv", "dkc", "dvc"),
                   oracle.bwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["do"], cu,
                                     window=window)))
    gh.check_fwd(got, ref)
    gh.check_grads(got, ref, 1)


def test_release_then_backward_again():
    """cart_release drops the helper stream; the next backward recreates it
    and gives the same bits."""
    s = _shape("release", 1, 140, 4, 2, 128, 130, seed=127)
    inp = synth.train_inputs(s)
    a = gh.run_train_gpu(s, inp)
    cartattn.release()
    b = gh.run_train_gpu(s, inp)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_backward_is_deterministic():
    s = _shape("det", 2, 200, 8, 2, 128, 300, seed=111)
    inp = synth.train_inputs(s)
    a = gh.run_train_gpu(s, inp)
    b = gh.run_train_gpu(s, inp)
    for k in ("o", "lse", "dq", "dk", "dv", "dkc", "dvc"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("d", [64, 128])
def test_f32_leaves_equal_cache_write_then_bf16_path(d):
    """Given f32 cartridge leaves, the forward's prep launch writes their
    bf16 copy itself.  That copy must be the bytes cart_write_to_cache
    writes (round to nearest even, pinned bit for bit elsewhere): the
    forward and the backward that reads the forward's workspace must then
    equal the bf16-cartridge path fed by cart_write_to_cache, bit for bit."""
    s = _shape(f"leaves_d{d}", 2, 200, 8, 2, d, 333, seed=115)
    g = gh.to_gpu(synth.train_inputs(s))
    assert g["kc"].dtype == torch.float32
    geom = cartattn.geom(s.B, s.n, s.Hq, s.Hkv, s.d, s.p, s.frozen_prefix, None, s.theta)
    kcb = torch.empty(g["kc"].shape, dtype=torch.bfloat16, device="cuda")
    vcb = torch.empty_like(kcb)
    cartattn.cart_write_to_cache(g["kc"], g["vc"], kcb, vcb)
    runs = []
    for kc, vc, cd in ((g["kc"], g["vc"], cartattn.CART_F32), (kcb, vcb, cartattn.CART_BF16)):
        ws = torch.empty(cartattn.fwd_workspace_size(geom, cartattn.CART_BF16, cd),
                         dtype=torch.uint8, device="cuda")
        o, lse = cartattn.cart_attn_fwd(g["q"], g["k"], g["v"], kc, vc, theta=s.theta,
                                        workspace=ws)
        grads = cartattn.cart_attn_bwd(g["q"], g["k"], g["v"], kc, vc, o, lse, g["do"],
                                       theta=s.theta, fwd_workspace=ws)
        runs.append((o, lse) + tuple(grads))
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    for nme, x, y in zip(("o", "lse", "dq", "dk", "dv", "dkc", "dvc"), *runs):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), nme


def test_chained_launches_keep_stream_order_over_reused_memory():
    """The cache write, the preps and the forward are launched as
    programmatic dependents of the launch before them.  Memory that a
    caching allocator hands out again on the same stream must still see
    plain stream order: (1) the cache write reads f32 leaves from a buffer
    freed right after the call, and the forward's workspace is then carved
    from that memory (the prep writes it); (2) the forward reads V from a
    buffer freed right after the call, and the backward's workspace is then
    carved from it (the forward lets the backward's prep launch once its
    loads are issued).  Both must give the fresh-buffer results bit for bit."""
    s = _shape("reused_mem", 2, 256, 8, 2, 128, 300, seed=114)
    g = gh.to_gpu(synth.train_inputs(s))
    geom = cartattn.geom(s.B, s.n, s.Hq, s.Hkv, s.d, s.p, s.frozen_prefix, None, s.theta)
    wf = cartattn.fwd_workspace_size(geom, cartattn.CART_BF16, cartattn.CART_BF16)
    wb = cartattn.bwd_reuse_workspace_size(geom, cartattn.CART_BF16, cartattn.CART_BF16)
    kcb = torch.empty(g["kc"].shape, dtype=torch.bfloat16, device="cuda")
    vcb = torch.empty_like(kcb)
    cartattn.cart_write_to_cache(g["kc"], g["vc"], kcb, vcb)
    ws_f = torch.empty(wf, dtype=torch.uint8, device="cuda")
    o_ref, lse_ref = cartattn.cart_attn_fwd(g["q"], g["k"], g["v"], kcb, vcb, theta=s.theta,
                                            workspace=ws_f)
    grads_ref = cartattn.cart_attn_bwd(g["q"], g["k"], g["v"], kcb, vcb, o_ref, lse_ref, g["do"],
                                       theta=s.theta, fwd_workspace=ws_f,
                                       workspace=torch.empty(wb, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    del ws_f
    nkc = g["kc"].numel()
    assert 2 * nkc * 4 <= wf
    nbv = max(wb, g["v"].numel() * 2)  # (a workspace may be larger than needed)
    reused = [0, 0]
    for _ in range(4):
        # (1) the leaves' f32 copies at the start of a block the size of the
        # forward's workspace, freed once the cache write is enqueued
        blk = torch.empty(wf, dtype=torch.uint8, device="cuda")
        leaves = blk[: 2 * nkc * 4].view(torch.float32)
        leaves[:nkc].copy_(g["kc"].reshape(-1))
        leaves[nkc:].copy_(g["vc"].reshape(-1))
        kcb2, vcb2 = torch.empty_like(kcb), torch.empty_like(vcb)
        cartattn.cart_write_to_cache(leaves[:nkc].view(g["kc"].shape),
                                     leaves[nkc:].view(g["vc"].shape), kcb2, vcb2)
        addr = blk.data_ptr()
        del leaves, blk
        ws_f = torch.empty(wf, dtype=torch.uint8, device="cuda")
        reused[0] += ws_f.data_ptr() == addr
        # (2) V copied into a block, freed once the forward is enqueued; the
        # backward's workspace is a block of the same size
        blk = torch.empty(nbv, dtype=torch.uint8, device="cuda")
        v_tmp = blk[: g["v"].numel() * 2].view(torch.bfloat16).view(g["v"].shape)
        v_tmp.copy_(g["v"])
        o, lse = cartattn.cart_attn_fwd(g["q"], g["k"], v_tmp, kcb2, vcb2, theta=s.theta,
                                        workspace=ws_f)
        addr = blk.data_ptr()
        del v_tmp, blk
        ws_b = torch.empty(nbv, dtype=torch.uint8, device="cuda")
        reused[1] += ws_b.data_ptr() == addr
        grads = cartattn.cart_attn_bwd(g["q"], g["k"], g["v"], kcb2, vcb2, o, lse, g["do"],
                                       theta=s.theta, fwd_workspace=ws_f, workspace=ws_b)
        torch.cuda.synchronize()
        assert cartattn.device_status(clear=True) == 0
        assert torch.equal(kcb2.view(torch.uint8), kcb.view(torch.uint8))
        assert torch.equal(o.view(torch.uint8), o_ref.view(torch.uint8))
        assert torch.equal(lse, lse_ref)
        for nme, x, y in zip(("dq", "dk", "dv", "dkc", "dvc"), grads, grads_ref):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), nme
        del ws_f, ws_b
    # the allocator did hand the freed blocks out again (else nothing was tested)
    assert reused[0] > 0 and reused[1] > 0, reused


def test_cache_write_bitwise():
    rng = np.random.default_rng(7)
    p, Hkv, d = 300, 4, 128
    kc = torch.from_numpy((rng.standard_normal((p, Hkv, d)) * 3).astype(np.float32))
    vc = torch.from_numpy((rng.standard_normal((p, Hkv, d)) * 1e-3).astype(np.float32))
    rows = 320
    kd = torch.zeros((rows, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros((rows, Hkv, d), dtype=torch.bfloat16, device="cuda")
    cartattn.cart_write_to_cache(kc.cuda(), vc.cuda(), kd, vd, dst_row0=7)
    torch.cuda.synchronize()
    for src, dst in ((kc, kd), (vc, vd)):
        want = np.zeros((rows, Hkv, d), dtype=np.uint16)
        oracle.write_to_cache(src.numpy(), want, dst_row0=7)
        got = dst.cpu().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, want)


def test_cache_write_f32_destination():
    rng = np.random.default_rng(8)
    kc = torch.from_numpy(rng.standard_normal((33, 2, 64)).astype(np.float32))
    kd = torch.zeros((40, 2, 64), dtype=torch.float32, device="cuda")
    vd = torch.zeros((40, 2, 64), dtype=torch.float32, device="cuda")
    cartattn.cart_write_to_cache(kc.cuda(), kc.cuda(), kd, vd, dst_row0=5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kd.cpu().numpy()[5:38], kc.numpy())
    assert (kd.cpu().numpy()[:5] == 0).all() and (kd.cpu().numpy()[38:] == 0).all()


# ------------------------------------------------------------- decode ----
def _decode_case(name, B, Hq, Hkv, d, p, max_private, lens=(), seed=200):
    return synth.DecodeShape(name, B=B, Hq=Hq, Hkv=Hkv, d=d, p=p, max_private=max_private,
                             seed=seed, fixed_len=tuple(lens))


DECODE_SMALL = [
    _decode_case("ragged", 3, 4, 2, 64, 16, 39, lens=(0, 17, 39)),
    _decode_case("p0", 2, 8, 2, 128, 0, 200, lens=(0, 130)),
    _decode_case("g8_p300", 4, 8, 1, 128, 300, 300, lens=(0, 1, 127, 300)),
    _decode_case("g1_big", 5, 4, 4, 128, 1000, 600, lens=(600, 0, 128, 129, 255)),
]


def _run_decode(s, inp):
    g = {k: v.cuda() for k, v in inp.items()}
    o = cartattn.cart_attn_decode(g["q"], g["k_new"], g["v_new"], g["kc"], g["vc"], g["k_cache"],
                                  g["v_cache"], g["lens"], theta=s.theta)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    return synth.f64(o), g["k_cache"].cpu(), g["v_cache"].cpu()


def _check_decode(s, inp, o, kcache, vcache):
    a = {k: synth.f64(v) for k, v in inp.items() if k != "lens"}
    lens = inp["lens"].numpy()
    o_ref, kref, vref = oracle.decode(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"],
                                      a["k_cache"], a["v_cache"], lens, theta=s.theta)
    assert gh.max_abs(o, o_ref) <= gh.FWD_MAXABS, gh.max_abs(o, o_ref)
    assert gh.rel_l2(o, o_ref) <= gh.FWD_RELL2, gh.rel_l2(o, o_ref)
    kc_new = synth.f64(kcache)
    vc_new = synth.f64(vcache)
    for b in range(s.B):
        L = int(lens[b])
        # rows other than the appended one are untouched
        mask = np.ones(s.cache_rows, bool)
        mask[L] = False
        np.testing.assert_array_equal(kc_new[b][mask], a["k_cache"][b][mask])
        np.testing.assert_array_equal(vc_new[b][mask], a["v_cache"][b][mask])
        np.testing.assert_array_equal(vc_new[b, L], a["v_new"][b])
        # the appended key is the rotated new key, rounded once to bf16
        np.testing.assert_allclose(kc_new[b, L], kref[b, L], rtol=2 ** -8, atol=1e-6)


@pytest.mark.parametrize("s", DECODE_SMALL, ids=[s.name for s in DECODE_SMALL])
def test_decode_parity_small(s):
    inp = synth.decode_inputs(s)
    o, kc, vc = _run_decode(s, inp)
    _check_decode(s, inp, o, kc, vc)


# Edge cases of the single-token step: kv-head counts 1 to 8, d = 64, p = 0
# (no cartridge pass), lengths at and around the 256-row unit and 128-row
# tile edges, one conversation over many units, and NaN in every cache row
# past a conversation's length (rows a unit or tile reads beyond the length
# must never reach a product).
EDGE_DECODE = [
    (_decode_case("e_hkv8_nan", 5, 32, 8, 128, 200, 800, lens=(0, 15, 16, 17, 700)), True),
    (_decode_case("e_hkv1_g8_d64", 4, 8, 1, 64, 100, 400, lens=(127, 128, 0, 300)), True),
    (_decode_case("e_hkv4_g2", 7, 8, 4, 128, 129, 300, lens=(1, 2, 3, 299, 7, 8, 9)), False),
    (_decode_case("e_hkv2_p0_tiny", 3, 8, 2, 128, 0, 600, lens=(0, 0, 0)), True),
    (_decode_case("e_long", 2, 32, 8, 128, 4096, 8000, lens=(8000, 3)), False),
]


def _nan_tails(inp):
    """Private cache rows past each conversation's new row set to NaN."""
    out = dict(inp)
    for name in ("k_cache", "v_cache"):
        t = inp[name].clone()
        for b, L in enumerate(inp["lens"].tolist()):
            t[b, L + 1:] = float("nan")
        out[name] = t
    return out


@pytest.mark.parametrize("case", EDGE_DECODE, ids=[c[0].name for c in EDGE_DECODE])
def test_decode_edge_parity(case):
    s, nan_tail = case
    inp = synth.decode_inputs(s)
    if nan_tail:
        inp = _nan_tails(inp)
    o, kc, vc = _run_decode(s, inp)
    assert not np.isnan(o).any()
    _check_decode(s, inp, o, kc, vc)


def test_decode_many_small_conversations():
    """12000 conversations of 1-5 rows each behind a 64-row cartridge."""
    s = _decode_case("e_many", 12000, 8, 2, 64, 64, 4, seed=201)
    inp = synth.decode_inputs(s)
    o, kc, vc = _run_decode(s, inp)
    _check_decode(s, inp, o, kc, vc)


SPAN_CASES = [
    # (case, span): G*span query columns from 4 to 32 (one to four groups of
    # 8); lengths at 0, at the last slot that fits the span, and spans that
    # cross 64-row chunks and 256-row units
    (_decode_case("span2", 3, 4, 2, 64, 16, 39, lens=(0, 17, 37)), 2),
    (_decode_case("span3_units", 4, 8, 2, 128, 300, 300, lens=(0, 62, 254, 297)), 3),
    (_decode_case("span8_g4", 3, 8, 2, 128, 200, 520, lens=(250, 0, 513)), 8),
    (_decode_case("span4_g8_p0", 2, 8, 1, 128, 0, 300, lens=(0, 129)), 4),
    (_decode_case("span5_g1_d64", 5, 4, 4, 64, 130, 260, lens=(0, 60, 128, 251, 256)), 5),
    (_decode_case("span6_g4", 2, 8, 2, 128, 64, 200, lens=(190, 3)), 6),
]


@pytest.mark.parametrize("case", SPAN_CASES, ids=[c[0].name for c in SPAN_CASES])
def test_decode_span_parity(case):
    s, span = case
    inp = synth.decode_span_inputs(s, span)
    g = {k: v.cuda() for k, v in inp.items()}
    o = cartattn.cart_attn_decode_span(g["q"], g["k_new"], g["v_new"], g["kc"], g["vc"],
                                       g["k_cache"], g["v_cache"], g["lens"], theta=s.theta)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    a = {k: synth.f64(v) for k, v in inp.items() if k != "lens"}
    lens = inp["lens"].numpy()
    o_ref, kref, vref = oracle.decode_span(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"],
                                           a["k_cache"], a["v_cache"], lens, theta=s.theta)
    o = synth.f64(o)
    assert gh.max_abs(o, o_ref) <= gh.FWD_MAXABS, gh.max_abs(o, o_ref)
    assert gh.rel_l2(o, o_ref) <= gh.FWD_RELL2, gh.rel_l2(o, o_ref)
    kc_new, vc_new = synth.f64(g["k_cache"]), synth.f64(g["v_cache"])
    for b in range(s.B):
        L = int(lens[b])
        mask = np.ones(s.cache_rows, bool)
        mask[L:L + span] = False
        np.testing.assert_array_equal(kc_new[b][mask], a["k_cache"][b][mask])
        np.testing.assert_array_equal(vc_new[b][mask], a["v_cache"][b][mask])
        np.testing.assert_array_equal(vc_new[b, L:L + span], a["v_new"][b])
        np.testing.assert_allclose(kc_new[b, L:L + span], kref[b, L:L + span], rtol=2 ** -8,
                                   atol=1e-6)


def test_decode_span_one_equals_decode():
    """span = 1 is the single-token step, bit for bit."""
    s = DECODE_SMALL[3]
    inp = synth.decode_inputs(s)
    o1, _, _ = _run_decode(s, inp)
    g = {k: v.cuda() for k, v in inp.items()}
    o2 = cartattn.cart_attn_decode_span(g["q"][:, None], g["k_new"][:, None], g["v_new"][:, None],
                                        g["kc"], g["vc"], g["k_cache"], g["v_cache"], g["lens"],
                                        theta=s.theta)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o1, synth.f64(o2[:, 0]))


def test_decode_serving_workload():
    """64 conversations behind one p = 4096 cartridge, 0..1024 private rows."""
    s = synth.DECODE
    inp = synth.decode_inputs(s)
    o, kc, vc = _run_decode(s, inp)
    _check_decode(s, inp, o, kc, vc)


# ------------------------------------------------ full-size workloads ----
def test_equivalence_gate_bf16():
    """Cartridge = rotated bf16 K/V of 512 prefix tokens; the 256 continuation
    queries behind it match (a) the oracle on the same stored inputs and
    (b) causal attention over all 768 tokens (the zero-step gate)."""
    s = synth.EQUIV
    p, n = s.p, s.n
    kraw, vraw, rng = synth.token_kv(p + n, s.Hkv, s.d, seed=s.seed, std=s.qkv_std)
    qcont = synth.token_q(rng, n, s.Hq, s.d, std=s.qkv_std)
    inp = dict(q=synth.to_storage(qcont[None], "bf16"), k=synth.to_storage(kraw[None, p:], "bf16"),
               v=synth.to_storage(vraw[None, p:], "bf16"),
               kc=synth.to_storage(oracle.rope(kraw[:p], 0, theta=s.theta), "bf16"),
               vc=synth.to_storage(vraw[:p], "bf16"),
               do=synth.to_storage(np.zeros((1, n, s.Hq, s.d)), "bf16"))
    got = gh.run_train_gpu(s, inp, bwd=False)
    ref = gh.oracle_train(s, inp, bwd=False)
    gh.check_fwd(got, ref)
    # the prefill reference: every token real, positions 0..767, stored values
    kfull = synth.f64(synth.to_storage(kraw, "bf16"))[None]
    vfull = synth.f64(synth.to_storage(vraw, "bf16"))[None]
    qfull = np.zeros((1, p + n, s.Hq, s.d))
    qfull[0, p:] = synth.f64(inp["q"])[0]
    empty = np.zeros((0, s.Hkv, s.d))
    o_full, _ = oracle.fwd(qfull, kfull, vfull, empty, empty, theta=s.theta, rows=(p, p + n))
    assert gh.max_abs(got["o"][0], o_full[0, p:]) <= gh.FWD_MAXABS
    assert gh.rel_l2(got["o"][0], o_full[0, p:]) <= gh.FWD_RELL2


def test_selfstudy_workload_one_group():
    """B=4, Hq=32, Hkv=8, d=128, p=2048, n=1024: every output of kv-head
    group 0 (query heads 0-3) against the oracle, cartridge gradient included."""
    s = synth.SELFSTUDY
    inp = synth.train_inputs(s)
    got = gh.run_train_gpu(s, inp)
    G = s.Hq // s.Hkv
    ref = gh.oracle_train(s, inp, heads=(0, G), kv_heads=(0, 1))
    gh.check_fwd(got, ref, sl=(slice(None), slice(None), slice(0, G)),
                 lse_sl=(slice(None), slice(0, G)))
    gh.check_grads(got, ref, s.frozen_prefix,
                   sls=dict(dq=(slice(None), slice(None), slice(0, G)),
                            dk=(slice(None), slice(None), slice(0, 1)),
                            dv=(slice(None), slice(None), slice(0, 1)),
                            dkc=(slice(None), slice(0, 1)), dvc=(slice(None), slice(0, 1))))


def test_selfstudy_window_one_group():
    """The self-study workload under a 1024-key window (early queries see
    half of the cartridge, late ones none of it): kv-head group 0 against the
    oracle, cartridge gradient included."""
    s = synth.SELFSTUDY
    window = 1024
    inp = synth.train_inputs(s)
    got = gh.run_train_gpu(s, inp, window=window)
    G = s.Hq // s.Hkv
    ref = gh.oracle_train(s, inp, heads=(0, G), kv_heads=(0, 1), window=window)
    gh.check_fwd(got, ref, sl=(slice(None), slice(None), slice(0, G)),
                 lse_sl=(slice(None), slice(0, G)))
    gh.check_grads(got, ref, s.frozen_prefix,
                   sls=dict(dq=(slice(None), slice(None), slice(0, G)),
                            dk=(slice(None), slice(None), slice(0, 1)),
                            dv=(slice(None), slice(None), slice(0, 1)),
                            dkc=(slice(None), slice(0, 1)), dvc=(slice(None), slice(0, 1))))
    # rows before the first query's window: exactly zero
    assert (got["dkc"][:s.p - window + 1] == 0).all()


def test_packed_selfstudy_one_group():
    """Eight packed conversations of up to 1024 tokens with the self-study
    heads and cartridge: kv-head group 0 against the oracle."""
    s = synth.SELFSTUDY
    lens = synth.packed_lengths(s.n, 8, seed=7)
    inp = synth.packed_inputs(s, lens)
    g = gh.to_gpu({k: v for k, v in inp.items() if k != "max_seqlen"})
    n = inp["max_seqlen"]
    o, lse = cartattn.cart_attn_fwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], g["cu"], n)
    grads = cartattn.cart_attn_bwd_packed(g["q"], g["k"], g["v"], g["kc"], g["vc"], o, lse,
                                          g["do"], g["cu"], n)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    got = {k: synth.f64(v) for k, v in zip(("o", "lse", "dq", "dk", "dv", "dkc", "dvc"),
                                           (o, lse, *grads))}
    a = {k: synth.f64(v) for k, v in inp.items() if k not in ("cu", "max_seqlen")}
    cu = inp["cu"].numpy()
    G = s.Hq // s.Hkv
    ref = dict(zip(("o", "lse"), oracle.fwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], cu,
                                                   heads=(0, G))))
    ref.update(zip(("dq", "dk", "dv", "dkc", "dvc"),
                   oracle.bwd_packed(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["do"], cu,
                                     kv_heads=(0, 1))))
    gh.check_fwd(got, ref, sl=(slice(None), slice(0, G)), lse_sl=(slice(0, G),))
    gh.check_grads(got, ref, s.frozen_prefix,
                   sls=dict(dq=(slice(None), slice(0, G)), dk=(slice(None), slice(0, 1)),
                            dv=(slice(None), slice(0, 1)), dkc=(slice(None), slice(0, 1)),
                            dvc=(slice(None), slice(0, 1))))


def test_decode_serving_workload_windowed():
    """The serving workload with a 512-key window: most conversations see
    only the last cartridge tiles (the cartridge pass skips the rest)."""
    s = synth.DECODE
    inp = synth.decode_inputs(s)
    g = {k: v.cuda() for k, v in inp.items()}
    o = cartattn.cart_attn_decode_span(g["q"][:, None], g["k_new"][:, None], g["v_new"][:, None],
                                       g["kc"], g["vc"], g["k_cache"], g["v_cache"], g["lens"],
                                       theta=s.theta, window=512)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    a = {k: synth.f64(v) for k, v in inp.items() if k != "lens"}
    o_ref, _, _ = oracle.decode(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["k_cache"],
                                a["v_cache"], inp["lens"].numpy(), theta=s.theta, window=512)
    o = synth.f64(o[:, 0])
    assert gh.max_abs(o, o_ref) <= gh.FWD_MAXABS, gh.max_abs(o, o_ref)
    assert gh.rel_l2(o, o_ref) <= gh.FWD_RELL2, gh.rel_l2(o, o_ref)


def test_longctx_workload_one_group():
    """B=1, Hq=64, Hkv=8, d=128, p=8192, n=4096: every output of kv-head
    group 3 (query heads 24-31, all 4096 query rows) against the oracle, the
    p = 8192 cartridge gradient of that group included; then properties that
    hold for every group."""
    s = synth.LONGCTX
    inp = synth.train_inputs(s)
    got = gh.run_train_gpu(s, inp)
    G = s.Hq // s.Hkv
    g0 = 3
    ref = gh.oracle_group_parallel(s, inp, g0)
    hs = slice(g0 * G, g0 * G + G)
    grp = {"o": got["o"][:, :, hs], "lse": got["lse"][:, hs], "dq": got["dq"][:, :, hs],
           "dk": got["dk"][:, :, g0:g0 + 1], "dv": got["dv"][:, :, g0:g0 + 1],
           "dkc": got["dkc"][:, g0:g0 + 1], "dvc": got["dvc"][:, g0:g0 + 1]}
    gh.check_fwd(grp, ref)
    gh.check_grads(grp, ref, s.frozen_prefix)
    # frozen sink row exactly zero; the other rows do not depend on the freeze
    assert (got["dkc"][0] == 0).all() and (got["dvc"][0] == 0).all()
    unfrozen = gh.run_train_gpu(s, inp, frozen_prefix=0)
    np.testing.assert_array_equal(unfrozen["dkc"][1:], got["dkc"][1:])
    np.testing.assert_array_equal(unfrozen["dvc"][1:], got["dvc"][1:])
    assert np.abs(unfrozen["dvc"][0]).max() > 0
    # value gradients over every attended row sum to the summed upstream
    # gradient of the group (softmax weights sum to one)
    do = synth.f64(inp["do"])
    for g in range(s.Hkv):
        lhs = unfrozen["dvc"][:, g].sum(0) + got["dv"][:, :, g].sum((0, 1))
        rhs = do[:, :, g * G:(g + 1) * G].sum((0, 1, 2))
        assert gh.rel_l2(lhs, rhs) <= gh.GRAD_RELL2
    # key gradients (rotated into the attended space) sum to zero
    for g in (0, 5):
        dk_att = oracle.rope(got["dk"][0, :, g:g + 1], s.p, theta=s.theta)[:, 0]
        lhs = unfrozen["dkc"][:, g].sum(0) + dk_att.sum(0)
        scale = np.abs(unfrozen["dkc"][:, g]).sum(0).max() + np.abs(dk_att).sum(0).max()
        assert np.abs(lhs).max() <= 1e-2 * scale


WINDOW_DECODE = [
    # (case, span, window): windows inside the private rows, cutting the
    # cartridge, reaching past several 256-row units, one key only
    (_decode_case("wdec_priv", 3, 8, 2, 128, 300, 600, lens=(0, 255, 599)), 1, 100),
    (_decode_case("wdec_cart", 4, 4, 2, 128, 400, 300, lens=(0, 17, 200, 300)), 1, 350),
    (_decode_case("wdec_units", 2, 8, 1, 128, 130, 900, lens=(899, 520)), 1, 700),
    (_decode_case("wdec_one", 2, 4, 4, 64, 64, 70, lens=(69, 3)), 1, 1),
    (_decode_case("wdec_span", 3, 8, 2, 128, 300, 600, lens=(0, 250, 595)), 4, 260),
]


@pytest.mark.parametrize("case", WINDOW_DECODE, ids=[c[0].name for c in WINDOW_DECODE])
def test_window_decode_parity(case):
    s, span, window = case
    inp = synth.decode_span_inputs(s, span)
    g = {k: v.cuda() for k, v in inp.items()}
    o = cartattn.cart_attn_decode_span(g["q"], g["k_new"], g["v_new"], g["kc"], g["vc"],
                                       g["k_cache"], g["v_cache"], g["lens"], theta=s.theta,
                                       window=window)
    torch.cuda.synchronize()
    assert cartattn.device_status(clear=True) == 0
    a = {k: synth.f64(v) for k, v in inp.items() if k != "lens"}
    o_ref, _, _ = oracle.decode_span(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"],
                                     a["k_cache"], a["v_cache"], inp["lens"].numpy(),
                                     theta=s.theta, window=window)
    o = synth.f64(o)
    assert gh.max_abs(o, o_ref) <= gh.FWD_MAXABS, gh.max_abs(o, o_ref)
    assert gh.rel_l2(o, o_ref) <= gh.FWD_RELL2, gh.rel_l2(o, o_ref)
