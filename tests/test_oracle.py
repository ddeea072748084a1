"""Pins for the fp64 oracle (CPU only).

Every check compares the oracle with something other than itself:
library routines (SDPA with an explicit mask, complex-number RoPE, autograd,
torch's float->bfloat16 cast), finite differences, the p = 0 reduction to
ordinary causal attention, the prefill-equivalence gate of the Cartridges
guide ("Evidence": an untrained corpus-init cartridge reproduces the real
prefill) and invariants of softmax attention.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import torch_formulation as tf
from trained_kv_prefix_gb300 import synth

THETA = 1.0e6


def _rand(rng, *shape, std=0.5):
    return rng.standard_normal(size=shape) * std


def _problem(seed, B, n, Hq, Hkv, d, p, std=0.5):
    rng = np.random.default_rng(seed)
    return dict(q=_rand(rng, B, n, Hq, d, std=std), k=_rand(rng, B, n, Hkv, d, std=std),
                v=_rand(rng, B, n, Hkv, d, std=std), kc=_rand(rng, p, Hkv, d, std=std),
                vc=_rand(rng, p, Hkv, d, std=std), do=_rand(rng, B, n, Hq, d, std=1.0))


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x))


SHAPES = [
    # B, n, Hq, Hkv, d, p
    (1, 32, 4, 2, 64, 16),     # the tiny workload's geometry
    (2, 7, 6, 3, 8, 5),        # ragged, odd p, G = 2
    (1, 9, 4, 4, 16, 1),       # MHA, sink only
    (3, 5, 8, 2, 4, 3),        # G = 4, several batches
]


# ---------------------------------------------------------------- RoPE ----
@pytest.mark.parametrize("d", [4, 8, 64, 128])
def test_rope_matches_complex_rotation(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((11, 3, d))
    got = oracle.rope(x, 37, theta=THETA)
    want = tf.rope_complex(_t(x).permute(1, 0, 2), torch.arange(37, 48), THETA)
    np.testing.assert_allclose(got, want.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    back = oracle.rope(got, 37, theta=THETA, inverse=True)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)


def test_rope_identity_at_zero_and_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 2, 64))
    np.testing.assert_array_equal(oracle.rope(x, 0), x)
    y = oracle.rope(rng.standard_normal((50, 2, 64)), 1000)
    x2 = oracle.rope(y, 1000, inverse=True)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x2, axis=-1),
                               rtol=1e-13)


def test_rope_relative_position():
    """<R(m) q, R(m') k> depends only on m - m'."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    dots = []
    for shift in (0, 5, 4096):
        qm = oracle.rope(q, 100 + shift)
        km = oracle.rope(k, 37 + shift)
        dots.append(float((qm * km).sum()))
    assert abs(dots[0] - dots[1]) < 1e-10 and abs(dots[0] - dots[2]) < 1e-10
    qm = oracle.rope(q, 101)
    km = oracle.rope(k, 37)
    assert abs(float((qm * km).sum()) - dots[0]) > 1e-6  # a shift of one changes it


# ------------------------------------------------------------- forward ----
@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_masked_sdpa(shape):
    B, n, Hq, Hkv, d, p = shape
    P = _problem(10 + d + p, *shape)
    o, lse = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], theta=THETA)
    o_ref, lse_ref = tf.cartridge_attention(*(_t(P[x]) for x in ("q", "k", "v", "kc", "vc")),
                                            theta=THETA)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=0, atol=1e-12)


def test_fwd_row_and_head_restriction():
    P = _problem(3, 2, 12, 4, 2, 16, 5)
    full, lse = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    part, lpart = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], heads=(1, 3), rows=(4, 9))
    np.testing.assert_array_equal(part[:, 4:9, 1:3], full[:, 4:9, 1:3])
    np.testing.assert_array_equal(lpart[:, 1:3, 4:9], lse[:, 1:3, 4:9])
    assert np.isnan(part[:, :4]).all() and np.isnan(part[:, :, 0]).all()


def test_p0_is_textbook_causal_attention():
    """With no cartridge rows the mask is the ordinary causal one and real
    tokens sit at positions 0..n-1."""
    rng = np.random.default_rng(4)
    B, n, H, d = 2, 13, 3, 16
    q, k, v = (rng.standard_normal((B, n, H, d)) for _ in range(3))
    empty = np.zeros((0, H, d))
    o, _ = oracle.fwd(q, k, v, empty, empty, theta=THETA)
    pos = torch.arange(n)
    qh = tf.rope_complex(_t(q).permute(0, 2, 1, 3), pos, THETA)
    kh = tf.rope_complex(_t(k).permute(0, 2, 1, 3), pos, THETA)
    ref = torch.nn.functional.scaled_dot_product_attention(qh, kh, _t(v).permute(0, 2, 1, 3),
                                                           is_causal=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_equivalence_gate_prefill():
    """Cartridge = the rotated K/V of the first p tokens; queries for the next
    n tokens behind it equal the last n rows of causal attention over all
    p + n tokens (the zero-step acceptance gate)."""
    p, n, Hq, Hkv, d = 24, 10, 4, 2, 32
    kraw, vraw, rng = synth.token_kv(p + n, Hkv, d, seed=5)
    qall = synth.token_q(rng, p + n, Hq, d)
    kc = oracle.rope(kraw[:p], 0, theta=THETA)
    vc = vraw[:p]
    o_cart, lse_cart = oracle.fwd(qall[None, p:], kraw[None, p:], vraw[None, p:], kc, vc,
                                  theta=THETA)
    empty = np.zeros((0, Hkv, d))
    o_full, lse_full = oracle.fwd(qall[None], kraw[None], vraw[None], empty, empty, theta=THETA)
    np.testing.assert_allclose(o_cart, o_full[:, p:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_cart, lse_full[:, :, p:], rtol=0, atol=1e-12)
    # a cartridge whose real tokens are rotated from position 0 instead of p
    # is "plausible but wrong": it must not pass the gate
    o_bad, _ = oracle.fwd(qall[None, p:], kraw[None, p:], vraw[None, p:],
                          np.zeros((0, Hkv, d)), np.zeros((0, Hkv, d)), theta=THETA)
    assert np.abs(o_bad - o_full[:, p:]).max() > 1e-3


def test_gqa_equals_repeated_heads():
    P = _problem(6, 2, 9, 8, 2, 16, 4)
    o, _ = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    rep = lambda a, ax: np.repeat(a, 4, axis=ax)  # noqa: E731
    o_mha, _ = oracle.fwd(P["q"], rep(P["k"], 2), rep(P["v"], 2), rep(P["kc"], 1),
                          rep(P["vc"], 1))
    np.testing.assert_allclose(o, o_mha, rtol=0, atol=1e-14)


def test_softmax_weights_sum_to_one():
    P = _problem(7, 1, 11, 4, 2, 8, 6)
    ones = np.ones_like(P["v"])
    o, _ = oracle.fwd(P["q"], P["k"], ones, P["kc"], np.ones_like(P["vc"]))
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_cartridge_rows_carry_no_position():
    """Permuting cartridge rows 1..p-1 (K and V together) leaves the output
    unchanged and permutes the cartridge gradients."""
    P = _problem(8, 2, 6, 4, 2, 8, 7)
    perm = np.concatenate([[0], 1 + np.random.default_rng(0).permutation(6)])
    o1, _ = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    o2, _ = oracle.fwd(P["q"], P["k"], P["v"], P["kc"][perm], P["vc"][perm])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    g1 = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    g2 = oracle.bwd(P["q"], P["k"], P["v"], P["kc"][perm], P["vc"][perm], P["do"])
    np.testing.assert_allclose(g1[3][perm], g2[3], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g1[4][perm], g2[4], rtol=0, atol=1e-13)


# ------------------------------------------------------------ backward ----
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("frozen", [0, 1, 2])
def test_bwd_matches_autograd(shape, frozen):
    B, n, Hq, Hkv, d, p = shape
    if frozen > p:
        pytest.skip("frozen rows exceed p")
    P = _problem(20 + d + p, *shape)
    got = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], frozen_prefix=frozen,
                     theta=THETA)
    want = tf.cartridge_grads(*(_t(P[x]) for x in ("q", "k", "v", "kc", "vc", "do")),
                              frozen_prefix=frozen, theta=THETA)
    for name, a, b in zip(("dq", "dk", "dv", "dkc", "dvc"), got, want):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-12, err_msg=name)
    assert (got[3][:frozen] == 0).all() and (got[4][:frozen] == 0).all()


def test_bwd_composed_parts_freeze_each_sink():
    """A composed cartridge (two parts concatenated along the rows, each with
    its own sink row) freezes both sinks: their gradients are exactly 0 and
    every other row's gradient is that of the all-trainable problem
    (autograd formulation), since freezing a leaf does not change the others'
    gradients."""
    shape = (2, 24, 4, 2, 64, 20)
    P = _problem(77, *shape)
    part_b = 9  # second part occupies rows 9..19; row 9 is its sink
    got = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], frozen_prefix=1,
                     theta=THETA, frozen_rows=(part_b,))
    want = tf.cartridge_grads(*(_t(P[x]) for x in ("q", "k", "v", "kc", "vc", "do")),
                              frozen_prefix=0, theta=THETA)
    for name, a, b in zip(("dq", "dk", "dv", "dkc", "dvc"), got, want):
        b = b.numpy().copy()
        if name in ("dkc", "dvc"):
            assert np.abs(b[part_b]).max() > 0  # the sink would otherwise get a gradient
            b[0] = 0.0
            b[part_b] = 0.0
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12, err_msg=name)
    assert (got[3][[0, part_b]] == 0).all() and (got[4][[0, part_b]] == 0).all()
    with pytest.raises(ValueError):
        oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], theta=THETA,
                   frozen_rows=(20,))


def test_bwd_finite_differences():
    """Central differences of the oracle's own forward (tiny geometry)."""
    B, n, Hq, Hkv, d, p = 1, 6, 4, 2, 8, 5
    P = _problem(30, B, n, Hq, Hkv, d, p)
    grads = dict(zip(("q", "k", "v", "kc", "vc"),
                     oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])))
    eps = 1e-6
    rng = np.random.default_rng(31)

    def loss(X):
        o, _ = oracle.fwd(X["q"], X["k"], X["v"], X["kc"], X["vc"])
        return float((o * P["do"]).sum())

    for name in ("q", "k", "v", "kc", "vc"):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in P[name].shape)
            if name in ("kc", "vc") and idx[0] == 0:
                idx = (1,) + idx[1:]
            Xp = {k2: a.copy() for k2, a in P.items()}
            Xm = {k2: a.copy() for k2, a in P.items()}
            Xp[name][idx] += eps
            Xm[name][idx] -= eps
            fd = (loss(Xp) - loss(Xm)) / (2 * eps)
            an = grads[name][idx]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, idx, fd, an)
    # the sink row is frozen: its gradient is exactly zero although the loss
    # does depend on it
    assert (grads["kc"][0] == 0).all() and (grads["vc"][0] == 0).all()


def test_bwd_batch_sum_is_sequential_sum():
    """Cartridge gradient of a batch equals the sum over one-sequence runs
    (packed vs sequential)."""
    P = _problem(40, 3, 5, 4, 2, 8, 6)
    full = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    acc_k = np.zeros_like(full[3])
    acc_v = np.zeros_like(full[4])
    for b in range(3):
        sl = slice(b, b + 1)
        g = oracle.bwd(P["q"][sl], P["k"][sl], P["v"][sl], P["kc"], P["vc"], P["do"][sl])
        acc_k += g[3]
        acc_v += g[4]
        np.testing.assert_allclose(g[0], full[0][sl], rtol=0, atol=1e-13)
    np.testing.assert_allclose(acc_k, full[3], rtol=0, atol=1e-12)
    np.testing.assert_allclose(acc_v, full[4], rtol=0, atol=1e-12)


def test_bwd_key_gradient_sums_vanish():
    """Softmax rows are shift invariant, so the gradients w.r.t. all attended
    keys (rotated back to the attended space) sum to zero, and the value
    gradients sum to the summed upstream gradient (weights sum to one)."""
    B, n, Hq, Hkv, d, p = 2, 7, 4, 2, 16, 5
    P = _problem(41, B, n, Hq, Hkv, d, p)
    dq, dk, dv, dkc, dvc = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"],
                                      frozen_prefix=0)
    G = Hq // Hkv
    for kh in range(Hkv):
        s_k = dkc[:, kh].sum(0)
        s_v = dvc[:, kh].sum(0)
        for b in range(B):
            s_k = s_k + oracle.rope(dk[b, :, kh:kh + 1], p)[:, 0].sum(0)
            s_v = s_v + dv[b, :, kh].sum(0)
        np.testing.assert_allclose(s_k, 0.0, atol=1e-12)
        np.testing.assert_allclose(s_v, P["do"][:, :, kh * G:(kh + 1) * G].sum((0, 1, 2)),
                                   atol=1e-12)


def test_bwd_kv_head_restriction():
    P = _problem(42, 2, 6, 4, 2, 8, 5)
    full = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    part = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], kv_heads=(1, 2))
    np.testing.assert_array_equal(part[0][:, :, 2:4], full[0][:, :, 2:4])
    np.testing.assert_array_equal(part[1][:, :, 1], full[1][:, :, 1])
    np.testing.assert_array_equal(part[3][:, 1], full[3][:, 1])


def test_bwd_row_partition_sums_to_full():
    """The loss is a sum over query rows, so per-row-range gradients add up
    to the full gradient (and dq of each row comes from its own range)."""
    P = _problem(43, 2, 9, 4, 2, 8, 5)
    full = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    parts = [oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], rows=r)
             for r in ((0, 4), (4, 9))]
    np.testing.assert_array_equal(parts[0][0][:, :4], full[0][:, :4])
    np.testing.assert_array_equal(parts[1][0][:, 4:], full[0][:, 4:])
    assert np.isnan(parts[0][0][:, 4:]).all()
    for t in (1, 2, 3, 4):
        np.testing.assert_allclose(parts[0][t] + parts[1][t], full[t], rtol=0, atol=1e-13)


def test_group_parallel_helper_equals_one_oracle_call():
    """The row-split, group-sliced oracle helper the long-context GPU test
    uses gives the outputs of one full oracle call restricted to the group."""
    from tests import gpu_helpers as gh
    s = synth.TrainShape("grp", B=2, n=37, Hq=8, Hkv=2, d=16, p=11, frozen_prefix=1,
                         dtype="f32", cart_dtype="f32", seed=44, qkv_std=0.5, do_std=1.0)
    inp = synth.train_inputs(s)
    a = {k: synth.f64(v) for k, v in inp.items()}
    o, lse = oracle.fwd(a["q"], a["k"], a["v"], a["kc"], a["vc"], theta=s.theta)
    dq, dk, dv, dkc, dvc = oracle.bwd(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["do"],
                                      theta=s.theta)
    G = s.Hq // s.Hkv
    for g in range(s.Hkv):
        ref = gh.oracle_group_parallel(s, inp, g, chunk_rows=8, workers=3)
        hs = slice(g * G, (g + 1) * G)
        np.testing.assert_array_equal(ref["o"], o[:, :, hs])
        np.testing.assert_array_equal(ref["lse"], lse[:, hs])
        np.testing.assert_array_equal(ref["dq"], dq[:, :, hs])
        for name, full in (("dk", dk), ("dv", dv)):
            np.testing.assert_allclose(ref[name], full[:, :, g:g + 1], rtol=0, atol=1e-12)
        for name, full in (("dkc", dkc), ("dvc", dvc)):
            np.testing.assert_allclose(ref[name], full[:, g:g + 1], rtol=0, atol=1e-12)
        assert (ref["dkc"][0] == 0).all() and (ref["dvc"][0] == 0).all()


# -------------------------------------------------------------- decode ----
def test_decode_is_last_row_of_forward():
    """Decoding behind the cartridge equals the training-time forward of the
    same tokens (serving parity)."""
    B, Hq, Hkv, d, p = 3, 4, 2, 16, 9
    lens = np.array([0, 5, 2], dtype=np.int32)
    rows = 7
    rng = np.random.default_rng(50)
    kc = rng.standard_normal((p, Hkv, d)) * 0.5
    vc = rng.standard_normal((p, Hkv, d)) * 0.5
    kraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    vraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    q = rng.standard_normal((B, Hq, d)) * 0.5
    k_cache = np.full((B, rows, Hkv, d), 7.0)
    v_cache = np.full((B, rows, Hkv, d), 7.0)
    for b in range(B):
        L = lens[b]
        k_cache[b, :L] = oracle.rope(kraw[b, :L], p)
        v_cache[b, :L] = vraw[b, :L]
    k_new = np.stack([kraw[b, lens[b]] for b in range(B)])
    v_new = np.stack([vraw[b, lens[b]] for b in range(B)])
    o, kc2, vc2 = oracle.decode(q, k_new, v_new, kc, vc, k_cache, v_cache, lens)
    for b in range(B):
        L = int(lens[b])
        qs = np.zeros((1, L + 1, Hq, d))
        qs[0, L] = q[b]
        of, _ = oracle.fwd(qs, kraw[None, b, :L + 1], vraw[None, b, :L + 1], kc, vc,
                           rows=(L, L + 1))
        np.testing.assert_allclose(o[b], of[0, L], rtol=0, atol=1e-13)
        np.testing.assert_allclose(kc2[b, L], oracle.rope(kraw[b, L:L + 1], p + L)[0],
                                   atol=1e-14)
        np.testing.assert_array_equal(vc2[b, L], vraw[b, L])
        np.testing.assert_array_equal(kc2[b, L + 1:], 7.0)


def test_decode_span_is_rows_of_forward():
    """Span verify (several new tokens per conversation in one step) equals
    the training-time forward of the same tokens: query t is row len + t of
    a sequence whose first len rows are the already-cached tokens."""
    B, Hq, Hkv, d, p, span = 3, 4, 2, 16, 9, 3
    lens = np.array([0, 4, 2], dtype=np.int32)
    rows = 8
    rng = np.random.default_rng(51)
    kc = rng.standard_normal((p, Hkv, d)) * 0.5
    vc = rng.standard_normal((p, Hkv, d)) * 0.5
    kraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    vraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    q = rng.standard_normal((B, span, Hq, d)) * 0.5
    k_cache = np.full((B, rows, Hkv, d), 7.0)
    v_cache = np.full((B, rows, Hkv, d), 7.0)
    for b in range(B):
        L = lens[b]
        k_cache[b, :L] = oracle.rope(kraw[b, :L], p)
        v_cache[b, :L] = vraw[b, :L]
    k_new = np.stack([kraw[b, lens[b]:lens[b] + span] for b in range(B)])
    v_new = np.stack([vraw[b, lens[b]:lens[b] + span] for b in range(B)])
    o, kc2, vc2 = oracle.decode_span(q, k_new, v_new, kc, vc, k_cache, v_cache, lens)
    for b in range(B):
        L = int(lens[b])
        qs = np.zeros((1, L + span, Hq, d))
        qs[0, L:] = q[b]
        of, _ = oracle.fwd(qs, kraw[None, b, :L + span], vraw[None, b, :L + span], kc, vc,
                           rows=(L, L + span))
        np.testing.assert_allclose(o[b], of[0, L:L + span], rtol=0, atol=1e-13)
        np.testing.assert_allclose(kc2[b, L:L + span], oracle.rope(kraw[b, L:L + span], p + L),
                                   atol=1e-14)
        np.testing.assert_array_equal(vc2[b, L:L + span], vraw[b, L:L + span])
        np.testing.assert_array_equal(kc2[b, L + span:], 7.0)


def test_decode_matches_sdpa_single_query():
    B, Hq, Hkv, d, p = 2, 4, 1, 8, 6
    lens = np.array([0, 3], dtype=np.int32)
    rng = np.random.default_rng(51)
    kc, vc = (rng.standard_normal((p, Hkv, d)) for _ in range(2))
    kcache, vcache = (rng.standard_normal((B, 4, Hkv, d)) for _ in range(2))
    q = rng.standard_normal((B, Hq, d))
    kn, vn = (rng.standard_normal((B, Hkv, d)) for _ in range(2))
    o, kc2, vc2 = oracle.decode(q, kn, vn, kc, vc, kcache, vcache, lens, theta=THETA)
    for b in range(B):
        L = int(lens[b])
        qh = tf.rope_complex(_t(q[b][:, None, :]), torch.tensor([p + L]), THETA)  # [Hq,1,d]
        knew = tf.rope_complex(_t(kn[b][:, None, :]), torch.tensor([p + L]), THETA)
        K = torch.cat([_t(kc).permute(1, 0, 2), _t(kcache[b, :L]).permute(1, 0, 2), knew], 1)
        V = torch.cat([_t(vc).permute(1, 0, 2), _t(vcache[b, :L]).permute(1, 0, 2),
                       _t(vn[b][:, None, :])], 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh, K.expand(Hq, -1, -1), V.expand(Hq, -1, -1))
        np.testing.assert_allclose(o[b], ref[:, 0].numpy(), rtol=0, atol=1e-12)


def test_bad_geometry_is_rejected():
    P = _problem(60, 1, 4, 4, 3, 8, 2)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    P = _problem(61, 1, 4, 4, 2, 8, 2)
    with pytest.raises(ValueError):
        oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], frozen_prefix=3)


# ---------------------------------------------------------- cache write ----
def test_write_to_cache_matches_torch_bf16_cast():
    rng = np.random.default_rng(70)
    x = (rng.standard_normal((9, 2, 8)) * 10 ** rng.uniform(-40, 38, (9, 2, 8))).astype(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                         1.0 + 2 ** -8 + 2 ** -20, 3.0e38, 1e-45, -1e-40, 65504.0, 1.00390625,
                         np.float32(1.0) + np.float32(2 ** -9), 2 ** -126, 2.0 ** -133,
                         float(np.finfo(np.float32).max)], dtype=np.float32)
    x.reshape(-1)[:specials.size] = specials
    dst = np.zeros((12, 2, 8), dtype=np.uint16)
    oracle.write_to_cache(x, dst, dst_row0=2)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(dst[2:11], want)
    assert (dst[:2] == 0).all() and (dst[11:] == 0).all()
    # ties to even: 1 + 2^-8 lies half way between 1 and 1 + 2^-7 -> 1.0
    assert dst[2, 0, 4] == 0x3F80
    # 1 + 3*2^-8 lies half way between 1 + 2^-7 and 1 + 2^-6 -> the even one
    assert dst[2, 0, 5] == 0x3F82


def test_write_to_cache_nan_stays_nan():
    x = np.array([[[np.nan, -np.nan, 1.0, 2.0]]], dtype=np.float32)
    dst = np.zeros((1, 1, 4), dtype=np.uint16)
    oracle.write_to_cache(x, dst)
    back = torch.from_numpy(dst.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.isnan(back[0, 0, 0]) and np.isnan(back[0, 0, 1])
    assert back[0, 0, 2] == 1.0 and back[0, 0, 3] == 2.0


PACKED_CASES = [
    # (cu_seqlens, Hq, Hkv, d, p): ragged segments, an empty one, a lone token
    ((0, 5, 5, 12, 13, 20), 4, 2, 16, 6),
    ((0, 9, 17), 6, 3, 8, 1),
    ((0, 3, 11), 2, 2, 8, 0),
]


@pytest.mark.parametrize("case", PACKED_CASES)
def test_packed_matches_block_diagonal_attention(case):
    """Packed segments equal ONE attention over the packed tokens with a block
    diagonal mask and RoPE restarting at p per segment (forward, lse and every
    gradient, sink frozen)."""
    cu, Hq, Hkv, d, p = case
    T = cu[-1]
    P = _problem(60 + T, 1, T, Hq, Hkv, d, max(p, 1))
    q, k, v, do = P["q"][0], P["k"][0], P["v"][0], P["do"][0]
    kc, vc = P["kc"][:p], P["vc"][:p]
    fp = min(1, p)
    o, lse = oracle.fwd_packed(q, k, v, kc, vc, cu, frozen_prefix=fp)
    o_t, lse_t = tf.packed_attention(_t(q), _t(k), _t(v), _t(kc), _t(vc), cu)
    np.testing.assert_allclose(o, o_t.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), rtol=0, atol=1e-12)
    g = oracle.bwd_packed(q, k, v, kc, vc, do, cu, frozen_prefix=fp)
    g_t = tf.packed_grads(_t(q), _t(k), _t(v), _t(kc), _t(vc), _t(do), cu, frozen_prefix=fp)
    for a, b in zip(g, g_t):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-11)
    if p:
        assert (g[3][0] == 0).all() and (g[4][0] == 0).all()


def test_packed_equal_segments_are_a_batch():
    """Equal-length segments are the batched call with B = segments."""
    B, n, Hq, Hkv, d, p = 3, 6, 4, 2, 8, 5
    P = _problem(70, B, n, Hq, Hkv, d, p)
    cu = [i * n for i in range(B + 1)]
    flat = {k2: P[k2].reshape(B * n, *P[k2].shape[2:]) for k2 in ("q", "k", "v", "do")}
    o, lse = oracle.fwd_packed(flat["q"], flat["k"], flat["v"], P["kc"], P["vc"], cu)
    o_b, lse_b = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    np.testing.assert_array_equal(o, o_b.reshape(B * n, Hq, d))
    np.testing.assert_array_equal(lse, lse_b.transpose(1, 0, 2).reshape(Hq, B * n))
    g = oracle.bwd_packed(flat["q"], flat["k"], flat["v"], P["kc"], P["vc"], flat["do"], cu)
    g_b = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    for a, b in zip(g[:3], g_b[:3]):
        np.testing.assert_array_equal(a, b.reshape(a.shape))
    np.testing.assert_allclose(g[3], g_b[3], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g[4], g_b[4], rtol=0, atol=1e-13)


def test_packed_rejects_bad_segment_tables():
    P = _problem(71, 1, 6, 2, 1, 8, 3)
    for cu in ((0, 7), (1, 6), (0, 4, 2, 6), (0,)):
        with pytest.raises(ValueError):
            oracle.fwd_packed(P["q"][0], P["k"][0], P["v"][0], P["kc"], P["vc"], cu)


@pytest.mark.parametrize("window", [1, 3, 8, 13, 40])
def test_window_matches_masked_sdpa(window):
    """Sliding window (the W most recent keys, counting itself; cartridge row
    j at position j): forward, lse and every gradient against masked SDPA
    with autograd.  p = 9, n = 7: W = 1 sees only itself, W = 3 / 8 cut
    through the cartridge (the sink among the cut rows), W = 13 cuts it for
    the late queries only, W = 40 cuts nothing."""
    B, n, Hq, Hkv, d, p = 2, 7, 4, 2, 8, 9
    P = _problem(80 + window, B, n, Hq, Hkv, d, p)
    o, lse = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], window=window)
    o_t, lse_t = tf.cartridge_attention(_t(P["q"]), _t(P["k"]), _t(P["v"]), _t(P["kc"]),
                                        _t(P["vc"]), window=window)
    np.testing.assert_allclose(o, o_t.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.permute(0, 1, 2).numpy(), rtol=0, atol=1e-12)
    g = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], window=window)
    g_t = tf.cartridge_grads(_t(P["q"]), _t(P["k"]), _t(P["v"]), _t(P["kc"]), _t(P["vc"]),
                             _t(P["do"]), window=window)
    for a, b in zip(g, g_t):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-11)
    if window <= 3:
        # rows that no query's window reaches get no gradient at all
        far = p + 0 - window  # query 0 at position p reaches back to p - W + 1
        assert (g[3][1:max(far + 1, 1)] == 0).all() and (g[4][1:max(far + 1, 1)] == 0).all()


def test_window_wider_than_the_sequence_is_no_window():
    B, n, Hq, Hkv, d, p = 2, 6, 4, 2, 8, 5
    P = _problem(90, B, n, Hq, Hkv, d, p)
    a = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], window=p + n)
    b = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    ga = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"], window=p + n)
    gb = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"])
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("window", [1, 4, 11])
def test_windowed_decode_span_is_rows_of_windowed_forward(window):
    """Serving parity under a sliding window: the span's queries equal rows
    len .. len + span - 1 of the windowed training forward."""
    B, Hq, Hkv, d, p, span = 3, 4, 2, 16, 9, 2
    lens = np.array([0, 5, 2], dtype=np.int32)
    rows = 8
    rng = np.random.default_rng(52 + window)
    kc = rng.standard_normal((p, Hkv, d)) * 0.5
    vc = rng.standard_normal((p, Hkv, d)) * 0.5
    kraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    vraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    q = rng.standard_normal((B, span, Hq, d)) * 0.5
    k_cache = np.full((B, rows, Hkv, d), 7.0)
    v_cache = np.full((B, rows, Hkv, d), 7.0)
    for b in range(B):
        L = lens[b]
        k_cache[b, :L] = oracle.rope(kraw[b, :L], p)
        v_cache[b, :L] = vraw[b, :L]
    k_new = np.stack([kraw[b, lens[b]:lens[b] + span] for b in range(B)])
    v_new = np.stack([vraw[b, lens[b]:lens[b] + span] for b in range(B)])
    o, _, _ = oracle.decode_span(q, k_new, v_new, kc, vc, k_cache, v_cache, lens, window=window)
    for b in range(B):
        L = int(lens[b])
        qs = np.zeros((1, L + span, Hq, d))
        qs[0, L:] = q[b]
        of, _ = oracle.fwd(qs, kraw[None, b, :L + span], vraw[None, b, :L + span], kc, vc,
                           rows=(L, L + span), window=window)
        np.testing.assert_allclose(o[b], of[0, L:], rtol=0, atol=1e-13)


@pytest.mark.parametrize("window", [1, 5, 9])
def test_packed_window_matches_block_diagonal_windowed_attention(window):
    """Packed segments under a sliding window: one SDPA over the packed
    tokens with the block-diagonal mask intersected with the window (key
    position > query position - W)."""
    cu, Hq, Hkv, d, p = (0, 5, 5, 12, 13, 20), 4, 2, 16, 6
    T = cu[-1]
    P = _problem(100 + window, 1, T, Hq, Hkv, d, p)
    q, k, v, do = P["q"][0], P["k"][0], P["v"][0], P["do"][0]
    o, lse = oracle.fwd_packed(q, k, v, P["kc"], P["vc"], cu, window=window)
    o_t, lse_t = tf.packed_attention(_t(q), _t(k), _t(v), _t(P["kc"]), _t(P["vc"]), cu,
                                     window=window)
    np.testing.assert_allclose(o, o_t.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), rtol=0, atol=1e-12)
    g = oracle.bwd_packed(q, k, v, P["kc"], P["vc"], do, cu, window=window)
    g_t = tf.packed_grads(_t(q), _t(k), _t(v), _t(P["kc"]), _t(P["vc"]), _t(do), cu,
                          window=window)
    for a, b in zip(g, g_t):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-11)


def test_window_pin_catches_an_off_by_one():
    """Sensitivity of the window pin: a window one key wider (a plausible
    mistake in the reading of 'the W most recent keys') is caught."""
    B, n, Hq, Hkv, d, p, W = 1, 7, 4, 2, 8, 9, 5
    P = _problem(110, B, n, Hq, Hkv, d, p)
    o_wrong, _ = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], window=W + 1)
    o_t, _ = tf.cartridge_attention(_t(P["q"]), _t(P["k"]), _t(P["v"]), _t(P["kc"]),
                                    _t(P["vc"]), window=W)
    assert np.abs(o_wrong - o_t.numpy()).max() > 1e-3


def test_packed_pin_catches_unrestarted_positions():
    """Sensitivity of the packed pin: running the packed tokens as one
    sequence (positions not restarted, no segment mask) is caught."""
    cu, Hq, Hkv, d, p = (0, 5, 12), 4, 2, 16, 6
    T = cu[-1]
    P = _problem(111, 1, T, Hq, Hkv, d, p)
    o_wrong, _ = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"])
    o_t, _ = tf.packed_attention(_t(P["q"][0]), _t(P["k"][0]), _t(P["v"][0]), _t(P["kc"]),
                                 _t(P["vc"]), cu)
    assert np.abs(o_wrong[0, cu[1]:] - o_t.numpy()[cu[1]:]).max() > 1e-3
    # ... while the first segment, which starts the sequence, agrees
    np.testing.assert_allclose(o_wrong[0, :cu[1]], o_t.numpy()[:cu[1]], rtol=0, atol=1e-12)


def test_span_pin_catches_a_shared_position():
    """Sensitivity of the span pin: placing every span token at p + len
    (not p + len + t) and letting it see only rows 0 .. len is caught."""
    B, Hq, Hkv, d, p, span = 1, 4, 2, 16, 9, 3
    lens = np.array([4], dtype=np.int32)
    rows = 8
    rng = np.random.default_rng(112)
    kc = rng.standard_normal((p, Hkv, d)) * 0.5
    vc = rng.standard_normal((p, Hkv, d)) * 0.5
    kraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    vraw = rng.standard_normal((B, rows, Hkv, d)) * 0.5
    q = rng.standard_normal((B, span, Hq, d)) * 0.5
    k_cache = np.zeros((B, rows, Hkv, d))
    v_cache = np.zeros((B, rows, Hkv, d))
    L = int(lens[0])
    k_cache[0, :L] = oracle.rope(kraw[0, :L], p)
    v_cache[0, :L] = vraw[0, :L]
    qs = np.zeros((1, L + span, Hq, d))
    qs[0, L:] = q[0]
    of, _ = oracle.fwd(qs, kraw[None, 0, :L + span], vraw[None, 0, :L + span], kc, vc,
                       rows=(L, L + span))
    for t in range(1, span):
        o_wrong, _, _ = oracle.decode(q[:, t], kraw[:, L + t], vraw[:, L + t], kc, vc, k_cache,
                                      v_cache, lens)
        assert np.abs(o_wrong[0] - of[0, L + t]).max() > 1e-3


@pytest.mark.parametrize("name", ["causal_p3", "window4_p3"])
def test_golden_fixtures(name):
    """The oracle still reproduces its stored records (written by
    tests/golden/make_golden.py from the oracle alone)."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name + ".json")
    c = json.load(open(path))
    g = c["geometry"]
    P = {k: np.asarray(v, dtype=np.float64) for k, v in c["inputs"].items()}
    o, lse = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"],
                        frozen_prefix=g["frozen_prefix"], theta=g["theta"], window=g["window"])
    got = dict(o=o, lse=lse)
    got.update(zip(("dq", "dk", "dv", "dkc", "dvc"),
                   oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"],
                              frozen_prefix=g["frozen_prefix"], theta=g["theta"],
                              window=g["window"])))
    for k, v in c["outputs"].items():
        np.testing.assert_allclose(got[k], np.asarray(v), rtol=0, atol=1e-12, err_msg=k)
