"""CPU checks of the work accounting bench.py reports against (the units
the roofline figures divide by), recomputed here by brute force."""
import numpy as np

import bench
from trained_kv_prefix_gb300 import synth


def _visible_pairs(n, p, window=0):
    """Visible (query, key) pairs of one head, counted key by key."""
    total = 0
    for i in range(n):
        qpos = p + i
        for kpos in range(p + i + 1):
            if window <= 0 or qpos - kpos < window:
                total += 1
    return total


def test_pairs_per_head_matches_brute_force():
    for n, p in ((1, 0), (7, 3), (33, 64)):
        s = synth.TrainShape("t", B=1, n=n, Hq=1, Hkv=1, d=64, p=p)
        assert s.pairs_per_head() == _visible_pairs(n, p)


def test_selfstudy_flop_figures():
    s = synth.SELFSTUDY
    assert s.pairs_per_head() == 2_621_952
    assert abs(s.fwd_flops() - 171.8e9) < 0.1e9
    assert abs(s.fwd_flops() + s.bwd_flops() - 601.4e9) < 0.1e9
    fwd, unit = bench.kernel_work("fwd", s, synth.DECODE, np.zeros(64, dtype=np.int32))
    dkdv, _ = bench.kernel_work("bwd_dkdv", s, synth.DECODE, np.zeros(64, dtype=np.int32))
    dq, _ = bench.kernel_work("bwd_dq", s, synth.DECODE, np.zeros(64, dtype=np.int32))
    assert unit == "flop" and fwd == s.fwd_flops()
    assert dkdv + dq == s.bwd_flops()  # the backward's five GEMMs split 4 : 1


def test_decode_bytes_by_hand():
    d = synth.DECODE
    lens = np.array([0, 5, 1024] + [7] * (d.B - 3), dtype=np.int32)
    row = d.Hkv * d.d * 2                        # one K or V row, bf16
    cart = 2 * d.p * row                         # the shared cartridge, once
    priv = sum(2 * (int(L) + 1) * row for L in lens)  # rows 0..L_b, K and V
    qo = d.B * 2 * d.Hq * d.d * 2                # q in, o out
    kv_new = d.B * 2 * row                       # k_new, v_new in
    append = d.B * 2 * row                       # the appended K and V rows
    lens_bytes = d.B * 4
    assert bench.decode_bytes(d, lens) == cart + priv + qo + kv_new + append + lens_bytes


def test_window_pair_count_used_in_the_notes():
    """The windowed throughput figures count min(p + i + 1, W) keys per query."""
    n, p = 40, 30
    for W in (1, 16, 50, 200):
        i = np.arange(n)
        assert int(np.minimum(p + i + 1, W).sum()) == _visible_pairs(n, p, W)
