"""cart_attn_decode_noalloc: the decode step for callers that cannot allocate
device memory (a serving loop under a fixed device-memory budget, where a
cudaMalloc would synchronize the device; a plain C host with no device
allocator).  Its scratch is a static device array inside the library.

Checked through the C ABI against cart_attn_decode (which takes a caller
workspace) on two calls in a row with different inputs, so that whatever the
first call leaves in the shared array cannot leak into the second.  This file
is collected last and builds / loads the library itself, so it also passes
when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from tests import gpu_helpers as gh
from trained_kv_prefix_gb300 import cartattn, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from trained_kv_prefix_gb300 import build
    build.build()
    L = cartattn.lib()
    vp = ctypes.c_void_p
    L.cart_attn_decode_noalloc.argtypes = [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_double] + \
        [vp] * 7 + [ctypes.c_int, vp, vp, vp]
    L.cart_attn_decode_noalloc.restype = ctypes.c_int
    return L


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def _noalloc(L, s, g):
    o = torch.empty_like(g["q"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.cart_attn_decode_noalloc(s.B, s.Hq, s.Hkv, s.d, s.p, s.scale, s.theta, _p(g["q"]),
                                    _p(g["k_new"]), _p(g["v_new"]), _p(g["kc"]), _p(g["vc"]),
                                    _p(g["k_cache"]), _p(g["v_cache"]), s.cache_rows, _p(g["lens"]),
                                    _p(o), stream)
    return rc, o


CASES = [
    synth.DECODE,   # 64 conversations behind one p = 4096 cartridge
    synth.DecodeShape("small", B=3, Hq=8, Hkv=2, d=128, p=300, max_private=200, seed=31,
                      fixed_len=(0, 129, 200)),
]


def test_noalloc_matches_workspace_decode_twice_in_a_row(lib):
    outs = []
    for s in CASES:                     # two calls in a row, different inputs
        inp = synth.decode_inputs(s)
        g1 = {k: v.cuda() for k, v in inp.items()}
        g2 = {k: v.cuda() for k, v in inp.items()}
        rc, o_na = _noalloc(lib, s, g1)
        assert rc == 0, cartattn.STATUS.get(rc, rc)
        o_ws = cartattn.cart_attn_decode(g2["q"], g2["k_new"], g2["v_new"], g2["kc"], g2["vc"],
                                         g2["k_cache"], g2["v_cache"], g2["lens"], theta=s.theta)
        torch.cuda.synchronize()
        assert cartattn.device_status() == 0
        a, b = synth.f64(o_na), synth.f64(o_ws)
        assert gh.max_abs(a, b) <= gh.FWD_MAXABS and gh.rel_l2(a, b) <= gh.FWD_RELL2
        for name in ("k_cache", "v_cache"):
            np.testing.assert_array_equal(g1[name].view(torch.int16).cpu().numpy(),
                                          g2[name].view(torch.int16).cpu().numpy())
        outs.append(a)
    # and once more on the first case after the second overwrote the scratch
    s = CASES[0]
    g = {k: v.cuda() for k, v in synth.decode_inputs(s).items()}
    rc, o = _noalloc(lib, s, g)
    torch.cuda.synchronize()
    assert rc == 0
    np.testing.assert_array_equal(synth.f64(o), outs[0])


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 4096 conversations x 32 heads x 128 dims of rotated bf16 queries alone
    # fill the 32 MiB scratch
    nb = 4096
    s = synth.DecodeShape("huge", B=nb, Hq=32, Hkv=8, d=128, p=4096, max_private=64, seed=1,
                          fixed_len=tuple([0] * nb))
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(nb, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.cart_attn_decode_noalloc(s.B, s.Hq, s.Hkv, s.d, s.p, s.scale, s.theta, _p(t), _p(t),
                                      _p(t), _p(t), _p(t), _p(t), _p(t), s.cache_rows, _p(lens),
                                      _p(t), stream)
    assert rc == -4  # CART_ERR_WORKSPACE: needs more than the static scratch
    assert (t.cpu() == 0).all()
