"""cart_attn_decode_noalloc: the decode step for callers that cannot allocate
device memory (a serving loop under a fixed device-memory budget, where a
cudaMalloc would synchronize the device; a plain C host with no device
allocator).  Its scratch is a static device array inside the library.

Checked through the C ABI against cart_attn_decode (which takes a caller
workspace): the same kernels run on the same inputs with the same split, so
the outputs and the appended cache rows must be identical bit for bit; the
output is also checked against the fp64 oracle at the forward tolerance.
Two calls in a row with different inputs, then the first again, so that
whatever one call leaves in the shared array cannot leak into the next.
This file is collected last and builds / loads the library itself, so it
also passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def _oracle_decode(s, inp):
    a = {k: synth.f64(v) for k, v in inp.items() if k != "lens"}
    o, _, _ = oracle.decode(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["k_cache"],
                            a["v_cache"], inp["lens"].numpy(), theta=s.theta)
    return o


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
        np.testing.assert_array_equal(o_na.view(torch.int16).cpu().numpy(),
                                      o_ws.view(torch.int16).cpu().numpy())
        for name in ("k_cache", "v_cache"):
            np.testing.assert_array_equal(g1[name].view(torch.int16).cpu().numpy(),
                                          g2[name].view(torch.int16).cpu().numpy())
        a, ref = synth.f64(o_na), _oracle_decode(s, inp)
        assert gh.max_abs(a, ref) <= gh.FWD_MAXABS and gh.rel_l2(a, ref) <= gh.FWD_RELL2
        outs.append(a)
    # and once more on the first case after the second overwrote the scratch
    s = CASES[0]
    g = {k: v.cuda() for k, v in synth.decode_inputs(s).items()}
    rc, o = _noalloc(lib, s, g)
    torch.cuda.synchronize()
    assert rc == 0
    np.testing.assert_array_equal(synth.f64(o), outs[0])


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 4096 conversations behind a p = 4096 cartridge: the cartridge pass's
    # f32 partials alone (16384 stacked query rows per kv head) are 64 MiB
    nb = 4096
    s = synth.DecodeShape("huge", B=nb, Hq=32, Hkv=8, d=128, p=4096, max_private=64, seed=1,
                          fixed_len=tuple([0] * nb))
    need = cartattn.decode_workspace_size(s.B, s.Hq, s.Hkv, s.d, s.p, s.cache_rows)
    assert need > 32 << 20  # more than CART_DECODE_NOALLOC_SCRATCH_BYTES
    # null tensors: the size check comes first, and if it ever stopped
    # refusing this problem the pointer check would (nothing is launched)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.cart_attn_decode_noalloc(s.B, s.Hq, s.Hkv, s.d, s.p, s.scale, s.theta, None, None,
                                      None, None, None, None, None, s.cache_rows, None, None,
                                      stream)
    assert rc == -4  # CART_ERR_WORKSPACE: needs more than the static scratch
