"""CPU-only checks of the C ABI boundary: the library builds for sm_103a,
loads, exports every entry point declared in include/cartattn.h, and rejects
bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

from trained_kv_prefix_gb300 import build as cbuild
from trained_kv_prefix_gb300 import cartattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cartattn.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "cartattn.h")).read()
    return sorted(set(re.findall(r"CART_API\s+[\w\s\*]+?\b(cart_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("cart_attn_fwd", "cart_attn_bwd", "cart_attn_decode", "cart_write_to_cache"):
        assert required in names
    assert set(names) == set(cartattn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.cart_status_string(0) == b"ok"
    assert lib.cart_status_string(-1) == b"bad geometry"
    assert lib.cart_status_string(-7) == b"a kernel gave up waiting"
    assert lib.cart_status_string(123) == b"unknown status"


@pytest.mark.parametrize("bad", [
    dict(Hq=6, Hkv=4),            # Hq % Hkv != 0
    dict(d=96),                   # unsupported head dim
    dict(frozen_prefix=5, p=4),   # frozen rows beyond the cartridge
    dict(n=0),                    # no real tokens
    dict(p=-1),
])
def test_workspace_query_rejects_bad_geometry(lib, bad):
    kw = dict(B=1, n=8, Hq=4, Hkv=2, d=64, p=4, frozen_prefix=1)
    kw.update(bad)
    g = cartattn.geom(**kw)
    assert cartattn.fwd_workspace_size(g, 0, 1) == 0
    assert cartattn.bwd_workspace_size(g, 0, 1) == 0


def test_workspace_sizes_are_positive_and_grow(lib):
    g1 = cartattn.geom(1, 128, 4, 2, 128, 16)
    g2 = cartattn.geom(2, 128, 4, 2, 128, 16)
    a, b = cartattn.fwd_workspace_size(g1, 0, 1), cartattn.fwd_workspace_size(g2, 0, 1)
    assert 0 < a < b
    assert cartattn.bwd_workspace_size(g1, 0, 1) > a
    assert cartattn.decode_workspace_size(64, 32, 8, 128, 4096, 1025) > 0
    assert cartattn.decode_workspace_size(4, 12, 4, 128, 16, 8) == 0   # G = 3 unsupported
    # span verify: the span's columns grow the workspace; G * span > 32 or a
    # span longer than the cache is refused
    one = cartattn.decode_span_workspace_size(64, 1, 32, 8, 128, 4096, 1025)
    assert one == cartattn.decode_workspace_size(64, 32, 8, 128, 4096, 1025)
    assert cartattn.decode_span_workspace_size(64, 8, 32, 8, 128, 4096, 1025) > one
    assert cartattn.decode_span_workspace_size(64, 9, 32, 8, 128, 4096, 1025) == 0
    assert cartattn.decode_span_workspace_size(4, 9, 8, 2, 128, 16, 8) == 0


def test_calls_validate_before_touching_the_device(lib):
    g = cartattn.geom(1, 8, 4, 2, 64, 4)
    null = ctypes.c_void_p(0)
    # NULL inputs
    rc = lib.cart_attn_fwd(ctypes.byref(g), 0, 1, null, null, null, null, null, null, null, null,
                           0, null)
    assert rc == -2
    # misaligned pointer
    odd = ctypes.c_void_p(0x1001)
    rc = lib.cart_attn_fwd(ctypes.byref(g), 0, 1, odd, odd, odd, odd, odd, odd, odd, odd, 0, null)
    assert rc == -2
    # bad dtype
    al = ctypes.c_void_p(0x1000)
    rc = lib.cart_attn_fwd(ctypes.byref(g), 7, 1, al, al, al, al, al, al, al, al, 1 << 30, null)
    assert rc == -3
    # workspace too small
    rc = lib.cart_attn_fwd(ctypes.byref(g), 0, 1, al, al, al, al, al, al, al, al, 16, null)
    assert rc == -4
    # cache write: stride smaller than a row
    rc = lib.cart_write_to_cache(al, al, 4, 2, 64, al, al, 64, 0, 0, null)
    assert rc == -1
    # composed-cartridge backward: a frozen row outside the cartridge, too many
    # rows, or a missing list
    rows = (ctypes.c_int * 65)(*([1] * 65))
    bad = (ctypes.c_int * 1)(4)  # p = 4: rows are 0..3
    for lst, cnt in ((bad, 1), (rows, 65), (None, 2)):
        rc = lib.cart_attn_bwd_parts(ctypes.byref(g), 0, 1, al, al, al, al, al, al, al, al, al,
                                     al, al, al, al, lst, cnt, 0, al, 1 << 30, null)
        assert rc == -1
    # packed segments: no table, a misaligned table, no tokens, more tokens
    # than B segments of n can hold
    gp = cartattn.geom(2, 8, 4, 2, 64, 4)
    odd4 = ctypes.c_void_p(0x1002)
    for total, cu in ((10, null), (10, odd4), (0, al), (17, al)):
        rc = lib.cart_attn_fwd_packed(ctypes.byref(gp), total, cu, 0, 1, al, al, al, al, al, al,
                                      al, al, 1 << 30, null)
        assert rc in (-1, -2), (total, cu, rc)
        rc = lib.cart_attn_bwd_packed(ctypes.byref(gp), total, cu, 0, 1, al, al, al, al, al, al,
                                      al, al, al, al, al, al, al, None, 0, 0, al, 1 << 30, null)
        assert rc in (-1, -2), (total, cu, rc)
    assert cartattn.fwd_packed_workspace_size(gp, 0, 0, 1) == 0
    assert cartattn.fwd_packed_workspace_size(gp, 16, 0, 1) > 0
    assert cartattn.bwd_packed_workspace_size(gp, 16, 0, 1) > cartattn.fwd_packed_workspace_size(
        gp, 16, 0, 1)
    # a negative sliding window
    gw = cartattn.geom(1, 8, 4, 2, 64, 4, window=-1)
    rc = lib.cart_attn_fwd(ctypes.byref(gw), 0, 1, al, al, al, al, al, al, al, al, 1 << 30, null)
    assert rc == -1
    rc = lib.cart_attn_decode_span(2, 1, -1, 16, 2, 128, 16, 0.1, 1e6, al, al, al, al, al, al,
                                   al, 8, al, al, al, 1 << 30, null)
    assert rc == -1
    # decode: unsupported group size
    rc = lib.cart_attn_decode(2, 6, 2, 128, 16, 0.1, 1e6, al, al, al, al, al, al, al, 8, al, al,
                              al, 1 << 20, null)
    assert rc == -1
    # span decode: span 0, span past the cache, too many query columns
    for span, rows in ((0, 8), (9, 8), (5, 64)):
        rc = lib.cart_attn_decode_span(2, span, 0, 16, 2, 128, 16, 0.1, 1e6, al, al, al, al, al, al,
                                       al, rows, al, al, al, 1 << 30, null)
        assert rc == -1, (span, rows)


def test_release_without_a_device_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.cart_release() == -5


def test_no_gpu_here_means_a_cuda_or_device_error(lib):
    """With valid arguments but no usable sm_103 device the call fails loudly
    instead of computing anything elsewhere."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    g = cartattn.geom(1, 8, 4, 2, 64, 4)
    al = ctypes.c_void_p(0x1000)
    ws = cartattn.fwd_workspace_size(g, 0, 1)
    rc = lib.cart_attn_fwd(ctypes.byref(g), 0, 1, al, al, al, al, al, al, al, al, ws, None)
    assert rc in (-5, -6)


def test_header_is_plain_c99():
    """The boundary header compiles as C99 (no C++ in the signatures)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-fsyntax-only", "-x", "c", os.path.join(ROOT, "include", "cartattn.h")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_plain_c_host_links_and_calls(lib, tmp_path):
    """A plain C program links only libcartattn.so and calls the ABI: the
    status strings and a workspace size (no device needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "host.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "cartattn.h"
int main(void) {
  cart_geom g = {2, 256, 8, 2, 128, 64, 1, 0.0883883f, 1.0e6, 0};
  size_t ws = cart_attn_fwd_workspace_size(&g, CART_BF16, CART_F32);
  g.window = -1;
  size_t bad = cart_attn_fwd_workspace_size(&g, CART_BF16, CART_F32);
  printf("%s|%s|%d|%d\n", cart_status_string(CART_OK), cart_status_string(CART_ERR_WORKSPACE),
         ws > 0, bad == 0);
  return 0;
}
""")
    so = cbuild.LIB
    exe = tmp_path / "host"
    r = subprocess.run([gcc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe), so, "-Wl,-rpath," + os.path.dirname(so)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok|workspace too small|1|1"
