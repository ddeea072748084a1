"""Builds ``libcartattn.so`` (sm_103a) in-tree with nvcc.

Each ``csrc/*.cu`` file is compiled in parallel into ``_build/*.o`` and the
objects are linked into ``_build/libcartattn.so``.  Nothing is installed
outside this directory.

``build_test_hooks()`` builds a second library, ``_build/hooks/
libcartattn_hooks.so``, from the same sources with ``-DCART_TEST_HOOKS``: a
20 ms device wait limit and a host-set flag that withholds one barrier
arrival (``cart_test_skip_arrival``), so that a test can make a bounded wait
run out.  Only the tests load it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libcartattn.so")
HOOKS_OUT = os.path.join(OUT, "hooks")
HOOKS_LIB = os.path.join(HOOKS_OUT, "libcartattn_hooks.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(INCLUDE, "cartattn.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    return _build_lib(LIB, OUT, [], force, verbose)


def build_test_hooks(force: bool = False) -> str:
    return _build_lib(HOOKS_LIB, HOOKS_OUT, ["-DCART_TEST_HOOKS"], force, False)


def _build_lib(lib: str, out: str, defines: list, force: bool, verbose: bool) -> str:
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
