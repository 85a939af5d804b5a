"""Build of the CUDA library libgbssim.so for sm_103a (nvcc, in-tree).

Each .cu under csrc/ compiles in parallel to an object file; the objects link
into ``_build/libgbssim.so``.  The same sources compiled with
``-DGBSSIM_TEST_HOOKS`` link into ``_build/test/libgbssim_test.so``: the
product library plus the hooks only the tests use (staging modes that make the
bounded waits run out, forced row segments, the per-stage statistics dump).
The product library exports exactly what include/gbssim.h declares.  A rebuild
happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libgbssim.so")
TEST_BUILD = os.path.join(BUILD, "test")
TEST_LIB = os.path.join(TEST_BUILD, "libgbssim_test.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]
TEST_FLAGS = ["-DGBSSIM_TEST_HOOKS"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgbssim.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [
            os.path.join(CSRC, "exports.map"), os.path.abspath(__file__)]


def _up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def up_to_date() -> bool:
    return _up_to_date(LIB) and _up_to_date(TEST_LIB)


def _compile_all(targets, cc, verbose):
    """targets: [(out_dir, extra_flags)]; every source of every target in parallel."""
    procs, objs = [], {d: [] for d, _ in targets}
    for out_dir, extra in targets:
        os.makedirs(out_dir, exist_ok=True)
        for src in sources():
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
            cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
            objs[out_dir].append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            print(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(os.path.basename(src))
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    return objs


EXPORTS = os.path.join(CSRC, "exports.map")


def _link(cc, objs, lib):
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-Xlinker", f"--version-script={EXPORTS}", "-o", tmp,
                    *objs], check=True)
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, test_lib: bool = True) -> str:
    """Compile and link the library (and, with test_lib, the test build); returns
    the product library's path."""
    todo = []
    if force or not _up_to_date(LIB):
        todo.append((BUILD, [], LIB))
    if test_lib and (force or not _up_to_date(TEST_LIB)):
        todo.append((TEST_BUILD, TEST_FLAGS, TEST_LIB))
    if not todo:
        return LIB
    cc = nvcc()
    objs = _compile_all([(d, f) for d, f, _ in todo], cc, verbose)
    for d, _, lib in todo:
        _link(cc, objs[d], lib)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
