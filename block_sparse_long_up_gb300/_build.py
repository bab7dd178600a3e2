"""Build libup.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each .cu file is compiled in parallel into _build/, then linked with
``nvcc -shared``.  A rebuild happens only when a source or header is newer than
the library.  ``build(checked=True)`` makes the checked variant instead
(_build_checked/libup_checked.so, compiled with -DUP_CHECK_BOUNDS: every kernel
tests its index ranges and reports a miss through UP_DEVERR_BOUNDS).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libup.so")
OUT_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(OUT_CHECKED, "libup_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libup.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [__file__])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    out, lib = (OUT_CHECKED, LIB_CHECKED) if checked else (OUT, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-DUP_CHECK_BOUNDS"] if checked else []

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        log = os.path.join(out, os.path.basename(src)[:-3] + ".ptxas.txt")
        with open(log, "w") as f:
            f.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    build(force=True, verbose=True)
