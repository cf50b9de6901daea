"""Build the sm_103a CUDA library in-tree (attention_forward_02_gb300/_build/).

Three translation units (forward, backward, decoding), one -gencode
(compute_103a -> sm_103a), static cudart, no link against libcuda (the TMA
encoder is fetched through the runtime's driver entry-point query).  The same
three units are compiled a second time with FA_BOUNDS_CHECK into the checked
build (libfa_gb300_checked.so, device-side address checks; a test build).  All
six compile in parallel.
"""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libfa_gb300.so"
LIB = os.path.join(OUT_DIR, LIB_NAME)
# The same sources with the device-side address checks compiled in
# (FA_BOUNDS_CHECK; see include/fa.h): a test build, never the product path.
LIB_CHECKED = os.path.join(OUT_DIR, "libfa_gb300_checked.so")
SOURCES = [os.path.join(CSRC, f) for f in ("fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("fa_fwd_kernel.cuh", "fa1_fwd_kernel.cuh",
                                                  "fa_bwd_kernel.cuh", "fa_decode_kernel.cuh", "fa_decode_tc_kernel.cuh",
                                                  "fa_common.cuh",
                                                  "fa_host.h", "sm100_ptx.cuh")] + [
    os.path.join(INCLUDE, "fa.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA 13 toolkit on PATH)")


def _flags():
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC]


def compile_commands(out, verbose_ptxas=False, checked=False):
    """One nvcc -c per translation unit, then the link of the shared library."""
    objs, compiles = [], []
    for src in SOURCES:
        obj = out + "." + os.path.splitext(os.path.basename(src))[0] + ".o"
        cmd = [nvcc_path(), *_flags(), *(["-DFA_BOUNDS_CHECK"] if checked else []), "-c", "-o", obj, src]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        compiles.append(cmd)
    link = [nvcc_path(), *ARCH, "-shared", "-o", out, *objs]
    return compiles, link, objs


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build_library(force=False, verbose_ptxas=False, checked=True):
    """Compile the library (and, with checked=True, its checked build) if a
    source is newer than it; return the product library's path.  All
    translation units compile in parallel."""
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = [(LIB, False)] + ([(LIB_CHECKED, True)] if checked else [])
    jobs = [(lib, chk) for lib, chk in jobs if force or _stale(lib)]
    if not jobs:
        return LIB
    plans = []
    for lib, chk in jobs:
        tmp = lib + ".tmp%d" % os.getpid()
        plans.append((lib, tmp) + compile_commands(tmp, verbose_ptxas and not chk, chk))
    compiles = [c for _, _, cs, _, _ in plans for c in cs]
    with ThreadPoolExecutor(len(compiles)) as ex:
        for f in [ex.submit(subprocess.run, c, check=True) for c in compiles]:
            f.result()
    for lib, tmp, _, link, objs in plans:
        subprocess.run(link, check=True)
        for o in objs:
            os.remove(o)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose_ptxas=True))
