"""Build the sm_103a CUDA library in-tree (attention_forward_02_gb300/_build/).

Three translation units (forward, backward, decoding) compiled in parallel, one
-gencode (compute_103a -> sm_103a), static cudart, no link against libcuda
(the TMA encoder is fetched through the runtime's driver entry-point query).
Compiles in well under a minute.
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
SOURCES = [os.path.join(CSRC, f) for f in ("fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("fa_fwd_kernel.cuh", "fa1_fwd_kernel.cuh",
                                                  "fa_bwd_kernel.cuh", "fa_decode_kernel.cuh",
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


def compile_commands(out, verbose_ptxas=False):
    """One nvcc -c per translation unit, then the link of the shared library."""
    objs, compiles = [], []
    for src in SOURCES:
        obj = out + "." + os.path.splitext(os.path.basename(src))[0] + ".o"
        cmd = [nvcc_path(), *_flags(), "-c", "-o", obj, src]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        compiles.append(cmd)
    link = [nvcc_path(), *ARCH, "-shared", "-o", out, *objs]
    return compiles, link, objs


def build_library(force=False, verbose_ptxas=False):
    """Compile the library if a source is newer than it; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(p) <= t for p in DEPS):
            return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    compiles, link, objs = compile_commands(tmp, verbose_ptxas)
    with ThreadPoolExecutor(len(compiles)) as ex:
        for f in [ex.submit(subprocess.run, c, check=True) for c in compiles]:
            f.result()
    subprocess.run(link, check=True)
    for o in objs:
        os.remove(o)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose_ptxas=True))
