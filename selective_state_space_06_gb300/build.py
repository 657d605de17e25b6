"""Builds libmambascan.so in-tree with nvcc for sm_103a (no torch extension machinery).

Each .cu file compiles to an object in parallel; the objects then link into one shared
library next to this file. ``python selective_state_space_06_gb300/build.py`` runs it (the
package itself cannot be imported before the library exists).

``build(checked=True)`` builds the bounds-checked variant, libmambascan_checked.so: the same
sources with -DMAMBA_BOUNDS_CHECK, in which every global access whose offset a kernel computes
is checked against its buffer's length and an access outside is recorded instead of made.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmambascan.so")
LIB_CHECKED = os.path.join(HERE, "libmambascan_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["scan_plan.cu", "scan_fwd.cu", "scan_bwd.cu", "scan_bwd_tmem.cu", "mamba_scan_abi.cu", "conv1d.cu", "conv_abi.cu", "mamba_scan_noalloc.cu"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmambascan.so")


def _flags(verbose_ptxas: bool, checked: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
    if checked:
        f += ["-DMAMBA_BOUNDS_CHECK"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose_ptxas: bool = False, force: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "mamba_scan.h"))
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= max(map(os.path.getmtime, deps)):
        return lib
    objdir = os.path.join(HERE, "_build_checked" if checked else "_build")
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        r = subprocess.run([cc, *_flags(verbose_ptxas, checked), "-c", src, "-o", obj],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, force=True, checked="--checked" in sys.argv))
