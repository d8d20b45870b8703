"""Build libgdn.so (the CUDA kernels + C ABI) in-tree for sm_103a, and its
checked variant libgdn_checked.so (-DGDN_CHECKS: the kernels range-check their
index arithmetic and report a failure as a device error bit).

Each .cu file compiles in parallel, once per variant, to an object under
``_build/``; the objects link into ``gated_delta_ssm_gb300/libgdn.so`` and
``gated_delta_ssm_gb300/libgdn_checked.so``. A source newer than a library
triggers a rebuild. Run ``python -m gated_delta_ssm_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgdn.so")
LIB_CHECKED = os.path.join(PKG, "libgdn_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                              + glob.glob(os.path.join(ROOT, "include", "*.h")))


def up_to_date() -> bool:
    for lib in (LIB, LIB_CHECKED):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(p) > t for p in _deps()):
            return False
    return True


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    variants = ((LIB, BUILD, []), (LIB_CHECKED, os.path.join(BUILD, "checked"), ["-DGDN_CHECKS"]))
    for _, objdir, _ in variants:
        os.makedirs(objdir, exist_ok=True)

    def compile_one(job) -> str:
        src, objdir, defs = job
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defs, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return obj

    jobs = [(src, objdir, defs) for _, objdir, defs in variants for src in sources()]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, jobs))
    n = len(sources())
    for k, (lib, _, _) in enumerate(variants):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs[k * n:(k + 1) * n], "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
