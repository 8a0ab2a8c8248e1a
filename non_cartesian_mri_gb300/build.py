"""Build libmri.so in-tree with nvcc for sm_103a.

The translation units compile in parallel to objects under ``_build/`` and
are linked into ``_build/libmri.so`` (CUDA runtime linked statically).  A
build is skipped when the library is newer than every source and header.
ptxas register / spill reports land in ``_build/ptxas_<unit>.log``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmri.so")

UNITS = ["mri_abi.cu", "kernels_single.cu", "kernels_coils.cu", "kernels_grid.cu",
         "kernels_grid_tc.cu", "kernels_toeplitz.cu", "kernels_gridding.cu", "microbench.cu",
         "noalloc.cu", "kernels_coils_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmri.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, defines=(), out: str | None = None) -> str:
    """Compile and link libmri.so; return its path.

    ``defines`` (e.g. ``["MRI_PAIR_NP_FP32_Q=2"]``) and ``out`` build a variant
    library elsewhere, for tuning sweeps; the default build is ``LIB``.
    """
    lib = LIB if out is None else out
    if not force and out is None and not defines and up_to_date():
        return LIB
    bdir = BUILD if out is None else os.path.dirname(os.path.abspath(out))
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    dflags = [f"-D{d}" for d in defines]
    tag = "" if out is None else "_" + os.path.basename(out).replace(".so", "")

    def compile_unit(unit):
        src = os.path.join(CSRC, unit)
        obj = os.path.join(bdir, unit.replace(".cu", f"{tag}.o"))
        cmd = [nvcc, *ARCH, *FLAGS, *dflags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(os.path.join(bdir, f"ptxas_{unit.replace('.cu', '')}{tag}.log"), "w") as fh:
            fh.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stderr[-4000:]}")
        if verbose:
            print(f"compiled {unit}")
        return obj

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libmri.so failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
