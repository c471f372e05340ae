"""Build step of the CUDA library: nvcc for sm_103a, one shared object, in-tree."""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libmamba_ssd.so")
LIB_CHECKED = os.path.join(PKG, "libmamba_ssd_checked.so")  # debug build: every kernel's global indices range-checked
SOURCES = ["ssd_api.cu", "ssd_simt.cu", "ssd_tc.cu", "ssd_step.cu", "ssd_varlen.cu", "ssd_conv.cu", "ssd_noalloc.cu", "ssd_host.cu",
           "ssd_segstate.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-I", os.path.join(ROOT, "include"), *extra]


def build(verbose: bool = False, ptxas_info: bool = False, checked: bool = False) -> str:
    """Compile every translation unit in parallel and link libmamba_ssd.so (checked: the bounds-checked debug
    library libmamba_ssd_checked.so, in which an out-of-range global index is reported instead of used)."""
    objdir = os.path.join(PKG, "_build_checked" if checked else "_build")
    os.makedirs(objdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checked:
        extra.append("-DSSD_BOUNDS_CHECK")
    out = LIB_CHECKED if checked else LIB

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
