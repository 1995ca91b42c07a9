"""Compile the CUDA sources of this package into ``libsa.so`` (in-tree).

nvcc for sm_103a only, one translation unit per process, linked with the
static CUDA runtime so that the library loads on machines without a GPU
(every call then returns SA_ERR_CUDA).  The same sources are also built with
SA_CHECKED into ``libsa_checked.so``: the same ABI, with the kernels testing
the addresses they compute from run-time values (a failed test sets the
error word's bounds bit, SA_ERR_BOUNDS, and skips the access).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libsa.so")
LIB_CHECKED = os.path.join(PKG, "libsa_checked.so")
BUILD_DIR = os.path.join(ROOT, "_build")
# library -> (extra nvcc flags, object directory)
VARIANTS = {LIB: ([], BUILD_DIR), LIB_CHECKED: (["-DSA_CHECKED"], os.path.join(BUILD_DIR, "checked"))}
SOURCES = ["sa_attn.cu", "sa_gemm.cu", "sa_topk.cu", "sa_quant.cu", "sa_api.cu", "sa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "sa.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build both libraries (the translation units of both in one pool) and
    return the path of ``libsa.so``."""
    todo = [lib for lib in VARIANTS if force or not up_to_date(lib)]
    if not todo:
        return LIB
    nvcc = _nvcc()
    for lib in todo:
        os.makedirs(VARIANTS[lib][1], exist_ok=True)

    def compile_one(job):
        lib, src = job
        defs, objdir = VARIANTS[lib]
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({os.path.basename(lib)}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    jobs = [(lib, src) for lib in todo for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for lib in todo:
        mine = [o for (l, _), o in zip(jobs, objs) if l == lib]
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *mine]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({os.path.basename(lib)}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
