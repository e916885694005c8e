"""Builds libmoe.so in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to an object in _build/, then nvcc
links the shared library next to this file. Run `python -m
token_dispatch_expert_moe_gb300.build` or call build().
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + INCLUDE, "-I" + CSRC]
SOURCES = ["api.cu", "route.cu", "route_bwd.cu", "dispatch.cu", "gemm_simt.cu", "gemm_tc.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, extra: list[str], obj_name: str) -> str:
    obj = os.path.join(BUILD, obj_name)
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


# The test build: the same library with the test hooks of gemm_tc.cu compiled
# in (MOE_FAULT_INJECT_STALL, MOE_GEMM_PAIR); only the failure-path and
# kernel-comparison tests load it, in processes of their own.
TEST_LIB = os.path.join(PKG, "libmoe_testhooks.so")
HOOKED = "gemm_tc.cu"


def _link(objs: list[str], out: str) -> None:
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-ldl"]   # -ldl: NVTX loads a profiler's hooks
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(verbose_ptxas: bool = False) -> str:
    """Compile and link libmoe.so (and the test build); returns libmoe.so's path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    jobs = [(s, extra, s.replace(".cu", ".o")) for s in SOURCES]
    jobs.append((HOOKED, ["-DMOE_TEST_HOOKS"], HOOKED.replace(".cu", "_hooks.o")))
    with ThreadPoolExecutor(len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(*j), jobs))
    prod = objs[:len(SOURCES)]
    _link(prod, LIB)
    hooked = [o for s, o in zip(SOURCES, prod) if s != HOOKED] + [objs[-1]]
    _link(hooked, TEST_LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
