"""Build libddp_gb300.so in-tree with nvcc for sm_103a.

    python -m gradient_sync_plan_gb300.build [--force] [--verbose-ptxas]

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  Only the GB300 target is built
(``-gencode arch=compute_103a,code=sm_103a``); the host side is plain C++17
with no architecture-specific flags, so the same command builds on x86-64 and
on the Arm (Grace) host of a GB300 node.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libddp_gb300.so")

SOURCES = ["ring_kernels.cu", "ring_tma.cu", "ring_static.cu", "ring_persistent.cu", "tree_kernels.cu", "bucket_kernels.cu", "ddp_api.cpp", "ddp_planner.cpp", "reducer.cpp"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(src: str, ptxas_verbose: bool) -> list:
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if src.endswith(".cu"):
        f = common + GENCODE + ["-lineinfo", "--expt-relaxed-constexpr"]
        if ptxas_verbose:
            f += ["-Xptxas", "-v"]
        return f
    return common + ["-x", "c++"]


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES]
    paths += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    paths += [os.path.join(INCLUDE, "ddp.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc, *_flags(src, ptxas_verbose), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if (ptxas_verbose or not quiet) and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *GENCODE, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.verbose_ptxas, quiet=False))


if __name__ == "__main__":
    main()
