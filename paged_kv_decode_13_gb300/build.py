"""Build libpkv.so in-tree with nvcc for sm_103a.

Nine attention translation units (three compute variants x three padded
head_dims) and the C-ABI unit compile in parallel, then link into one shared
library next to this file.  Objects go to ``_build/`` (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
         "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")


def _sources():
    units = []
    for variant in (0, 1, 2):
        for dp in (64, 128, 256):
            units.append((os.path.join(CSRC, "attend_inst.cu"), f"attend_{variant}_{dp}.o",
                          [f"-DPKV_INST_VARIANT={variant}", f"-DPKV_INST_DP={dp}"]))
    units.append((os.path.join(CSRC, "api.cu"), "api.o", []))
    return units


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "pkv.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libpkv.so."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(unit):
        src, obj, defs = unit
        cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", src, "-o", os.path.join(OUT, obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {obj}:\n{r.stderr}")
        return obj, r.stderr

    units = _sources()
    workers = min(len(units), max(2, os.cpu_count() or 2))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(compile_one, units))
    if verbose:
        for obj, err in results:
            sys.stderr.write(f"== {obj}\n{err}")
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [os.path.join(OUT, o) for _, o, _ in units]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
