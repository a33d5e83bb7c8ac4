"""Builds libmk.so (the decode megakernel and its C ABI) in-tree for sm_103a."""
from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
LIB = PKG / "libmk.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                     "-I", str(ROOT / "include")]
UNITS = ["megakernel.cu", "api.cu", "planner.cpp", "noalloc.cu", "pages.cpp"]


def _sources():
    return [CSRC / u for u in UNITS] + sorted(CSRC.glob("*.h")) + sorted(CSRC.glob("*.cuh")) + [
        ROOT / "include" / "mk.h"]


def build(force: bool = False, verbose_ptxas: bool = False) -> Path:
    if not force and LIB.exists():
        mt = LIB.stat().st_mtime
        if all(s.stat().st_mtime <= mt for s in _sources()):
            return LIB
    bdir = PKG / "_build"
    bdir.mkdir(exist_ok=True)
    objs = []
    for u in UNITS:
        src = CSRC / u
        obj = bdir / (src.stem + ".o")
        cmd = ["nvcc"] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose_ptxas and u == "megakernel.cu" else [])
        if src.suffix == ".cpp":
            cmd += ["-x", "c++"]
        cmd += ["-c", str(src), "-o", str(obj)]
        subprocess.check_call(cmd)
        objs.append(str(obj))
    tmp = LIB.with_suffix(".so.tmp")
    subprocess.check_call(["nvcc"] + ARCH + ["-shared", "-o", str(tmp)] + objs + ["-lcudart"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
