"""Compile libffpa.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

    python -m exact_headdim_attention_gb300.build [--force]

The library is written to ``exact_headdim_attention_gb300/_build/libffpa.so``
(git-ignored).  nvcc cross-compiles without a GPU, so this runs on any host
with the CUDA 13 toolkit.
"""
from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT = PKG / "_build" / "libffpa.so"
SOURCES = [CSRC / "ffpa_fwd.cu"]
DEPS = SOURCES + [CSRC / "ptx.cuh", INCLUDE / "ffpa.h"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or "/usr/local/cuda/bin/nvcc"
    return cand if Path(cand).exists() else "nvcc"


def flags() -> list[str]:
    return ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", f"-I{INCLUDE}", f"-I{CSRC}"]


def stale() -> bool:
    if not OUT.exists():
        return True
    t = OUT.stat().st_mtime
    return any(p.stat().st_mtime > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not stale():
        return OUT
    OUT.parent.mkdir(parents=True, exist_ok=True)
    tmp = OUT.with_suffix(".so.tmp")
    cmd = [nvcc(), *flags(), *map(str, SOURCES), "-o", str(tmp)]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
