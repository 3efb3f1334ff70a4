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
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT = PKG / "_build" / "libffpa.so"
# One translation unit per kernel plus the host side, compiled in parallel.
SOURCES = [CSRC / n for n in ("ffpa_cluster.cu", "ffpa_split.cu", "ffpa_bwd.cu", "ffpa_bwd_tiles.cu",
                              "ffpa_pair.cu", "ffpa_fp8.cu", "ffpa_fp8_split.cu", "ffpa_single.cu",
                              "ffpa_dual.cu", "ffpa_api.cu", "ffpa_noalloc.cu")]
DEPS = SOURCES + [CSRC / "ffpa_common.cuh", CSRC / "ffpa_bwd_common.cuh", CSRC / "ptx.cuh", INCLUDE / "ffpa.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or "/usr/local/cuda/bin/nvcc"
    return cand if Path(cand).exists() else "nvcc"


def flags() -> list[str]:
    """Compile flags of every translation unit."""
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}"]


def stale() -> bool:
    if not OUT.exists():
        return True
    t = OUT.stat().st_mtime
    return any(p.stat().st_mtime > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not stale():
        return OUT
    objdir = OUT.parent / "obj"
    objdir.mkdir(parents=True, exist_ok=True)
    jobs = [[nvcc(), *flags(), "-c", str(src), "-o", str(objdir / (src.stem + ".o"))]
            for src in SOURCES]
    if verbose:
        for cmd in jobs:
            print(" ".join(cmd))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, results):
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise subprocess.CalledProcessError(r.returncode, cmd)
    tmp = OUT.with_suffix(".so.tmp")
    link = [nvcc(), *ARCH, "-shared", *(str(objdir / (src.stem + ".o")) for src in SOURCES),
            "-o", str(tmp)]
    if verbose:
        print(" ".join(link))
    subprocess.run(link, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
