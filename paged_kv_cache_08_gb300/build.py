"""Build libpa.so (CUDA kernels + C ABI + host pool) for sm_103a, in-tree.

    python -m paged_kv_cache_08_gb300.build [--force]

Translation units compile in parallel; a unit is rebuilt when it or any header
under csrc/ or include/ is newer than its object file.
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
BUILD = PKG / "_build"
LIB = BUILD / "libpa.so"

CUDA_SOURCES = ["api.cu", "cache_write.cu", "copy_blocks.cu", "decode_fma.cu", "decode_mma.cu", "decode_persist.cu", "decode_planned.cu",
                "decode_static.cu",
                "prefill_mma.cu", "prefill_tc.cu"]
CXX_SOURCES = ["pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda")) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def _headers_mtime() -> float:
    hs = list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    return max((h.stat().st_mtime for h in hs), default=0.0)


def _compile(src: Path, obj: Path, extra: list[str]) -> None:
    if src.suffix == ".cu":
        cmd = [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "--expt-relaxed-constexpr", *extra, "-c", str(src), "-o", str(obj)]
    else:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)


def build(force: bool = False, verbose_ptxas: bool = False) -> Path:
    BUILD.mkdir(parents=True, exist_ok=True)
    hdr = _headers_mtime()
    jobs = []
    objs = []
    for name in CUDA_SOURCES + CXX_SOURCES:
        src = CSRC / name
        obj = BUILD / (name + ".o")
        objs.append(obj)
        stale = force or not obj.exists() or obj.stat().st_mtime < max(src.stat().st_mtime, hdr)
        if stale:
            jobs.append((src, obj))
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if jobs:
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            list(ex.map(lambda j: _compile(j[0], j[1], extra), jobs))
    if force or jobs or not LIB.exists():
        tmp = BUILD / f"libpa.so.tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv))
