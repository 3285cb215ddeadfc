"""Builds libmla_decode.so (the C-ABI CUDA library) in the package directory.

nvcc, sm_103a only, one translation unit per source compiled in parallel,
static CUDA runtime.  Object files go to the package's _build/ directory.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libmla_decode.so"
SOURCES = ["mla_decode.cu", "mla_decode_small.cu", "mla_sched.cu", "mla_cache.cu", "mla_api.cu", "mla_host.cu"]
HEADERS = ["sm103_ptx.cuh", "mla_internal.h", "mla_walk.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MLA decode library needs the CUDA 13 toolkit")


def _inputs():
    public = PKG.parent / "include" / "mla_decode.h"
    return [CSRC / s for s in SOURCES] + [CSRC / h for h in HEADERS] + [public, Path(__file__)]


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and up_to_date():
        return LIB
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", str(PKG.parent / "include"), "--expt-relaxed-constexpr"]
    if verbose:
        common += ["-Xptxas", "-v"]

    # object and library names carry the process id, so that builds started at
    # the same time (parallel test workers) never read each other's files
    def compile_one(src: str) -> Path:
        obj = BUILD / f"{Path(src).stem}.{os.getpid()}.o"
        cmd = [cc, "-c", str(CSRC / src), "-o", str(obj)] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    cmd = [cc, "-shared", "-o", str(tmp)] + [str(o) for o in objs] + ARCH + ["-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        o.unlink(missing_ok=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
