"""Builds libkvs.so (the C-ABI library) in-tree for sm_103a with nvcc.

Usage: python -m paged_kv_cache_flash_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "libkvs.so"
SOURCES = ["kvs_decode.cu", "kvs_combine.cu", "kvs_blocks.cu", "kvs_kivi.cu", "kvs_host.cpp", "kvs_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libkvs.so)")


def _flags(ptxas_verbose: bool) -> list:
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "--expt-relaxed-constexpr",
         "-I", str(ROOT / "include"), *ARCH]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = [CSRC / s for s in SOURCES] + [CSRC / "kvs_internal.h", CSRC / "kvs_launch.h", CSRC / "kvs_ptx.h",
                                         CSRC / "kvs_pdl.cuh", ROOT / "include" / "kvs.h", Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> Path:
    if not force and not _stale():
        return LIB
    OUT_DIR.mkdir(exist_ok=True)
    cc = nvcc()
    flags = _flags(ptxas_verbose)

    def compile_one(src: str):
        obj = OUT_DIR / (Path(src).stem + ".o")
        lang = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
        cmd = [cc, *lang, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if not quiet or ptxas_verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = OUT_DIR / f"libkvs.tmp{os.getpid()}.so"
    cmd = [cc, "-shared", *ARCH, "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.verbose_ptxas, quiet=False))
