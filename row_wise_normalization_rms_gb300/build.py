"""Builds librmsnorm.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel, then linked into a
shared library with the CUDA runtime linked statically.  The build is
skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = ROOT / "_build"
LIB_PATH = PKG / "librmsnorm.so"
SOURCES = ["api.cu", "fwd_registers.cu", "bwd_registers.cu", "scalar.cu", "staged.cu", "noalloc.cu",
           "layernorm.cu", "chunked.cu", "quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build librmsnorm.so")


def _inputs():
    files = [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h"))
    return files + list(INCLUDE.glob("*.h")) + [Path(__file__)]


def up_to_date() -> bool:
    if not LIB_PATH.exists():
        return False
    t = LIB_PATH.stat().st_mtime
    return all(f.stat().st_mtime <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile and link librmsnorm.so; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    BUILD_DIR.mkdir(exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = BUILD_DIR / (Path(src).stem + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *CFLAGS, "-Xptxas", "-v", "-c", str(CSRC / src), "-o", str(obj)]
        log = open(BUILD_DIR / (Path(src).stem + ".ptxas.txt"), "w")
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, p, log in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = "\n".join((BUILD_DIR / (Path(s).stem + ".ptxas.txt")).read_text()[-4000:] for s in failed)
        raise RuntimeError(f"nvcc failed for {failed}:\n{msgs}")
    tmp = LIB_PATH.with_suffix(".so.tmp")
    link = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        for src in SOURCES:
            sys.stdout.write((BUILD_DIR / (Path(src).stem + ".ptxas.txt")).read_text())
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
