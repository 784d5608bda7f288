"""Build ``lib/libspecverify.so`` (the CUDA verification library) in-tree.

One translation unit, compiled for sm_103a only.  The result is git-ignored;
every machine that runs the library builds it from source.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SRC_DIR = PKG / "csrc"
MAIN = SRC_DIR / "spec_verify.cu"
INCLUDE = ROOT / "include"
LIB = PKG / "lib" / "libspecverify.so"

NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo",
              "-gencode", "arch=compute_103a,code=sm_103a",
              "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify.so")


def sources():
    return [MAIN, *sorted(SRC_DIR.glob("*.cuh")), INCLUDE / "spec_verify.h"]


def is_stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(s.stat().st_mtime > t for s in sources())


def build_command(out: Path, defines=()):
    return [nvcc(), *NVCC_FLAGS, *[f"-D{d}" for d in defines], f"-I{INCLUDE}", str(MAIN),
            "-o", str(out)]


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile the library if it is missing or older than its sources."""
    if not force and not is_stale():
        return LIB
    LIB.parent.mkdir(parents=True, exist_ok=True)
    tmp = LIB.with_name(f".{LIB.name}.tmp{os.getpid()}")
    cmd = build_command(tmp)
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
