"""Compile the fp64 CPU oracle (``oracle.c``) into ``liboracle.so``.

Test infrastructure: only the test suite, the smoke check and the benchmark's
CPU-baseline leg load the result.  The flags keep IEEE semantics on every host
(no fast-math, no FMA contraction), so x86 and Arm builds agree.
"""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SRC = HERE / "oracle.c"
LIB = HERE / "liboracle.so"

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra", "-pthread", "-D_POSIX_C_SOURCE=200809L"]


def build_oracle(force: bool = False) -> Path:
    """Build ``liboracle.so`` if it is missing or older than its source."""
    if (not force and LIB.exists()
            and LIB.stat().st_mtime >= SRC.stat().st_mtime):
        return LIB
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    cmd = ["gcc", *CFLAGS, str(SRC), "-o", str(tmp), "-lm", "-pthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
