"""Compile the scalar C oracle (``kvcs_oracle.c``) into a shared library.

TEST INFRASTRUCTURE ONLY.  Plain gcc, no CUDA; runs on x86_64 and aarch64.
"""

from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SRC = HERE / "kvcs_oracle.c"
OUT_DIR = HERE / "_build"
LIB = OUT_DIR / "libkvcs_oracle.so"


def build(force: bool = False) -> Path:
    """Build ``_build/libkvcs_oracle.so`` unless it is newer than its source."""
    if not force and LIB.exists() and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    OUT_DIR.mkdir(exist_ok=True)
    tmp = OUT_DIR / f"libkvcs_oracle.so.tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
           "-pthread", str(SRC), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
