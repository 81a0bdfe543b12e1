"""Build the CUDA library ``_build/libkvcs.so`` for sm_103a with nvcc.

One translation unit, one ``-gencode``; the CUDA runtime is linked
statically so the library needs nothing but the driver at run time.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "libkvcs.so"
SOURCES = [CSRC / "kvcs.cu"]
DEPS = SOURCES + sorted(CSRC.glob("*.cuh")) + [INCLUDE / "kvcs.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required")
    return cand


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile unless the library is newer than every source and header."""
    if (not force and LIB.exists()
            and LIB.stat().st_mtime >= max(p.stat().st_mtime for p in DEPS)):
        return LIB
    OUT_DIR.mkdir(exist_ok=True)
    tmp = OUT_DIR / f"libkvcs.so.tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-std=c++17", "-lineinfo", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
           "-cudart", "static", f"-I{INCLUDE}", f"-I{CSRC}",
           *(["-Xptxas", "-v"] if verbose else []),
           *map(str, SOURCES), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
