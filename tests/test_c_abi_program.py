"""The C ABI from a plain C program (tests/c_abi_example.c): it compiles
against include/kvcs.h alone, links libkvcs.so, and on the GPU its results
equal a closed form."""

import shutil
import subprocess
from pathlib import Path

import pytest

import paged_kv_cache_kvcs_gb300 as K
from paged_kv_cache_kvcs_gb300 import _binding as B

ROOT = Path(__file__).resolve().parent.parent


def build_example(out_dir: Path) -> Path:
    K.load_library()                      # the library exists
    lib_dir = B.LIB_PATH.parent
    exe = out_dir / "c_abi_example"
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-o", str(exe), str(ROOT / "tests" / "c_abi_example.c"),
                    "-I", str(ROOT / "include"), "-L", str(lib_dir), "-lkvcs",
                    "-Xlinker", f"-rpath,{lib_dir}"], check=True, capture_output=True)
    return exe


def test_example_compiles_and_links(tmp_path):
    assert build_example(tmp_path).exists()


@pytest.mark.gpu
def test_example_runs(tmp_path):
    exe = build_example(tmp_path)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout
