"""bench.py keeps its JSON-line contract: the reference arm on the CPU (the
oracle needs no GPU), our arm on the GPU, each as a subprocess."""

import json
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"}


def run(*args, timeout=900):
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = run("--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3")
    assert BASE_KEYS <= set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["config"]["workload"] == "tiny_paged_kv_checksum"
    # the same config keys as our arm's line
    assert {"parallelism", "memory_layout", "columns", "verify"} <= set(d["config"])


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode != 0


@pytest.mark.gpu
def test_our_arm_line():
    d = run("--config", "llama3_8b_small", "--steps", "5", "--warmup", "3", "--e2e-steps", "1",
            "--cpu-seconds", "1", "--other-cpu-seconds", "0.5")
    assert BASE_KEYS | {"roofline", "clocks", "gpu_launches", "ms_per_step"} <= set(d)
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    # with a workspace every step is the zeroing kernel and the checksum kernel
    per_step = 2 if d["config"]["work_share"].startswith("dynamic") else 1
    assert d["gpu_launches"] == 5 * per_step and d["higher_is_better"] is True
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    # the timed call's output against the oracle's sampled values
    assert d["parity"]["positions"] > 0 and d["parity"]["mismatches"] == 0
    cb = d["cpu_baseline"]
    assert cb["one_thread"]["cores"] == 1 and cb["one_thread"]["value"] > 0
    assert cb["python_tiny"]["value"] > 0
    assert {"parallelism", "memory_layout", "columns", "verify"} <= set(d["config"])


@pytest.mark.gpu
def test_write_line():
    d = run("--config", "llama3_8b_write_small", "--steps", "5", "--warmup", "3",
            "--cpu-seconds", "1")
    assert {"metric", "value", "unit", "roofline", "clocks", "cpu_baseline", "gpu_launches"} <= set(d)
    assert d["gpu_launches"] == 5 and d["roofline"]["kernel"] == "kvcs_write_kernel"
    assert d["parity"]["positions"] > 0 and d["parity"]["mismatches"] == 0


@pytest.mark.gpu
def test_replica_columns_line_checks_its_output():
    d = run("--config", "llama3_8b_small", "--steps", "3", "--warmup", "3", "--no-e2e",
            "--columns", "2", "--verify", "--cpu-seconds", "1", "--other-cpu-seconds", "0.5")
    assert d["parity"]["positions"] > 0 and d["parity"]["mismatches"] == 0
    assert "other_configs" not in d
