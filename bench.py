"""Benchmark: KV-cache block checksums on one GB300 (or N replicas).

One *step* is one ``kvcs_block_checksums`` call over the whole workload: every
block position of every request, over every layer's paged K/V.  The default
workload is the Llama-3-8B-shaped one (32 layers, 8 KV heads, head_size 128,
bf16, block_size 16, 64 requests of 512..4096 tokens, ~19 GB of KV).

Printed (rank 0, one JSON line):
  value      KV GB/s read, device-timed with CUDA events over K steps, KV
             already resident in HBM.  The KV (tens of GB) is far larger than
             the 129 MB L2, so no flush is needed between steps.
  e2e        the same metric through the public API with host buffers: each
             step copies the KV pools and block tables from pinned host
             memory into the device pools (a load of offloaded KV), runs the
             call and reads the checksums back.
  roofline   the bulk-copy kernel against measured HBM bandwidth.
  cpu_baseline  the CPU oracle (scalar C, all host cores) on a sample.

``--impl reference`` times the CPU oracle instead (the reference arm).
With ``torchrun --nproc-per-node N`` every rank checksums its own replica of
the workload (weak scaling); the checksum needs no exchange between ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

METRIC = ("KV checksum GB/s read + blocks/s (device-timed, 1×GB300) and "
          "% of HBM peak")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_workload(name: str, seed: int, device):
    from paged_kv_cache_kvcs_gb300 import workloads as W
    if name == "llama3_8b":
        return W.llama3_8b(seed, device)
    if name == "llama3_8b_small":      # 2.5 GB, 8 x 152 positions: ncu captures
        return W.llama3_8b(seed, device, num_requests=19, min_len=1024, max_len=1024)
    if name == "llama3_8b_mid":        # 5.1 GB, 16 x 152 positions, 1024 units a SM: the
        # smallest 8B-shaped call with the dynamic share-out (ncu captures)
        return W.llama3_8b(seed, device, num_requests=38, min_len=1024, max_len=1024)
    if name == "mla":
        return W.mla(seed, device)
    if name == "mla_small":            # 608 positions = 4 x 152, 2.7 GB: ncu captures
        return W.mla(seed, device, num_requests=19, tokens=2048)
    if name == "llama3_70b":
        return W.llama3_70b(seed, device)
    if name == "llama3_70b_small":     # 608 positions = 4 x 152, 1.6 GB: ncu captures
        return W.llama3_70b(seed, device, num_requests=19, tokens=512)
    if name.startswith("llama3_70b_r"):  # request-count sweep point
        return W.llama3_70b(seed, device, num_requests=int(name[len("llama3_70b_r"):]))
    if name == "tiny":
        return W.tiny(seed, device)
    if name == "llama3_8b_decode_hnd":  # newest block of 16384 requests, 1 token each, HND
        return W.llama3_8b_decode(seed, device)
    if name == "llama3_8b_decode_nhd":
        return W.llama3_8b_decode(seed, device, layout=W.LAYOUT_NHD)
    if name == "llama3_8b_decode_hnd_small":   # 2048 requests: ncu captures
        return W.llama3_8b_decode(seed, device, num_requests=2048)
    if name == "mamba2":                # Mamba2-shaped running states, 10.9 GB
        return W.mamba2(seed, device)
    if name == "mamba2_small":          # 16 requests, 2.7 GB: ncu captures
        return W.mamba2(seed, device, num_requests=16)
    raise SystemExit(f"unknown config {name}")


def relayout(wl, layout: str):
    """The same KV in another memory layout (NHD source pools; data
    movement with torch only, before any timing)."""
    import dataclasses
    from paged_kv_cache_kvcs_gb300 import workloads as W
    if layout == "nhd":
        return wl
    caches = []
    for c in wl.caches:
        if layout == "misaligned":   # the same pools starting 8 bytes past a 16-byte boundary
            buf = torch.empty(c.pool.numel() + 8, dtype=torch.uint8, device=c.pool.device)
            pool = buf[8:]
            pool.copy_(c.pool)
            caches.append(dataclasses.replace(c, pool=pool))
            c.pool = None
            continue
        assert c.layout == W.LAYOUT_NHD
        bs, H, hb, nb = wl.block_size, c.num_heads, c.head_bytes, c.num_blocks
        page = bs * H * hb
        v = c.pool.view(2, nb, bs, H, hb)
        if layout in ("misaligned_hnd", "misaligned_hnd_sub4", "misaligned_xsplit"):
            # HND (plain or in 4-slot kernel sub-blocks) or x-split pools
            # starting 8 bytes past a 16-byte boundary
            buf = torch.empty(c.pool.numel() + 8, dtype=torch.uint8, device=c.pool.device)
            pool = buf[8:]
            if layout == "misaligned_hnd":
                pool.copy_(v.permute(0, 1, 3, 2, 4).reshape(-1))
                caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_HND))
            elif layout == "misaligned_hnd_sub4":
                pool.copy_(v.view(2, nb, bs // 4, 4, H, hb).permute(0, 1, 2, 4, 3, 5).reshape(-1))
                caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_HND,
                                                  kernel_block_size=4))
            else:
                pool.copy_(v.view(2, nb, bs, H, hb // 16, 16).permute(0, 1, 3, 4, 2, 5).reshape(-1))
                caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_XSPLIT))
            c.pool = None
            continue
        if layout == "hnd":
            pool = v.permute(0, 1, 3, 2, 4).contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_HND))
        elif layout == "hnd_sub4":
            pool = v.view(2, nb, bs // 4, 4, H, hb).permute(0, 1, 2, 4, 3, 5).contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_HND,
                                              kernel_block_size=4))
        elif layout == "interleaved":   # [num_blocks, 2, page]
            pool = v.view(2, nb, page).transpose(0, 1).contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=pool, half_stride=page,
                                              block_stride=2 * page))
        elif layout == "separate_kv":
            k, vv = v[0].contiguous().view(-1), v[1].contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=k, v_pool=vv))
        elif layout == "xsplit":
            pool = v.view(2, nb, bs, H, hb // 16, 16).permute(0, 1, 3, 4, 2, 5).contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=pool, layout=W.LAYOUT_XSPLIT))
        else:
            raise SystemExit(f"unknown layout {layout}")
        c.pool = None               # free the NHD copy
    torch.cuda.empty_cache()
    return type(wl)(wl.name, wl.block_size, caches, wl.pos_offsets, wl.first_position,
                    wl.num_tokens, wl.block_ids, {**wl.info, "relayout": layout})


def kv_bytes(wl) -> int:
    """Algorithmic KV bytes one step reads: valid tokens of every position
    times the bytes a token occupies across all caches (for Mamba states:
    the state pages of the requests' block position 0)."""
    if wl.caches and wl.caches[0].layout == 4:
        state = sum(c.num_heads * c.head_bytes for c in wl.caches)
        po = wl.pos_offsets.cpu().tolist()
        fp = wl.first_position.cpu().tolist()
        return state * sum(1 for r in range(len(fp)) if fp[r] == 0 and po[r + 1] > po[r])
    per_token = sum((1 if c.layout == 2 else 2) * c.num_heads * c.head_bytes
                    for c in wl.caches)
    po = wl.pos_offsets.cpu().tolist()
    fp = wl.first_position.cpu().tolist()
    nt = wl.num_tokens.cpu().tolist()
    bs = wl.block_size
    tokens = 0
    for r in range(len(fp)):
        lo = fp[r] * bs
        hi = (fp[r] + po[r + 1] - po[r]) * bs
        tokens += max(0, min(hi, nt[r]) - lo)
    return tokens * per_token


def describe(wl, name) -> dict:
    i = wl.info
    return {"workload": f"{name}_paged_kv_checksum", "layers": i.get("layers"),
            "kv_heads": i.get("heads"), "head_bytes": i.get("head_bytes"),
            "block_size": wl.block_size,
            "layout": ["NHD", "HND", "LATENT", "XSPLIT", "STATE"][i.get("layout", 0)],
            "kv_recipe": i.get("kind"), "requests": wl.num_requests,
            "positions": wl.num_positions, "kv_bytes": kv_bytes(wl),
            "seed": i.get("seed"),
            "l2": ("KV working set far above the 129 MB L2; no flush between steps"
                   if kv_bytes(wl) > (1 << 30) else
                   "KV working set within a few L2 sizes; steps run back to back "
                   "(a latency case, not a bandwidth figure)")}


def arm_config(wl, args, ws) -> dict:
    """The ``config`` object of a line: the workload and how it is run (the
    same keys in both arms)."""
    return {**describe(wl, args.config), "parallelism": f"replicas{ws}",
            "memory_layout": args.layout, "columns": max(1, args.columns),
            "verify": bool(args.verify),
            "work_share": work_share(wl, args)}


def work_share(wl, args) -> str:
    """How the bulk kernel's units are shared out among its CTAs (planned
    for this GPU, or for a GB300's 152 SMs where no GPU is visible: the
    reference arm describes the same run on the host)."""
    if args.static:
        return "fixed"
    import paged_kv_cache_kvcs_gb300 as kvcs
    sms = (torch.cuda.get_device_properties(0).multi_processor_count
           if torch.cuda.is_available() else 152)
    plan = kvcs.plan_for(wl.caches, wl.block_size, wl.num_positions, num_sms=sms,
                         num_requests=wl.num_requests)
    if plan["kernel"] == 1:
        return "fixed (no bulk-copy launch: the direct-load kernel's warps own fixed ranges)"
    return ("dynamic (workspace)" if plan["dynamic"]
            else "fixed (workspace given; call below the dynamic threshold)")


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = Path(os.environ.get("TMPDIR", "/tmp")) / f"kvcs_clocks_{os.getpid()}.csv"
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in self.path.read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, parts))
            except (ValueError, IndexError):
                continue
        try:
            self.path.unlink()
        except OSError:
            pass
        inside = [p for ts, p in rows if t0 - 0.15 <= ts <= t1 + 0.15]
        if not inside and rows:  # too short a region: nearest samples
            inside = [p for ts, p in sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:2]]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in inside if num(p[2]) is not None]
        mx = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in inside for k in range(4)
                          if p[6 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((num(p[4]) or 0.0) for p in inside) if inside else None}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peak():
    f = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(f.read_text())
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources that make each profiled kernel: the host side that plans and
# launches it, the shared device code and the kernel's own file.
KERNEL_SOURCES = {
    "kvcs_bulk_kernel": ["kvcs.cu", "kvcs_common.cuh", "kvcs_ptx.cuh", "kvcs_bulk.cuh"],
    "kvcs_write_kernel": ["kvcs.cu", "kvcs_common.cuh", "kvcs_ptx.cuh", "kvcs_write.cuh"],
    "kvcs_direct_kernel": ["kvcs.cu", "kvcs_common.cuh", "kvcs_ptx.cuh", "kvcs_direct.cuh"],
    "kvcs_slots_kernel": ["kvcs.cu", "kvcs_common.cuh", "kvcs_ptx.cuh", "kvcs_direct.cuh",
                          "kvcs_slots.cuh"],
}


def source_code(text: str) -> str:
    """C/C++ source without its comments and blank lines (so that a comment
    edit does not count as a kernel change)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str = "kvcs_bulk_kernel", read=None) -> str:
    """SHA-256 prefix of the code (comments stripped) of the sources that
    make ``kernel``; ``read(path)`` returns a file's text (default: the
    working tree)."""
    read = read or (lambda rel: (ROOT / rel).read_text())
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        h.update(source_code(read(f"paged_kv_cache_kvcs_gb300/csrc/{name}")).encode())
    h.update(source_code(read("include/kvcs.h")).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, units_per_launch: int, kernel: str = "kvcs_bulk_kernel"):
    """DRAM bytes per launch from the committed ncu summary of this workload's
    kernel, scaled to this launch by units processed; None when the summary
    is missing or was taken on different kernel sources."""
    f = ROOT / "profiles" / f"{kernel}_{workload}.md"
    if not f.exists():
        return None
    text = f.read_text()
    m_src = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_unit:\s*([0-9.eE+]+)", text)
    if not (m_src and m_b) or m_src.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_b.group(1)) * units_per_launch


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def _reduce(x: float, ws: int, op: str) -> float:
    """Reduce one number over the ranks (NCCL on GPUs, gloo on CPUs)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def all_max(x: float, ws: int) -> float:
    return _reduce(x, ws, "max")


def all_sum(x: float, ws: int) -> float:
    return _reduce(x, ws, "sum")


def job_throughput(local_bytes: float, local_seconds: float, ws: int) -> float:
    """Whole-job GB/s of replicas: every rank's bytes over the slowest rank's
    time."""
    return all_sum(local_bytes, ws) / all_max(local_seconds, ws) / 1e9


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_inputs(wl, n: int, seed: int):
    """Host inputs of the oracle for ``n`` random block positions of the
    workload (only the pages they read): (caches, requests, KV bytes they
    hold, number of positions, the positions)."""
    import numpy as np
    from oracle.kvcs_oracle import OracleCache, OracleRequests
    from paged_kv_cache_kvcs_gb300 import workloads as W

    rng = np.random.default_rng(seed)
    P = wl.num_positions
    po = wl.pos_offsets.cpu()
    pos = torch.as_tensor(np.sort(rng.choice(P, size=min(n, P), replace=False)))
    req = torch.searchsorted(po, pos, right=True) - 1
    q = wl.first_position.cpu()[req] + (pos - po[req])
    nt = wl.num_tokens.cpu()[req]
    ids = wl.block_ids.cpu()[pos].to(torch.int64)
    caches = []
    state = bool(wl.caches) and wl.caches[0].layout == 4
    for c in wl.caches:
        pages = W.gather_pages(c, wl.block_size, ids).cpu().numpy()
        caches.append(OracleCache(pages.reshape(-1), len(pos), c.layout, c.layer,
                                  c.head_offset, c.num_heads, c.head_bytes,
                                  c.piece_bytes or 8, c.kernel_block_size))
    reqs = OracleRequests(list(range(len(pos) + 1)), q.tolist(), nt.tolist(),
                          list(range(len(pos))))
    if state:
        per_state = sum(c.num_heads * c.head_bytes for c in wl.caches)
        return caches, reqs, per_state * int((q == 0).sum()), len(pos), pos.numpy()
    per_token = sum((1 if c.layout == 2 else 2) * c.num_heads * c.head_bytes
                    for c in wl.caches)
    bs = wl.block_size
    valid = sum(max(0, min(bs, int(t) - int(qq) * bs)) for qq, t in zip(q, nt))
    return caches, reqs, valid * per_token, len(pos), pos.numpy()


def oracle_run(wl, n: int, threads: int, seed: int):
    """One timed oracle run over ``n`` random positions: (seconds, KV bytes,
    positions)."""
    from oracle import c_oracle
    caches, reqs, nbytes, npos, _ = _oracle_inputs(wl, n, seed)
    t0 = time.perf_counter()
    c_oracle.block_checksums(caches, wl.block_size, reqs, num_threads=threads)
    return time.perf_counter() - t0, nbytes, npos


def oracle_timed(wl, seconds: float, threads: int, seed: int) -> dict:
    """About ``seconds`` of oracle work on one sample of the workload (the
    sample is repeated when the whole workload takes less).  Returns GB/s,
    blocks/s, a description, and the sampled positions with the oracle's
    values there (for checking the GPU's output)."""
    from oracle import c_oracle
    n = oracle_calibrate(wl, seconds, threads, seed)
    caches, reqs, nbytes, npos, pos = _oracle_inputs(wl, n, seed + 7)
    spent, runs = 0.0, 0
    vals = None
    while runs == 0 or (spent < 0.8 * seconds and runs < 100):
        t0 = time.perf_counter()
        vals, _ = c_oracle.block_checksums(caches, wl.block_size, reqs, num_threads=threads)
        spent += time.perf_counter() - t0
        runs += 1
    desc = (f"{npos} random block positions of the workload ({nbytes / 1e9:.2f} GB "
            f"of KV), {runs} oracle run(s) totalling {spent:.1f} s on {threads} threads")
    return {"gbs": nbytes * runs / spent / 1e9, "bps": npos * runs / spent, "desc": desc,
            "positions": pos, "values": vals}


def oracle_calibrate(wl, seconds: float, threads: int, seed: int) -> int:
    """Positions whose oracle run takes about ``seconds``."""
    n = 8
    while True:
        dt, _, npos = oracle_run(wl, n, threads, seed)
        if dt >= 0.5 * seconds or npos >= wl.num_positions:
            return max(1, min(wl.num_positions, int(round(n * seconds / max(dt, 1e-4)))))
        n = min(wl.num_positions, max(2 * n, int(n * 0.6 * seconds / max(dt, 1e-4))))


def python_oracle_tiny(seed: int) -> dict:
    """The pure-Python oracle over the whole tiny workload (2 layers, 2 heads,
    one request of 100 tokens), timed on one host thread."""
    from oracle import kvcs_oracle
    from oracle.kvcs_oracle import OracleCache, OracleRequests
    from paged_kv_cache_kvcs_gb300 import workloads as W
    wl = W.tiny(seed, "cpu")
    caches = [OracleCache(c.pool.numpy(), c.num_blocks, c.layout, c.layer, c.head_offset,
                          c.num_heads, c.head_bytes) for c in wl.caches]
    reqs = OracleRequests(wl.pos_offsets.tolist(), wl.first_position.tolist(),
                          wl.num_tokens.tolist(), wl.block_ids.tolist())
    runs, spent = 0, 0.0
    while runs == 0 or (spent < 1.0 and runs < 20):
        t0 = time.perf_counter()
        kvcs_oracle.block_checksums(caches, wl.block_size, reqs)
        spent += time.perf_counter() - t0
        runs += 1
    nbytes = kv_bytes(wl)
    return {"value": round(nbytes * runs / spent / 1e9, 6), "unit": "GB/s", "cores": 1,
            "kind": "oracle (pure Python, exact ints)",
            "blocks_per_s": round(wl.num_positions * runs / spent, 2),
            "sample": f"the whole tiny workload ({nbytes} B of KV, {wl.num_positions} "
                      f"positions), {runs} run(s) totalling {spent:.2f} s"}


def parity_check(got, positions, expected) -> dict:
    """The timed run's output at the oracle's sampled positions: how many
    positions were compared and how many differ (bit for bit)."""
    import numpy as np
    g = np.asarray(got).view(np.uint64)
    e = np.asarray(expected, dtype=np.uint64)
    bad = int(np.count_nonzero(g[positions] != e))
    return {"positions": int(len(positions)), "mismatches": bad,
            "against": "C oracle at the cpu_baseline sample's positions"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, ws, rank):
    """The CPU oracle, as it stands, on the machine's host cores."""
    if rank != 0:
        return
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    from oracle import c_oracle
    wl = make_workload(args.config, args.seed, dev)
    cores = host_cores()
    # about 90 s of oracle work over all steps (at most 1.5 s a step), on one
    # sample of positions gathered to the host once
    per_step = min(1.5, max(0.005, 90.0 / (args.warmup + args.steps)))
    n = oracle_calibrate(wl, per_step, cores, args.seed)
    caches, reqs, nbytes, npos, _ = _oracle_inputs(wl, n, args.seed + 1)
    times = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        c_oracle.block_checksums(caches, wl.block_size, reqs, num_threads=cores)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append((nbytes / dt / 1e9, npos / dt))
    sample = (f"each step: the same {npos} random block positions of the workload "
              f"({nbytes / 1e9:.3f} GB of KV), scalar C oracle on {cores} threads")
    value = statistics.mean(t[0] for t in times)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3),
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u64", "data": "synthetic",
            "blocks_per_s": round(statistics.mean(t[1] for t in times), 3),
            "config": arm_config(wl, args, ws),
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_write(args, ws, rank, local):
    """The KV write fused with the checksum (kvcs_write_kv): a prefill chunk
    of new tokens written into every layer's paged pool in one call, each
    token's checksum share added to its block's running word.  Compared with
    the same write without the running words, and with writing and then
    checksumming the written blocks in a separate pass."""
    import paged_kv_cache_kvcs_gb300 as kvcs
    from paged_kv_cache_kvcs_gb300 import workloads as W
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # decode: one new token per request; "_layer": one layer per call, as a
    # forward pass writes it
    decode = args.config.startswith("llama3_8b_write_decode")
    one_layer = args.config == "llama3_8b_write_decode_layer"
    lay = {"nhd": (W.LAYOUT_NHD, 0), "hnd": (W.LAYOUT_HND, 0), "hnd_sub4": (W.LAYOUT_HND, 4),
           "xsplit": (W.LAYOUT_XSPLIT, 0)}.get(args.layout)
    if lay is None:
        raise SystemExit(f"the write bench has no layout {args.layout}")
    wb = W.llama3_8b_write(args.seed + rank, dev, kind="decode" if decode else "prefill",
                           num_requests=8 if args.config == "llama3_8b_write_small" else None,
                           layout=lay[0], kernel_block_size=lay[1],
                           layers=1 if one_layer else 32)
    caches, keys, vals, slots, pos = wb.caches, wb.keys, wb.values, wb.slot_mapping, wb.positions
    bs, nb, layers = wb.block_size, wb.num_blocks, len(wb.caches)
    heads, hb = wb.info["heads"], wb.info["head_bytes"]
    R = wb.info["requests"]
    n = slots.numel()
    L = n // R
    po, fp, nt, bids = wb.pos_offsets, wb.first_position, wb.num_tokens, wb.block_ids
    npos = int(bids.numel())
    sums = torch.zeros(nb, dtype=torch.int64, device=dev)
    # the written blocks as checksum positions (for the unfused comparison)
    ck = kvcs.Checksummer(caches, bs, po, fp, nt, bids, npos)
    out = torch.empty(npos, dtype=torch.int64, device=dev)
    stream = torch.cuda.Stream(dev)
    raw = stream.cuda_stream

    # the decode step's data fits in L2: flush it before every timed step,
    # outside the events, by reading a 256 MB buffer (a read leaves no dirty
    # lines whose write-back would land inside the timed step)
    scrub = torch.ones(32 << 20, dtype=torch.int64, device=dev) if decode else None
    scrub_out = torch.empty((), dtype=torch.int64, device=dev)

    def timed(fn, k):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fn()
            if scrub is None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(k):
                    fn()
                e1.record(stream)
            else:
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(k)]
                for a, b in ev:
                    torch.sum(scrub, dim=0, out=scrub_out)
                    a.record(stream)
                    fn()
                    b.record(stream)
        torch.cuda.synchronize(dev)
        if scrub is None:
            return e0.elapsed_time(e1) / 1e3 / k
        return sum(a.elapsed_time(b) for a, b in ev) / 1e3 / k

    # prepared calls, as an engine with fixed buffers makes them
    fused_w = kvcs.KVWriter(caches, bs, keys, vals, slots, pos, block_sums=sums)
    plain_w = kvcs.KVWriter(caches, bs, keys, vals, slots, pos)
    fused = lambda: fused_w(raw)
    plain = lambda: plain_w(raw)

    def unfused():
        plain()
        ck(out, None, raw)

    launches0 = kvcs.launch_count()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    t_wall0 = time.time()
    t_fused = timed(fused, args.steps)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    launches = (kvcs.launch_count() - launches0) // (args.steps + max(3, args.warmup))
    t_plain = timed(plain, args.steps)
    t_unfused = timed(unfused, args.steps)
    # the same fused call replayed from a CUDA graph, as a serving engine
    # replays its captured step: no host work per call
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fused_w(raw)
    t_graph = timed(graph.replay, args.steps)
    moved = 2 * n * layers * 2 * heads * hb          # bytes read + written
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    achieved = moved / t_fused / 1e9
    line = {"metric": "KV write fused with the block checksum, GB/s of bytes read + written",
            "value": round(moved / t_fused / 1e9, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_fused * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u64", "data": "synthetic",
            "config": {"workload": ("llama3_8b_decode_write_one_layer" if one_layer else
                                    "llama3_8b_decode_write" if decode
                                    else "llama3_8b_prefill_write"), "layers": layers,
                       "kv_heads": heads, "head_bytes": hb, "block_size": bs,
                       "requests": R, "new_tokens_per_request": L,
                       "bytes_moved_per_step": moved, "memory_layout": args.layout,
                       "l2": "L2 flushed (256 MB read) before every timed step" if decode
                       else "new K/V and written pages far above the 129 MB L2; no flush"},
            "gpu_launches_per_step": launches,
            "gpu_launches": launches * args.steps,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": None if decode else profiled_traffic(
                             "llama3_8b_write", n, kernel="kvcs_write_kernel"),
                         "kernel": "kvcs_write_kernel", "launch_ms": round(t_fused * 1e3, 4)},
            "clocks": clocks,
            "graph_ms_per_step": round(t_graph * 1e3, 4),
            "graph_gbs": round(moved / t_graph / 1e9, 2),
            "write_only_ms": round(t_plain * 1e3, 4),
            "write_then_checksum_ms": round(t_unfused * 1e3, 4),
            "fused_vs_write_only": round(t_plain / t_fused, 4),
            "fused_vs_write_then_checksum": round(t_unfused / t_fused, 4)}
    if one_layer:
        line["per_layer_calls"] = per_layer_calls(args, dev, stream, lay, rank, scrub, scrub_out)
    if ws == 1 and not args.no_cpu_baseline:
        # the oracle computing the same block words from the written pages
        cores = host_cores()
        ot = oracle_timed(wb.checksum_workload(), args.cpu_seconds, cores, args.seed)
        line["cpu_baseline"] = {"value": round(ot["gbs"], 3),
                                "unit": "GB/s of written KV checksummed",
                                "cores": cores, "kind": "oracle",
                                "blocks_per_s": round(ot["bps"], 2), "sample": ot["desc"]}
        # the timed call once more on zeroed running words (every timed step
        # added its terms again), read at the sampled blocks
        with torch.cuda.stream(stream):
            sums.zero_()
            fused()
        torch.cuda.synchronize(dev)
        words = sums[bids.long()].cpu().numpy()
        line["parity"] = parity_check(words, ot["positions"], ot["values"])
    print(json.dumps(line), flush=True)


def per_layer_calls(args, dev, stream, lay, rank, scrub, scrub_out) -> dict:
    """A decode forward pass writes its layers one call at a time.  Here 32
    one-layer calls (each its own pool and new rows) run back to back after
    one L2 flush, timed per call; beside them the isolated event pattern of
    the one-layer line with a one-element fill kernel in place of the call,
    the floor that pattern puts under any kernel."""
    import paged_kv_cache_kvcs_gb300 as kvcs
    from paged_kv_cache_kvcs_gb300 import workloads as W
    wb = W.llama3_8b_write(args.seed + rank + 1, dev, kind="decode", layout=lay[0],
                           kernel_block_size=lay[1], layers=32)
    sums = torch.zeros(wb.num_blocks, dtype=torch.int64, device=dev)
    writers = [kvcs.KVWriter([c], wb.block_size, [k], [v], wb.slot_mapping, wb.positions,
                             block_sums=sums)
               for c, k, v in zip(wb.caches, wb.keys, wb.values)]
    raw = stream.cuda_stream
    tiny = torch.zeros(1, dtype=torch.int64, device=dev)
    k = max(5, args.steps)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for w in writers:
                w(raw)
            tiny.fill_(1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(k)]
        for a, b in ev:
            torch.sum(scrub, dim=0, out=scrub_out)
            a.record(stream)
            for w in writers:
                w(raw)
            b.record(stream)
        fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(k)]
        for a, b in fl:
            torch.sum(scrub, dim=0, out=scrub_out)
            a.record(stream)
            tiny.fill_(1)
            b.record(stream)
    torch.cuda.synchronize(dev)
    t_pass = sum(a.elapsed_time(b) for a, b in ev) / k / 1e3
    t_floor = sum(a.elapsed_time(b) for a, b in fl) / k / 1e3
    moved = 2 * wb.slot_mapping.numel() * 2 * wb.info["heads"] * wb.info["head_bytes"]
    return {"calls": len(writers), "us_per_call": round(t_pass / len(writers) * 1e6, 3),
            "gbs_per_call": round(moved / (t_pass / len(writers)) / 1e9, 2),
            "pass_us": round(t_pass * 1e6, 2),
            "isolated_event_floor_us": round(t_floor * 1e6, 3),
            "what": "32 one-layer calls back to back after one L2 flush; floor: the one-layer "
                    "line's event pattern around a one-element fill kernel"}


def time_checksums(wl, args, dev, stream, ws, rank, steps, warmup, clocks=True) -> dict:
    """Warm-up, then ``steps`` timed calls over the whole workload, each
    bracketed by CUDA events on the launching stream (after a barrier and a
    synchronize).  The output buffer keeps the last timed call's result."""
    import paged_kv_cache_kvcs_gb300 as kvcs
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    plan = kvcs.plan_for(wl.caches, wl.block_size, wl.num_positions,
                         num_requests=wl.num_requests)
    raw_stream = stream.cuda_stream
    ncols = max(1, args.columns)
    values = None
    # a workspace lets the bulk kernel balance its work dynamically (the
    # default); --static keeps every CTA's share fixed
    wspace = None if args.static else torch.zeros(kvcs.KVCS_WORKSPACE_WORDS,
                                                   dtype=torch.int64, device=dev)
    if args.columns > 1 or args.verify:
        # the replica-key path: one column per key, plus (--verify) the
        # tagged row sums compared with stored values in the same call
        values = torch.empty((wl.num_positions, ncols), dtype=torch.int64, device=dev)
        extras = {}
        if args.verify:
            n = wl.num_positions
            g = torch.Generator(device=dev).manual_seed(args.seed)
            hashes = torch.randint(0, 256, (n, 32), dtype=torch.uint8, device=dev, generator=g)
            tags = kvcs.block_checksum_tags(hashes, 0x5EED)
            stored = torch.empty(n, dtype=torch.int64, device=dev)
            kvcs.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                                 wl.num_tokens, wl.block_ids, ncols, values=values,
                                 row_sums=stored, tags=tags, total_positions=n)
            extras = dict(tags=tags, expected=stored,
                          mismatch=torch.empty(n, dtype=torch.uint8, device=dev),
                          mismatch_count=torch.zeros(1, dtype=torch.int32, device=dev))
        n_pos = wl.num_positions       # read once: the property syncs the device

        def step():
            kvcs.group_checksums(wl.caches, wl.block_size, wl.pos_offsets,
                                 wl.first_position, wl.num_tokens, wl.block_ids, ncols,
                                 values=values, status=status, stream=raw_stream,
                                 total_positions=n_pos, workspace=wspace, **extras)
        ck = None
    else:
        ck = kvcs.workload_checksummer(wl, workspace=wspace)

        def step():
            ck(out, status, raw_stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise SystemExit(f"status {int(status.item())} during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if (clocks and rank == 0) else None
    barrier(ws)
    torch.cuda.synchronize(dev)
    launches0 = kvcs.launch_count()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for k in range(steps):
            starts[k].record(stream)
            step()
            ends[k].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(ws)
    launches = kvcs.launch_count() - launches0
    clk = sampler.stop(t_wall0, t_wall1) if sampler else None
    if int(status.item()) != 0:
        raise SystemExit(f"status {int(status.item())} during the timed steps")
    per = [a.elapsed_time(b) / 1e3 for a, b in zip(starts, ends)]
    total_s = all_max(starts[0].elapsed_time(ends[-1]) / 1e3, ws)
    if values is not None:
        # a position's checksum is its row of column partials summed mod 2^64
        import numpy as np
        result = values.cpu().numpy().view(np.uint64).sum(axis=1, dtype=np.uint64)
    else:
        result = out.cpu().numpy()
    return {"state": bool(wl.caches) and wl.caches[0].layout == 4, "ws": wspace,
            "total_s": total_s, "launch_s": statistics.mean(per), "launches": int(launches),
            "clocks": clk, "plan": plan, "nbytes": kv_bytes(wl), "ck": ck, "out": out,
            "status": status, "result": result}


def request_sweep(wl, stream, out, status, ws=None) -> list:
    """The first 1, 2, 4, ... requests of the workload alone: GB/s per call
    timed back to back, and the same call replayed from a CUDA graph."""
    import paged_kv_cache_kvcs_gb300 as kvcs
    raw_stream = stream.cuda_stream
    sweep = []
    n = 1
    while n <= wl.num_requests:
        sub = type(wl)(wl.name, wl.block_size, wl.caches, wl.pos_offsets[:n + 1],
                       wl.first_position[:n], wl.num_tokens[:n],
                       wl.block_ids[:int(wl.pos_offsets[n])], wl.info)
        sck = kvcs.workload_checksummer(sub, workspace=ws)
        sb = kv_bytes(sub)
        k = max(10, min(500, int(2e10 / max(sb, 1))))
        with torch.cuda.stream(stream):
            for _ in range(5):
                sck(out, status, raw_stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(k):
                sck(out, status, raw_stream)
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / k
        # the same call captured in a CUDA graph (no host work per step)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            sck(out, status, raw_stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                graph.replay()
            e0.record(stream)
            for _ in range(k):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        tg = e0.elapsed_time(e1) / 1e3 / k
        sp = kvcs.plan_for(sub.caches, sub.block_size, sub.num_positions)
        sweep.append({"requests": n, "kv_bytes": sb, "ms": round(t * 1e3, 4),
                      "gbs": round(sb / t / 1e9, 1), "graph_ms": round(tg * 1e3, 4),
                      "graph_gbs": round(sb / tg / 1e9, 1), "split": sp["split"]})
        n *= 2
    if int(status.item()) != 0:
        raise SystemExit(f"status {int(status.item())} during the sweep")
    return sweep


def direct_kernel_name(r) -> str:
    """The kernel of a call the bulk kernel does not take: the direct-load
    kernel for KV caches, the state-row kernel for Mamba states."""
    return "kvcs_state_kernel" if r["state"] else "kvcs_direct_kernel"


def roofline_of(r, workload: str) -> dict:
    """The dominant kernel against the measured copy peak; ``workload`` names
    the committed ncu summary that gives its DRAM traffic."""
    peak, peak_kind = measured_peak()
    achieved = r["nbytes"] / r["launch_s"] / 1e9
    plan = r["plan"]
    kernel = (direct_kernel_name(r) if plan["kernel"] == 1 else
              "kvcs_slots_kernel" if plan["kernel"] == 3 else "kvcs_bulk_kernel")
    traffic = (profiled_traffic(workload, plan["units"], kernel=kernel)
               if kernel in KERNEL_SOURCES else None)
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "kernel": kernel,
            "launch_ms": round(r["launch_s"] * 1e3, 4)}


def cpu_leg(wl, r, seconds: float, seed: int) -> tuple[dict, dict]:
    """The oracle on all host cores over a sample of the workload, and the
    timed run's output checked against it at the sampled positions."""
    cores = host_cores()
    ot = oracle_timed(wl, seconds, cores, seed)
    base = {"value": round(ot["gbs"], 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "blocks_per_s": round(ot["bps"], 2), "sample": ot["desc"]}
    return base, parity_check(r["result"], ot["positions"], ot["values"])


def oracle_one_thread(wl, seconds: float, seed: int) -> dict:
    """The C oracle on one host thread over a sample of the workload."""
    ot = oracle_timed(wl, seconds, 1, seed + 11)
    return {"value": round(ot["gbs"], 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "blocks_per_s": round(ot["bps"], 2), "sample": ot["desc"]}


def other_configs(args, dev, stream) -> dict:
    """The DeepSeek-V3-shaped MLA and Llama-3-70B-shaped fp8 workloads, each
    timed on its own (the previous one freed first), with the oracle on a
    sample and the 70B request-count sweep."""
    res = {}
    for name in ("mla", "llama3_70b"):
        torch.cuda.empty_cache()
        wl = make_workload(name, args.seed, dev)
        r = time_checksums(wl, args, dev, stream, 1, 0, args.steps, args.warmup)
        entry = {"workload": describe(wl, name),
                 "value": round(r["nbytes"] * args.steps / r["total_s"] / 1e9, 2),
                 "unit": "GB/s",
                 "ms_per_step": round(r["total_s"] / args.steps * 1e3, 4),
                 "blocks_per_s": round(wl.num_positions * args.steps / r["total_s"], 1),
                 "gpu_launches": r["launches"],
                 "plan": {k: r["plan"][k] for k in ("kernel", "split", "launches", "memsets",
                                                    "grid", "stage_bytes", "units")},
                 "roofline": roofline_of(r, name), "clocks": r["clocks"]}
        if name == "llama3_70b":
            entry["sweep"] = request_sweep(wl, stream, r["out"], r["status"], r["ws"])
        if not args.no_cpu_baseline:
            entry["cpu_baseline"], entry["parity"] = cpu_leg(wl, r, args.other_cpu_seconds,
                                                             args.seed)
            entry["cpu_baseline"]["one_thread"] = oracle_one_thread(
                wl, args.other_cpu_seconds / 2, args.seed)
        res[name] = entry
        del wl, r
    torch.cuda.empty_cache()
    return res


def run_ours(args, ws, rank, local):
    import paged_kv_cache_kvcs_gb300 as kvcs

    kvcs.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = make_workload(args.config, args.seed + rank, dev)
    if args.layout != "nhd":
        wl = relayout(wl, args.layout)
    if args.columns > 1:
        for i, c in enumerate(wl.caches):
            c.column = i % args.columns
    stream = torch.cuda.Stream(dev)
    r = time_checksums(wl, args, dev, stream, ws, rank, args.steps, args.warmup)
    total_s = r["total_s"]
    job_bytes = all_sum(r["nbytes"] * args.steps, ws)
    job_blocks = all_sum(wl.num_positions * args.steps, ws)
    value = job_bytes / total_s / 1e9

    sweep = request_sweep(wl, stream, r["out"], r["status"], r["ws"]) if args.sweep else None

    # ---- end to end: host buffers through the public API ----
    e2e = None
    if not args.no_e2e and r["ck"] is not None:
        e2e = run_e2e(args, wl, dev, stream, ws, r["ck"], r["ws"])

    if rank != 0:
        return
    plan = r["plan"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u64", "data": "synthetic",
        "blocks_per_s": round(job_blocks / total_s, 1),
        "hbm_frac_of_nominal_8tbs": round(value / ws / NOMINAL_HBM_GBS, 4),
        "config": arm_config(wl, args, ws),
        "plan": {k: plan[k] for k in ("kernel", "split", "launches", "memsets", "grid",
                                      "threads", "smem_bytes", "stage_bytes", "units")},
        "gpu_launches": r["launches"],
        "roofline": roofline_of(r, args.config if args.layout == "nhd"
                                else f"{args.config}_{args.layout}"),
        "clocks": r["clocks"],
        "e2e": e2e,
    }
    if sweep is not None:
        line["sweep"] = sweep
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = cpu_leg(wl, r, args.cpu_seconds, args.seed)
        line["cpu_baseline"]["one_thread"] = oracle_one_thread(wl, args.other_cpu_seconds,
                                                               args.seed)
        line["cpu_baseline"]["python_tiny"] = python_oracle_tiny(args.seed)
    headline = (args.config == "llama3_8b" and args.layout == "nhd" and args.columns <= 1
                and not args.verify)
    if ws == 1 and headline and not args.no_other_configs:
        del wl, r
        line["other_configs"] = other_configs(args, dev, stream)
    print(json.dumps(line), flush=True)
    bad = [k for k, v in [("headline", line.get("parity"))] +
           [(k, v.get("parity")) for k, v in line.get("other_configs", {}).items()]
           if v and v["mismatches"]]
    if bad:
        raise SystemExit(f"GPU output differs from the oracle on: {', '.join(bad)}")


def run_e2e(args, wl, dev, stream, ws, ck, workspace=None):
    """Each step: pinned host -> device copies of every KV pool and of the
    request tables, the checksum, and a device -> host read of the checksums
    and the status word.  The layers arrive in ``--e2e-groups`` groups, as a
    layer-wise KV load delivers them: each group's checksum is added into the
    position words (KVCS_OUT_ACCUMULATE) as soon as that group has landed,
    while the next group is still on the host link."""
    import paged_kv_cache_kvcs_gb300 as kvcs
    host_pools = [torch.empty(c.pool.numel(), dtype=torch.uint8, pin_memory=True)
                  for c in wl.caches]
    for h, c in zip(host_pools, wl.caches):
        h.copy_(c.pool)
    tabs = [wl.pos_offsets, wl.first_position, wl.num_tokens, wl.block_ids]
    host_tabs = [t.cpu().pin_memory() for t in tabs]
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    host_out = torch.empty(wl.num_positions, dtype=torch.int64, pin_memory=True)
    host_status = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h2d = sum(h.numel() for h in host_pools) + sum(t.numel() * t.element_size() for t in host_tabs)
    d2h = host_out.numel() * 8 + 4
    steps = max(1, min(args.steps, args.e2e_steps))
    ngroups = max(1, min(args.e2e_groups, len(wl.caches)))
    bounds = [len(wl.caches) * g // ngroups for g in range(ngroups + 1)]
    groups = [list(range(bounds[g], bounds[g + 1])) for g in range(ngroups)]
    group_ck = [kvcs.Checksummer([wl.caches[i] for i in grp], wl.block_size, wl.pos_offsets,
                                 wl.first_position, wl.num_tokens, wl.block_ids,
                                 wl.num_positions, workspace=workspace) for grp in groups]
    copy_stream = torch.cuda.Stream(dev)
    raw = stream.cuda_stream

    def one():
        go = torch.cuda.Event()
        go.record(stream)                 # the previous step's reads are done
        copy_stream.wait_event(go)
        with torch.cuda.stream(copy_stream):
            for h, t in zip(host_tabs, tabs):
                t.copy_(h, non_blocking=True)
        status.zero_()
        for g, grp in enumerate(groups):
            with torch.cuda.stream(copy_stream):
                for i in grp:
                    wl.caches[i].pool.copy_(host_pools[i], non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(copy_stream)
            stream.wait_event(landed)
            group_ck[g](out, status, raw, accumulate=g > 0)
        host_out.copy_(out, non_blocking=True)
        host_status.copy_(status, non_blocking=True)

    with torch.cuda.stream(stream):
        one()
    torch.cuda.synchronize(dev)
    barrier(ws)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps):
            one()
        t1.record(stream)
    torch.cuda.synchronize(dev)
    if int(host_status.item()) != 0:
        raise SystemExit("status set during the end-to-end run")
    secs = all_max(t0.elapsed_time(t1) / 1e3, ws)
    total = all_sum(kv_bytes(wl) * steps, ws)
    del host_pools
    return {"value": round(total / secs / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": round(secs / steps * 1e3, 3),
            "layer_groups": ngroups,
            "what": "pinned-host KV pools + block tables -> device in layer groups, "
                    "each group checksummed (accumulating) as it lands, "
                    "checksums -> pinned host, every step"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="llama3_8b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-groups", type=int, default=8,
                    help="layer groups the end-to-end load delivers and checksums")
    ap.add_argument("--sweep", action="store_true",
                    help="also time the first 1, 2, 4, ... requests alone")
    ap.add_argument("--layout", default="nhd",
                    choices=("nhd", "hnd", "hnd_sub4", "interleaved", "separate_kv", "xsplit",
                             "misaligned", "misaligned_hnd", "misaligned_hnd_sub4",
                             "misaligned_xsplit"),
                    help="re-lay-out the (NHD) workload's pools before timing")
    ap.add_argument("--columns", type=int, default=1,
                    help="replica-key columns (caches assigned round-robin)")
    ap.add_argument("--verify", action="store_true",
                    help="time the tagged row sums and their comparison too")
    ap.add_argument("--static", action="store_true",
                    help="no workspace: every CTA's share of the work is fixed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--other-cpu-seconds", type=float, default=4.0,
                    help="oracle seconds per extra workload and for the one-thread figure")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time only the chosen workload (the default line also times "
                         "the MLA and 70B workloads and the 70B request sweep)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    ws, rank, local = dist_setup() if torch.cuda.is_available() else (1, 0, 0)
    if ws != args.gpus and rank == 0:
        print(f"note: --gpus {args.gpus} but WORLD_SIZE {ws}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        elif args.config in ("llama3_8b_write", "llama3_8b_write_small",
                             "llama3_8b_write_decode", "llama3_8b_write_decode_layer"):
            run_write(args, ws, rank, local)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
