"""Shared test plumbing: turn a seeded workload into the oracle's host inputs.

Only data movement lives here (device -> host copies, dataclass packing);
none of the checksum's arithmetic.
"""

from __future__ import annotations

import os
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

from oracle import c_oracle, kvcs_oracle  # noqa: E402
from oracle.kvcs_oracle import OracleCache, OracleRequests  # noqa: E402
from paged_kv_cache_kvcs_gb300 import workloads as W  # noqa: E402


def host_bytes(t) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8).reshape(-1)


def oracle_caches(caches) -> list[OracleCache]:
    """Host copies of the pools.  A separate V tensor is appended to the K
    bytes (data movement only), its pages then half_stride = len(K) bytes
    after the K pages."""
    out = []
    for c in caches:
        data = host_bytes(c.pool)
        half = getattr(c, "half_stride", 0)
        v_pool = getattr(c, "v_pool", None)
        if v_pool is not None:
            half = data.size
            data = np.concatenate([data, host_bytes(v_pool)])
        out.append(OracleCache(data, c.num_blocks, c.layout, c.layer, c.head_offset,
                               c.num_heads, c.head_bytes, getattr(c, "piece_bytes", 0) or 8,
                               getattr(c, "kernel_block_size", 0), half,
                               getattr(c, "block_stride", 0)))
    return out


def oracle_requests(wl) -> OracleRequests:
    return OracleRequests(wl.pos_offsets.cpu().tolist(),
                          wl.first_position.cpu().tolist(),
                          wl.num_tokens.cpu().tolist(),
                          wl.block_ids.cpu().tolist())


def oracle_inputs(wl):
    return oracle_caches(wl.caches), oracle_requests(wl)


def py_form(caches, block_size, reqs):
    out, status = kvcs_oracle.block_checksums(caches, block_size, reqs)
    return [int(v) for v in out], status


def c_form(caches, block_size, reqs, threads: int | None = None):
    out, status = c_oracle.block_checksums(
        caches, block_size, reqs,
        num_threads=threads or min(8, c_oracle.default_threads()))
    return [int(v) for v in out], status


FORMS = {"python": py_form, "c": c_form}


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def env_int(name: str, default: int) -> int:
    return int(os.environ.get(name, default))
