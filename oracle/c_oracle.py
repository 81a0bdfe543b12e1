"""ctypes wrapper over the scalar C oracle (``kvcs_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Takes the same host-side description as the
pure-Python form (``OracleCache`` and ``OracleRequests``) and returns numpy
uint64 checksums plus the status word.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

import numpy as np

from . import build as _build
from .kvcs_oracle import OracleCache, OracleRequests


class _OracleCacheC(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("data_bytes", ctypes.c_int64),
                ("num_blocks", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("layer", ctypes.c_int32),
                ("head_offset", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_bytes", ctypes.c_int32), ("piece_bytes", ctypes.c_int32),
                ("kernel_block_size", ctypes.c_int32), ("half_stride", ctypes.c_int64),
                ("block_stride", ctypes.c_int64)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(_build.build()))
        f = lib.oracle_block_checksums
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.POINTER(_OracleCacheC), ctypes.c_int32,
                      ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32),
                      ctypes.c_int32]
        _lib = lib
    return _lib


def default_threads() -> int:
    """Host cores this process may use."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def block_checksums(caches: Sequence[OracleCache], block_size: int,
                    requests: OracleRequests,
                    num_threads: int = 1) -> tuple[np.ndarray, int]:
    """uint64 checksum per global position index, and the status word."""
    lib = _load()
    datas = [np.ascontiguousarray(c.data, dtype=np.uint8) for c in caches]
    arr = (_OracleCacheC * max(1, len(caches)))()
    for k, (c, d) in enumerate(zip(caches, datas)):
        arr[k] = _OracleCacheC(d.ctypes.data, d.size, c.num_blocks, c.layout, c.layer,
                               c.head_offset, c.num_heads, c.head_bytes,
                               getattr(c, "piece_bytes", 8),
                               getattr(c, "kernel_block_size", 0),
                               getattr(c, "half_stride", 0), getattr(c, "block_stride", 0))
    po = np.ascontiguousarray(requests.pos_offsets, dtype=np.int64)
    fp = np.ascontiguousarray(requests.first_position, dtype=np.int64)
    nt = np.ascontiguousarray(requests.num_tokens, dtype=np.int64)
    bi = np.ascontiguousarray(requests.block_ids, dtype=np.int32)
    total = int(po[-1]) if po.size else 0
    out = np.zeros(max(total, 1), dtype=np.uint64)
    status = ctypes.c_uint32(0)
    rc = lib.oracle_block_checksums(arr, len(caches), block_size, po.size - 1,
                                    po.ctypes.data, fp.ctypes.data,
                                    nt.ctypes.data, bi.ctypes.data,
                                    out.ctypes.data, ctypes.byref(status),
                                    num_threads)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return out[:total], int(status.value)
