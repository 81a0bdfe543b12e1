"""ctypes binding to ``libkvcs.so``: argument marshalling only.

Every step of the checksum runs in the library's CUDA kernels.  There is no
fallback: if the library has not been built, loading raises.
"""

from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Sequence

LIB_PATH = Path(__file__).resolve().parent / "_build" / "libkvcs.so"

KVCS_LAYOUT_NHD = 0
KVCS_LAYOUT_HND = 1
KVCS_LAYOUT_LATENT = 2
KVCS_LAYOUT_XSPLIT = 3
KVCS_LAYOUT_STATE = 4
KVCS_MAX_KV_HEADS_PER_LAYER = 65536
KVCS_BLOCK_CHECKSUM_BYTES = 8

KVCS_OK = 0
KVCS_EINVAL = -1
KVCS_EUNSUPPORTED = -2
KVCS_ECUDA = -3
KVCS_ETOOLARGE = -4

KVCS_STATUS_BAD_BLOCK_ID = 1
KVCS_STATUS_BAD_REQUESTS = 2
KVCS_STATUS_TIMEOUT = 4

KVCS_OUT_ACCUMULATE = 1
KVCS_OUT_WORKSPACE = 2
KVCS_WORKSPACE_WORDS = 16
KVCS_NOALLOC_MAX_CACHES = 1024


class kvcs_cache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("layer", ctypes.c_int32),
                ("head_offset", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_bytes", ctypes.c_int32), ("column", ctypes.c_int32),
                ("half_stride", ctypes.c_int64), ("block_stride", ctypes.c_int64),
                ("kernel_block_size", ctypes.c_int32), ("piece_bytes", ctypes.c_int32)]


class kvcs_outputs(ctypes.Structure):
    _fields_ = [("num_columns", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("values", ctypes.c_void_p), ("row_sums", ctypes.c_void_p),
                ("tags", ctypes.c_void_p), ("expected", ctypes.c_void_p),
                ("mismatch", ctypes.c_void_p), ("mismatch_count", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p)]


class kvcs_requests(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int64),
                ("pos_offsets", ctypes.c_void_p),
                ("first_position", ctypes.c_void_p),
                ("num_tokens", ctypes.c_void_p),
                ("block_ids", ctypes.c_void_p)]


class kvcs_plan_info(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("split", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("memsets", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("dynamic", ctypes.c_int32),
                ("slot_launches", ctypes.c_int32),
                ("units", ctypes.c_int64), ("kv_bytes_max", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# Every symbol kvcs.h declares, with its ctypes signature.
SIGNATURES = {
    "kvcs_block_checksums": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(kvcs_requests), ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p]),
    "kvcs_block_checksums_noalloc": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(kvcs_requests), ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p]),
    "kvcs_group_checksums": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(kvcs_requests), ctypes.c_int64, ctypes.POINTER(kvcs_outputs),
        ctypes.c_void_p, ctypes.c_void_p]),
    "kvcs_block_checksum_tags": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
        ctypes.c_void_p, ctypes.c_void_p]),
    "kvcs_write_kv": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
        ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvcs_plan": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(kvcs_plan_info)]),
    "kvcs_plan_requests": (ctypes.c_int, [
        ctypes.POINTER(kvcs_cache), ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(kvcs_plan_info)]),
    "kvcs_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_void_p]),
    "kvcs_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "kvcs_launch_count": (ctypes.c_uint64, []),
    "kvcs_version": (ctypes.c_int32, []),
}

_lib = None


class KvcsError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} (code {code})")
        self.code = code


def load_library() -> ctypes.CDLL:
    """Load ``_build/libkvcs.so``; raise if it was not built."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load_library().kvcs_strerror(code).decode()


def launch_count() -> int:
    return int(load_library().kvcs_launch_count())


def version() -> int:
    return int(load_library().kvcs_version())


def _addr(t) -> int:
    return t if isinstance(t, int) else t.data_ptr()


def cache_array(caches: Sequence) -> ctypes.Array:
    """Pack cache descriptors.  Each item has ``pool`` (a tensor, or an int
    device address), ``num_blocks``, ``layout``, ``layer``, ``head_offset``,
    ``num_heads`` and ``head_bytes``; optionally ``column``,
    ``half_stride``, ``block_stride``, ``kernel_block_size`` and ``v_pool``
    (a separate tensor holding the V pages: the half stride is then the
    distance from ``pool`` to it)."""
    arr = (kvcs_cache * max(1, len(caches)))()
    for i, c in enumerate(caches):
        base = _addr(c.pool)
        v_pool = getattr(c, "v_pool", None)
        half_stride = getattr(c, "half_stride", 0)
        if v_pool is not None:
            half_stride = _addr(v_pool) - base
        arr[i] = kvcs_cache(base, c.num_blocks, c.layout, c.layer, c.head_offset,
                            c.num_heads, c.head_bytes, getattr(c, "column", 0),
                            half_stride, getattr(c, "block_stride", 0),
                            getattr(c, "kernel_block_size", 0),
                            getattr(c, "piece_bytes", 0))
    return arr


def kvcs_block_checksums(caches: ctypes.Array, num_caches: int, block_size: int,
                         reqs: kvcs_requests, total_positions: int, out: int,
                         status: int | None, stream: int | None) -> int:
    """The C entry point, one-to-one; raises ``KvcsError`` on a negative
    return."""
    rc = load_library().kvcs_block_checksums(
        caches, num_caches, block_size, ctypes.byref(reqs), total_positions,
        out, status or None, stream or None)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_block_checksums")
    return rc


def kvcs_block_checksums_noalloc(caches: ctypes.Array, num_caches: int, block_size: int,
                                 reqs: kvcs_requests, total_positions: int, out: int,
                                 status: int | None, stream: int | None) -> int:
    """The C entry point, one-to-one; raises ``KvcsError`` on a negative
    return."""
    rc = load_library().kvcs_block_checksums_noalloc(
        caches, num_caches, block_size, ctypes.byref(reqs), total_positions,
        out, status or None, stream or None)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_block_checksums_noalloc")
    return rc


def kvcs_plan(caches: ctypes.Array, num_caches: int, block_size: int,
              total_positions: int, num_sms: int = 0) -> dict:
    info = kvcs_plan_info()
    rc = load_library().kvcs_plan(caches, num_caches, block_size,
                                  total_positions, num_sms, ctypes.byref(info))
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_plan")
    return info.as_dict()


def kvcs_plan_requests(caches: ctypes.Array, num_caches: int, block_size: int,
                       total_positions: int, num_requests: int, num_sms: int = 0) -> dict:
    info = kvcs_plan_info()
    rc = load_library().kvcs_plan_requests(caches, num_caches, block_size, total_positions,
                                           num_requests, num_sms, ctypes.byref(info))
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_plan_requests")
    return info.as_dict()


def _current_device():
    import torch
    return torch.device("cuda", torch.cuda.current_device())


def _check_tensor(name: str, t, dtypes, min_numel: int, device) -> None:
    """``t`` is a contiguous CUDA tensor of one of ``dtypes`` on ``device``
    holding at least ``min_numel`` elements: the kernels get only its
    address, so a CPU tensor, another device's tensor or a short one must be
    refused here."""
    if not (getattr(t, "is_cuda", False) and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be a {' or '.join(map(str, dtypes))} tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call runs on {device}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs {min_numel}")


def _check_requests(pos_offsets, first_position, num_tokens, block_ids,
                    total_positions: int):
    """The request table: int64 pos_offsets [R+1], first_position [R],
    num_tokens [R] and int32 block_ids [>= total_positions], all on the
    current CUDA device.  Returns that device."""
    import torch
    for name, t in (("pos_offsets", pos_offsets), ("first_position", first_position),
                    ("num_tokens", num_tokens), ("block_ids", block_ids)):
        if not getattr(t, "is_cuda", False):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if pos_offsets.numel() < 1:
        raise ValueError("pos_offsets must hold num_requests + 1 elements")
    dev = _current_device()
    R = pos_offsets.numel() - 1
    _check_tensor("pos_offsets", pos_offsets, (torch.int64,), R + 1, dev)
    for name, t in (("first_position", first_position), ("num_tokens", num_tokens)):
        _check_tensor(name, t, (torch.int64,), R, dev)
        if t.numel() != R:
            raise ValueError(f"{name} must hold one element per request ({R})")
    if total_positions < 0:
        raise ValueError("total_positions must be >= 0")
    _check_tensor("block_ids", block_ids, (torch.int32,), total_positions, dev)
    return dev


def _check_status(status, dev) -> None:
    import torch
    if status is not None:
        _check_tensor("status", status, (torch.int32, torch.uint32), 1, dev)


WORDS = None


def _words():
    """dtypes that hold uint64 bits"""
    global WORDS
    if WORDS is None:
        import torch
        WORDS = (torch.int64, torch.uint64)
    return WORDS


def _check_pool(c, block_size: int) -> None:
    """Every page the descriptor can address lies inside its tensor, on the
    current device."""
    t = c.pool
    if isinstance(t, int):
        return
    v_pool = getattr(c, "v_pool", None)
    for x in (t, v_pool):
        if x is not None and not (x.is_cuda and x.is_contiguous()):
            raise ValueError("cache pools must be contiguous CUDA tensors")
    dev = _current_device()
    for x in (t, v_pool):
        if x is not None and x.device != dev:
            raise ValueError(f"a cache pool is on {x.device}, the call runs on {dev}")
    page = (1 if c.layout == KVCS_LAYOUT_STATE else block_size) * c.num_heads * c.head_bytes
    bstride = getattr(c, "block_stride", 0) or page
    span = (c.num_blocks - 1) * bstride + page if c.num_blocks > 0 else 0
    if c.layout in (KVCS_LAYOUT_LATENT, KVCS_LAYOUT_STATE):
        halves = [(t, 0)]
    elif v_pool is not None:
        halves = [(t, 0), (v_pool, 0)]
    else:
        hs = getattr(c, "half_stride", 0) or c.num_blocks * page
        if hs < 0:
            raise ValueError("a negative half stride needs a separate v_pool tensor")
        halves = [(t, 0), (t, hs)]
    for x, off in halves:
        if off + span > x.numel() * x.element_size():
            raise ValueError("cache pool is smaller than its declared geometry")


def block_checksums(caches: Sequence, block_size: int, pos_offsets, first_position,
                    num_tokens, block_ids, out=None, status=None, stream=None,
                    total_positions: int | None = None):
    """Torch front end of ``kvcs_block_checksums``.

    ``pos_offsets``/``first_position``/``num_tokens`` are int64 CUDA tensors,
    ``block_ids`` an int32 CUDA tensor.  Returns ``out``: an int64 CUDA tensor
    whose elements hold the uint64 checksums' bits (view it as uint64 on the
    host).  ``status``, if given, is an int32 CUDA tensor of one element into
    which ``KVCS_STATUS_*`` bits are OR-ed.
    """
    import torch
    for c in caches:
        _check_pool(c, block_size)
    if total_positions is None:
        if not getattr(pos_offsets, "is_cuda", False) or pos_offsets.numel() < 1:
            raise ValueError("pos_offsets must be a CUDA int64 tensor of num_requests + 1")
        total_positions = int(pos_offsets[-1].item())
    dev = _check_requests(pos_offsets, first_position, num_tokens, block_ids, total_positions)
    if out is None:
        out = torch.empty(max(total_positions, 0), dtype=torch.int64, device=dev)
    else:
        _check_tensor("out", out, _words(), total_positions, dev)
    _check_status(status, dev)
    reqs = kvcs_requests(pos_offsets.numel() - 1, pos_offsets.data_ptr(),
                         first_position.data_ptr(), num_tokens.data_ptr(),
                         block_ids.data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    arr = cache_array(caches)
    kvcs_block_checksums(arr, len(caches), block_size, reqs, total_positions,
                         out.data_ptr() if total_positions > 0 else None,
                         status.data_ptr() if status is not None else None, stream)
    return out


def block_checksums_noalloc(caches: Sequence, block_size: int, pos_offsets, first_position,
                            num_tokens, block_ids, out, total_positions: int, status=None,
                            stream=None):
    """Torch front end of ``kvcs_block_checksums_noalloc``: arguments as
    ``block_checksums``, except that ``out`` and ``total_positions`` are
    required, so that nothing on this path allocates device memory or
    synchronises.  Calls on one device share the library's scratch and must
    not overlap on the GPU (one stream order)."""
    import torch
    for c in caches:
        _check_pool(c, block_size)
    dev = _check_requests(pos_offsets, first_position, num_tokens, block_ids, total_positions)
    _check_tensor("out", out, _words(), total_positions, dev)
    _check_status(status, dev)
    reqs = kvcs_requests(pos_offsets.numel() - 1, pos_offsets.data_ptr(),
                         first_position.data_ptr(), num_tokens.data_ptr(),
                         block_ids.data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    arr = cache_array(caches)
    kvcs_block_checksums_noalloc(arr, len(caches), block_size, reqs, total_positions,
                                 out.data_ptr() if total_positions > 0 else None,
                                 status.data_ptr() if status is not None else None, stream)
    return out


class Checksummer:
    """A checksum call prepared once for a fixed set of caches and request
    arrays: the descriptors are checked and marshalled here, so each call
    is a single ctypes call into ``kvcs_block_checksums`` (or, with a
    ``workspace`` of ``KVCS_WORKSPACE_WORDS`` 64-bit CUDA words, into
    ``kvcs_group_checksums``, which then balances its work dynamically).

    The request tensors may be refilled in place between calls (for
    example by host-to-device copies); their addresses must not change.
    """

    def __init__(self, caches: Sequence, block_size: int, pos_offsets,
                 first_position, num_tokens, block_ids, total_positions: int,
                 workspace=None):
        for c in caches:
            _check_pool(c, block_size)
        self.device = _check_requests(pos_offsets, first_position, num_tokens, block_ids,
                                      total_positions)
        if workspace is not None:
            _check_tensor("workspace", workspace, _words(), KVCS_WORKSPACE_WORDS, self.device)
        self.workspace = workspace
        self._keep = (list(caches), pos_offsets, first_position, num_tokens, block_ids,
                      workspace)
        self.num_caches = len(caches)
        self.block_size = block_size
        self.total_positions = total_positions
        self.caches = cache_array(caches)
        self.reqs = kvcs_requests(pos_offsets.numel() - 1, pos_offsets.data_ptr(),
                                  first_position.data_ptr(), num_tokens.data_ptr(),
                                  block_ids.data_ptr())
        self._fn = load_library().kvcs_block_checksums
        self._group_fn = load_library().kvcs_group_checksums
        self._reqs_ref = ctypes.byref(self.reqs)

    def __call__(self, out, status=None, stream: int | None = None, accumulate: bool = False):
        """Enqueue one call writing ``out`` (int64/uint64 CUDA tensor of at
        least ``total_positions`` words) on ``stream`` (a raw handle);
        ``accumulate`` adds this call's checksums into ``out`` instead."""
        if out.device != self.device or out.numel() < self.total_positions or \
                out.dtype not in _words() or not out.is_contiguous():
            _check_tensor("out", out, _words(), self.total_positions, self.device)
        if status is not None and status.device != self.device:
            _check_status(status, self.device)
        import torch
        if torch.cuda.current_device() != self.device.index:
            raise ValueError(f"the call was prepared on {self.device}; make it current")
        if accumulate or self.workspace is not None:
            flags = (KVCS_OUT_ACCUMULATE if accumulate else 0) | \
                (KVCS_OUT_WORKSPACE if self.workspace is not None else 0)
            outs = kvcs_outputs(1, flags, out.data_ptr() if self.total_positions > 0 else None,
                                None, None, None, None, None,
                                _ptr(self.workspace))
            rc = self._group_fn(self.caches, self.num_caches, self.block_size, self._reqs_ref,
                                self.total_positions, ctypes.byref(outs),
                                status.data_ptr() if status is not None else None,
                                stream or None)
            if rc != KVCS_OK:
                raise KvcsError(rc, "kvcs_group_checksums")
            return out
        rc = self._fn(self.caches, self.num_caches, self.block_size, self._reqs_ref,
                      self.total_positions,
                      out.data_ptr() if self.total_positions > 0 else None,
                      status.data_ptr() if status is not None else None,
                      stream or None)
        if rc != KVCS_OK:
            raise KvcsError(rc, "kvcs_block_checksums")
        return out


def workload_checksums(wl, out=None, status=None, stream=None):
    """``block_checksums`` over a ``workloads.Workload``."""
    return block_checksums(wl.caches, wl.block_size, wl.pos_offsets,
                           wl.first_position, wl.num_tokens, wl.block_ids,
                           out=out, status=status, stream=stream,
                           total_positions=wl.num_positions)


def workload_checksummer(wl, workspace=None) -> Checksummer:
    """A prepared call over a ``workloads.Workload`` (with a workspace: the
    dynamically balanced form)."""
    return Checksummer(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                       wl.num_tokens, wl.block_ids, wl.num_positions, workspace=workspace)


def plan_for(caches: Sequence, block_size: int, total_positions: int,
             num_sms: int = 0, num_requests: int | None = None) -> dict:
    """The plan of a call (``kvcs_plan``, or ``kvcs_plan_requests`` when
    ``num_requests`` is given)."""
    if num_requests is None:
        return kvcs_plan(cache_array(caches), len(caches), block_size,
                         total_positions, num_sms)
    return kvcs_plan_requests(cache_array(caches), len(caches), block_size,
                              total_positions, num_requests, num_sms)


def selftest_wait_timeout(status, limit_ns: int, stream=None) -> None:
    """Run ``kvcs_selftest_wait_timeout`` on an int32 CUDA status tensor."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(status.device).cuda_stream
    rc = load_library().kvcs_selftest_wait_timeout(status.data_ptr(), limit_ns, stream)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_selftest_wait_timeout")


def _ptr(t):
    return t.data_ptr() if t is not None else None


def group_checksums(caches: Sequence, block_size: int, pos_offsets, first_position,
                    num_tokens, block_ids, num_columns: int, values=None,
                    row_sums=None, tags=None, expected=None, mismatch=None,
                    mismatch_count=None, status=None, stream=None,
                    total_positions: int | None = None, accumulate: bool = False,
                    workspace=None):
    """Torch front end of ``kvcs_group_checksums``.  Each cache names its
    replica-key ``column``; returns ``values`` (int64 CUDA tensor
    ``[total_positions, num_columns]`` holding uint64 bits).  ``row_sums``,
    ``tags``, ``expected`` are int64 CUDA tensors of ``total_positions``;
    ``mismatch`` a uint8 one; ``mismatch_count`` an int32 one-element one.
    ``accumulate`` adds the partials into the given ``values``.  ``workspace``
    (``KVCS_WORKSPACE_WORDS`` 64-bit CUDA words, used by this call alone)
    lets the bulk kernel balance its work dynamically."""
    import torch
    for c in caches:
        _check_pool(c, block_size)
    if total_positions is None:
        if not getattr(pos_offsets, "is_cuda", False) or pos_offsets.numel() < 1:
            raise ValueError("pos_offsets must be a CUDA int64 tensor of num_requests + 1")
        total_positions = int(pos_offsets[-1].item())
    dev = _check_requests(pos_offsets, first_position, num_tokens, block_ids, total_positions)
    if not 1 <= num_columns <= 64:
        raise ValueError("num_columns must be in [1, 64]")
    if values is None:
        if accumulate:
            raise ValueError("accumulate needs the values to add into")
        values = torch.empty((max(total_positions, 0), num_columns), dtype=torch.int64,
                             device=dev)
    else:
        _check_tensor("values", values, _words(), total_positions * num_columns, dev)
    for name, t in (("row_sums", row_sums), ("tags", tags), ("expected", expected)):
        if t is not None:
            _check_tensor(name, t, _words(), total_positions, dev)
    if mismatch is not None:
        _check_tensor("mismatch", mismatch, (torch.uint8, torch.bool), total_positions, dev)
    if mismatch_count is not None:
        _check_tensor("mismatch_count", mismatch_count, (torch.int32, torch.uint32), 1, dev)
    _check_status(status, dev)
    if workspace is not None:
        _check_tensor("workspace", workspace, _words(), KVCS_WORKSPACE_WORDS, dev)
    flags = (KVCS_OUT_ACCUMULATE if accumulate else 0) | \
        (KVCS_OUT_WORKSPACE if workspace is not None else 0)
    outs = kvcs_outputs(num_columns, flags,
                        values.data_ptr() if total_positions > 0 else None,
                        _ptr(row_sums), _ptr(tags), _ptr(expected), _ptr(mismatch),
                        _ptr(mismatch_count), _ptr(workspace))
    reqs = kvcs_requests(pos_offsets.numel() - 1, pos_offsets.data_ptr(),
                         first_position.data_ptr(), num_tokens.data_ptr(),
                         block_ids.data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    arr = cache_array(caches)
    rc = load_library().kvcs_group_checksums(arr, len(caches), block_size,
                                             ctypes.byref(reqs), total_positions,
                                             ctypes.byref(outs), _ptr(status), stream)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_group_checksums")
    return values


def block_checksum_tags(block_hashes, fingerprint: int, tags=None, stream=None):
    """Torch front end of ``kvcs_block_checksum_tags``: ``block_hashes`` is a
    uint8 CUDA tensor ``[n, hash_bytes]`` (hash_bytes >= 8); returns an int64
    tensor of ``n`` tags (uint64 bits)."""
    import torch
    if not (block_hashes.is_cuda and block_hashes.dtype == torch.uint8
            and block_hashes.dim() == 2 and block_hashes.stride(1) == 1):
        raise ValueError("block_hashes must be a CUDA uint8 [n, hash_bytes] tensor")
    n = block_hashes.shape[0]
    if tags is None:
        tags = torch.empty(n, dtype=torch.int64, device=block_hashes.device)
    if stream is None:
        stream = torch.cuda.current_stream(block_hashes.device).cuda_stream
    rc = load_library().kvcs_block_checksum_tags(
        block_hashes.data_ptr() if n else None, block_hashes.stride(0), n,
        fingerprint & ((1 << 64) - 1), tags.data_ptr() if n else None, stream)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_block_checksum_tags")
    return tags


def write_kv(caches, block_size: int, keys, values, slot_mapping, positions,
             block_sums=None, status=None, stream=None) -> None:
    """Torch front end of ``kvcs_write_kv`` over one cache or a list of
    caches: ``keys``/``values`` are CUDA tensors ``[num_tokens, heads,
    head_size]`` (any dtype; their bytes are written), one per cache, with
    ``values[k]`` None for a latent cache; ``slot_mapping`` and ``positions``
    int64 CUDA tensors; ``block_sums`` an int64 CUDA tensor of running words
    (uint64 bits) or None."""
    import torch
    if not isinstance(caches, (list, tuple)):
        caches, keys, values = [caches], [keys], [values]
    n = slot_mapping.numel()
    for c, k, v in zip(caches, keys, values):
        _check_pool(c, block_size)
        row = c.num_heads * c.head_bytes
        for name, t in (("key", k), ("value", v)):
            if t is not None and not (t.is_cuda and t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
            if t is not None and t.numel() * t.element_size() < n * row:
                raise ValueError(f"{name} is smaller than num_tokens rows")
    for name, t in (("slot_mapping", slot_mapping), ("positions", positions)):
        if not (t.is_cuda and t.dtype == torch.int64 and t.is_contiguous() and t.numel() == n):
            raise ValueError(f"{name} must be a contiguous CUDA int64 tensor of num_tokens")
    dev = _current_device()
    for name, t in (("slot_mapping", slot_mapping), ("positions", positions)):
        _check_tensor(name, t, (torch.int64,), n, dev)
    for k, v in zip(keys, values):
        for name, t in (("key", k), ("value", v)):
            if t is not None and t.device != dev:
                raise ValueError(f"a {name} tensor is on {t.device}, the call runs on {dev}")
    if block_sums is not None and block_sums.numel() < min(c.num_blocks for c in caches):
        raise ValueError("block_sums needs one word per block")
    if block_sums is not None:
        _check_tensor("block_sums", block_sums, _words(),
                      min(c.num_blocks for c in caches), dev)
    _check_status(status, dev)
    if stream is None:
        stream = torch.cuda.current_stream(slot_mapping.device).cuda_stream
    arr = cache_array(caches)
    kp = (ctypes.c_void_p * len(caches))(*[_ptr(k) for k in keys])
    vp = (ctypes.c_void_p * len(caches))(*[_ptr(v) for v in values])
    rc = load_library().kvcs_write_kv(arr, len(caches), block_size, n, kp, vp,
                                      slot_mapping.data_ptr() if n else None,
                                      positions.data_ptr() if n else None,
                                      _ptr(block_sums), _ptr(status), stream)
    if rc != KVCS_OK:
        raise KvcsError(rc, "kvcs_write_kv")


class KVWriter:
    """A ``kvcs_write_kv`` call prepared once for fixed caches and fixed
    new-token buffers (as a serving engine keeps them): the arguments are
    checked and marshalled here, so each call is a single ctypes call.  The
    buffers may be refilled in place between calls; ``num_tokens`` may be
    lowered per call (the first tokens of the buffers are written)."""

    def __init__(self, caches, block_size: int, keys, values, slot_mapping, positions,
                 block_sums=None, status=None):
        if not isinstance(caches, (list, tuple)):
            caches, keys, values = [caches], [keys], [values]
        write_kv(caches, block_size, keys, values, slot_mapping[:0], positions[:0],
                 block_sums, status)                     # argument checks only
        n = slot_mapping.numel()
        for c, k, v in zip(caches, keys, values):
            row = c.num_heads * c.head_bytes
            for t in (k, v):
                if t is not None and t.numel() * t.element_size() < n * row:
                    raise ValueError("key/value buffers are smaller than the slot mapping")
        if positions.numel() != n:
            raise ValueError("positions and slot_mapping differ in length")
        self._keep = (list(caches), list(keys), list(values), slot_mapping, positions,
                      block_sums, status)
        self.max_tokens = n
        self.num_caches = len(caches)
        self.block_size = block_size
        self.caches = cache_array(caches)
        self.kp = (ctypes.c_void_p * len(caches))(*[_ptr(k) for k in keys])
        self.vp = (ctypes.c_void_p * len(caches))(*[_ptr(v) for v in values])
        self.slots = slot_mapping.data_ptr()
        self.pos = positions.data_ptr()
        self.sums = _ptr(block_sums)
        self.status = _ptr(status)
        self._fn = load_library().kvcs_write_kv

    def __call__(self, stream: int | None = None, num_tokens: int | None = None):
        n = self.max_tokens if num_tokens is None else num_tokens
        if not 0 <= n <= self.max_tokens:
            raise ValueError("num_tokens outside the prepared buffers")
        rc = self._fn(self.caches, self.num_caches, self.block_size, n, self.kp, self.vp,
                      self.slots if n else None, self.pos if n else None, self.sums,
                      self.status, stream or None)
        if rc != KVCS_OK:
            raise KvcsError(rc, "kvcs_write_kv")
