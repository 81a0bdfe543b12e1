"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and its host-side validation and planning behave."""

import ctypes
import re
from pathlib import Path

import pytest

import paged_kv_cache_kvcs_gb300 as K
from paged_kv_cache_kvcs_gb300 import _binding as B

HEADER = Path(__file__).resolve().parent.parent / "include" / "kvcs.h"


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kvcs_[a-z_]+)\s*\(",
                                 text, re.M)))


def test_header_declares_the_bound_symbols():
    names = declared_functions()
    assert names == sorted(B.SIGNATURES), names


def test_library_exports_every_declared_symbol():
    lib = K.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_header_constants_match_the_binding():
    text = HEADER.read_text()
    consts = {m.group(1): int(m.group(2).rstrip("u"))
              for m in re.finditer(r"#define (KVCS_[A-Z_]+) \(?(-?[0-9]+u?)\)?", text)}
    consts.update({m.group(1): int(m.group(2))
                   for m in re.finditer(r"(KVCS_LAYOUT_[A-Z]+) = ([0-9]+)", text)})
    assert len(consts) >= 15, consts
    for name, value in consts.items():
        assert getattr(B, name) == value, name


def test_version_and_strerror():
    assert K.version() >> 16 == 1 and K.version() & 0xffff >= 2
    for code in (K.KVCS_OK, K.KVCS_EINVAL, K.KVCS_EUNSUPPORTED, K.KVCS_ECUDA, 99):
        assert isinstance(K.strerror(code), str) and K.strerror(code)


class FakeCache:
    def __init__(self, base=1 << 20, num_blocks=100, layout=0, layer=0,
                 head_offset=0, num_heads=8, head_bytes=256, column=0,
                 half_stride=0, block_stride=0, kernel_block_size=0, piece_bytes=0):
        self.column = column
        self.piece_bytes = piece_bytes
        self.half_stride = half_stride
        self.block_stride = block_stride
        self.kernel_block_size = kernel_block_size
        self.pool = base
        self.num_blocks = num_blocks
        self.layout = layout
        self.layer = layer
        self.head_offset = head_offset
        self.num_heads = num_heads
        self.head_bytes = head_bytes


def plan(caches, bs=16, positions=1000, sms=152):
    return K.plan_for(caches, bs, positions, num_sms=sms)


def code_of(caches, bs=16, positions=10):
    try:
        plan(caches, bs, positions)
        return 0
    except K.KvcsError as e:
        return e.code


def test_validation_codes():
    ok = FakeCache()
    assert code_of([ok]) == 0
    assert code_of([FakeCache(head_bytes=12)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(head_bytes=0)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layout=5)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layout=2, num_heads=2)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layer=-1)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(base=0)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(base=(1 << 20) + 4)]) == K.KVCS_EINVAL
    assert code_of([ok], bs=0) == K.KVCS_EINVAL
    assert code_of([FakeCache(head_offset=65530, num_heads=7)]) == K.KVCS_EUNSUPPORTED
    assert code_of([FakeCache(head_offset=65528, num_heads=8)]) == 0
    # overlapping (layer, global head) between two caches
    assert code_of([FakeCache(head_offset=0, num_heads=4),
                    FakeCache(head_offset=3, num_heads=4)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(head_offset=0, num_heads=4),
                    FakeCache(head_offset=4, num_heads=4)]) == 0
    assert code_of([FakeCache(layer=0), FakeCache(layer=1)]) == 0
    # columns: in range and each used (planning sees max(column) + 1)
    assert code_of([FakeCache(layer=0), FakeCache(layer=1, column=1)]) == 0
    assert code_of([FakeCache(layer=0), FakeCache(layer=1, column=2)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layer=0, column=-1)]) == K.KVCS_EINVAL
    # strides and sub-blocks (page = 16 * 8 * 256 = 32 KiB)
    page = 16 * 8 * 256
    assert code_of([FakeCache(half_stride=page, block_stride=2 * page)]) == 0
    assert code_of([FakeCache(half_stride=-page)]) == 0
    assert code_of([FakeCache(half_stride=page // 2)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(block_stride=page - 8)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(block_stride=page + 4)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layout=1, kernel_block_size=4)]) == 0
    assert code_of([FakeCache(layout=1, kernel_block_size=5)]) == K.KVCS_EINVAL
    # x-split: 16-byte chunks
    assert code_of([FakeCache(layout=3)]) == 0
    assert code_of([FakeCache(layout=3, head_bytes=24)]) == K.KVCS_EINVAL
    # Mamba states: 2- or 4-byte elements, not mixed with KV caches
    assert code_of([FakeCache(layout=4)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layout=4, num_heads=100, head_bytes=6, piece_bytes=2)]) == 0
    assert code_of([FakeCache(layout=4, head_bytes=6, piece_bytes=4)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layout=4, head_bytes=8, piece_bytes=8)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(layer=0, layout=4, head_bytes=8, piece_bytes=4),
                    FakeCache(layer=1)]) == K.KVCS_EINVAL
    assert code_of([FakeCache(piece_bytes=2)]) == K.KVCS_EINVAL
    # strides that are 8- but not 16-byte multiples: NHD rows and HND heads
    # stay on the bulk kernel (its misaligned instances); HND in kernel
    # sub-blocks goes to the direct kernel
    assert plan([FakeCache(block_stride=page + 8)])["kernel"] == 0
    assert plan([FakeCache(block_stride=page + 16)])["kernel"] == 0
    assert plan([FakeCache(layout=1, block_stride=page + 8)])["kernel"] == 0
    assert plan([FakeCache(layout=1, block_stride=page + 16)])["kernel"] == 0
    assert plan([FakeCache(layout=1, block_stride=page + 8, kernel_block_size=4)])["kernel"] == 1
    assert plan([FakeCache(layout=1, block_stride=page + 8, kernel_block_size=16)])["kernel"] == 0
    assert plan([FakeCache(layout=3, block_stride=page + 8)])["kernel"] == 0   # x-split
    # NHD heads of 8 mod 16 bytes (a 16-byte column would straddle two heads)
    assert plan([FakeCache(head_bytes=24)])["kernel"] == 1


def test_block_checksums_rejects_before_any_cuda_call():
    arr = K.cache_array([FakeCache(head_bytes=12)])
    reqs = B.kvcs_requests(1, 16, 32, 48, 64)
    rc = K.load_library().kvcs_block_checksums(arr, 1, 16, ctypes.byref(reqs), 4,
                                               128, None, None)
    assert rc == K.KVCS_EINVAL
    arr = K.cache_array([FakeCache()])
    rc = K.load_library().kvcs_block_checksums(arr, 1, 16, ctypes.byref(reqs), 4,
                                               None, None, None)
    assert rc == K.KVCS_EINVAL          # null output
    rc = K.load_library().kvcs_block_checksums(arr, 1, 16, ctypes.byref(reqs), 0,
                                               None, None, None)
    assert rc == K.KVCS_OK              # nothing to do, nothing enqueued


def test_noalloc_rejects_before_any_cuda_call():
    """kvcs_block_checksums_noalloc: bad arguments and more than
    KVCS_NOALLOC_MAX_CACHES caches are refused on the host (no GPU here, so
    any CUDA call would have returned KVCS_ECUDA instead)."""
    fn = K.load_library().kvcs_block_checksums_noalloc
    reqs = B.kvcs_requests(1, 16, 32, 48, 64)
    arr = K.cache_array([FakeCache(head_bytes=12)])
    assert fn(arr, 1, 16, ctypes.byref(reqs), 4, 128, None, None) == K.KVCS_EINVAL
    arr = K.cache_array([FakeCache()])
    assert fn(arr, 1, 16, ctypes.byref(reqs), 4, None, None, None) == K.KVCS_EINVAL
    assert fn(arr, 1, 16, ctypes.byref(reqs), 4, 132, None, None) == K.KVCS_EINVAL
    assert fn(arr, 1, 16, None, 4, 128, None, None) == K.KVCS_EINVAL
    assert fn(arr, 1, 16, ctypes.byref(reqs), 0, None, None, None) == K.KVCS_OK
    n = K.KVCS_NOALLOC_MAX_CACHES
    many = K.cache_array([FakeCache(layer=i, num_heads=1, head_bytes=16) for i in range(n + 1)])
    assert fn(many, n + 1, 16, ctypes.byref(reqs), 4, 128, None, None) == K.KVCS_ETOOLARGE
    assert "1024" in K.strerror(K.KVCS_ETOOLARGE)
    # within the limit the arguments pass the host checks and the call goes
    # on to its first CUDA call, which fails here without a GPU
    assert fn(many, n, 16, ctypes.byref(reqs), 4, 128, None, None) == K.KVCS_ECUDA


def test_plan_shapes():
    llama8b = [FakeCache(layer=i, num_blocks=9300) for i in range(32)]
    p = plan(llama8b, positions=9220)
    assert p["kernel"] == 0 and p["split"] == 0 and p["memsets"] == 0
    assert p["launches"] == 1 and p["grid"] == 152
    # one 32 KiB page (K or V of a layer) per unit
    assert p["units"] == 9220 * 32 * 2 and p["stage_bytes"] == 32768
    assert p["stages"] == 7 and p["smem_bytes"] <= 232448
    assert p["kv_bytes_max"] == 9220 * 32 * 2 * 32768
    # with a workspace this call would share its last units out (>= 1024
    # units per SM) ...
    assert p["dynamic"] == 1
    # 70B-shaped fp8: 16 KiB pages, a unit each, three packed per 48 KiB stage
    p = plan([FakeCache(layer=i, head_bytes=128) for i in range(80)], positions=16384)
    assert p["units"] == 16384 * 160 and p["stage_bytes"] == 49152 and p["stages"] == 4
    # one 70B-shaped request: too few positions for whole-position CTAs
    p = plan([FakeCache(layer=i, head_bytes=128) for i in range(80)], positions=128)
    assert p["split"] == 1 and p["memsets"] == 1 and p["grid"] == 152
    # ... this one (134 units per SM) keeps the fixed split; the threshold
    # is 1024 units per SM of the planned GPU
    assert p["dynamic"] == 0
    assert plan([FakeCache(layer=i, head_bytes=128) for i in range(80)],
                positions=973)["dynamic"] == 1
    assert plan([FakeCache(layer=i, head_bytes=128) for i in range(80)],
                positions=972)["dynamic"] == 0
    assert plan([FakeCache(layer=i, head_bytes=128) for i in range(80)],
                positions=972, sms=100)["dynamic"] == 1
    # latent rows of 1152 B: two units of 32 rows per 64-slot page
    p = plan([FakeCache(layout=2, num_heads=1, head_bytes=1152, layer=i)
              for i in range(61)], bs=64, positions=4096)
    assert p["units"] == 4096 * 61 * 2 and p["split"] == 0
    assert p["stage_bytes"] == 32 * 1152 and p["stages"] == 6
    # HND with 16 KiB per head (block_size 64): three heads per unit
    p = plan([FakeCache(layout=1, layer=i) for i in range(4)], bs=64, positions=500)
    assert p["units"] == 500 * 4 * 2 * 3 and p["stage_bytes"] == 49152
    # tiny pages (4 KiB): all four pages of a position packed in one stage;
    # few small positions are read one per CTA, with no zeroing
    p = plan([FakeCache(layer=i, num_heads=2, head_bytes=128) for i in range(2)],
             positions=7)
    assert p["units"] == 7 * 4 and p["stage_bytes"] == 16384 and p["split"] == 0
    assert p["grid"] == 7 and p["memsets"] == 0
    # ... but positions over 128 KiB, fewer than the SMs, are split at units
    p = plan([FakeCache(layer=i, num_heads=2, head_bytes=128) for i in range(20)],
             positions=100)
    assert p["split"] == 1 and p["memsets"] == 1 and p["grid"] == 152
    # mixed geometry: no packing
    p = plan([FakeCache(layer=0, head_bytes=128), FakeCache(layer=1, head_bytes=64)],
             positions=10)
    assert p["units"] == 10 * 4
    # odd per-head bytes, or rows too wide to stage: generic kernel, whose
    # per-(position, cache) sums are added into a zeroed output
    p = plan([FakeCache(head_bytes=24)])
    assert p["kernel"] == 1 and p["memsets"] == 1 and p["launches"] == 1
    assert plan([FakeCache(num_heads=512, head_bytes=256)])["kernel"] == 1
    # some caches for each kernel: two launches
    p = plan([FakeCache(layer=0), FakeCache(layer=1, head_bytes=24)])
    assert p["kernel"] == 2 and p["launches"] == 2 and p["memsets"] == 1
    # Mamba-like states: 32 KiB fp32 rows (bulk) and 6-byte conv rows (generic)
    ssm = [FakeCache(layer=i, layout=4, num_heads=80, head_bytes=32768, piece_bytes=4,
                     head_offset=0) for i in range(4)]
    conv = [FakeCache(layer=i, layout=4, num_heads=5376, head_bytes=6, piece_bytes=2,
                      head_offset=80) for i in range(4)]
    p = plan(ssm, positions=64)
    assert p["kernel"] == 0 and p["split"] == 1 and p["stage_bytes"] == 32768
    assert p["units"] == 64 * 4 * 80
    assert plan(conv, positions=64)["kernel"] == 1
    p = plan(ssm + conv, positions=64)
    assert p["kernel"] == 2 and p["launches"] == 2
    # more caches than one launch takes
    p = plan([FakeCache(layer=i, num_heads=1, head_bytes=16) for i in range(300)])
    assert p["launches"] == 3 and p["memsets"] == 1


def test_plan_requests_routes_mostly_partial_calls():
    """kvcs_plan_requests: with at most two positions per request, latent and
    HND caches (alike, aligned, no sub-blocks) and NHD caches of pages up to
    8 KiB go to the valid-slot kernel (kernel 3), larger NHD pages stay on
    the bulk kernel, and a mixed call reports
    its valid-slot launches among the others; more positions per request,
    or an unknown request count, plan as kvcs_plan does."""
    def pr(caches, positions, requests, bs=16):
        return K.plan_for(caches, bs, positions, num_sms=152, num_requests=requests)

    hnd = [FakeCache(layout=1, layer=i) for i in range(32)]
    nhd = [FakeCache(layout=0, layer=i) for i in range(32)]
    lat = [FakeCache(layout=2, layer=i, num_heads=1, head_bytes=1152) for i in range(61)]
    for caches, bs in ((hnd, 16), (lat, 64)):
        p = pr(caches, 4096, 4096, bs)
        halves = 1 if caches is lat else 2
        assert p["kernel"] == 3 and p["slot_launches"] == 1 and p["launches"] == 1
        assert p["threads"] == 256 and p["smem_bytes"] == 0 and p["memsets"] == 1
        assert p["units"] == 4096 * len(caches) * halves
        assert p["grid"] == 304
        assert pr(caches, 8193, 4096, bs)["slot_launches"] == 0     # > 2 a request
        assert pr(caches, 4096, -1, bs) == plan(caches, bs, 4096)   # not known
    p = pr(nhd, 4096, 4096)                      # 32 KiB NHD pages: the bulk kernel
    assert p["kernel"] == 0 and p["slot_launches"] == 0
    small = [FakeCache(layout=0, layer=i, num_heads=8, head_bytes=128) for i in range(4)]
    assert pr(small, 100, 100, bs=8)["kernel"] == 3      # 8 KiB pages
    assert pr(small, 100, 100, bs=16)["kernel"] == 0     # 16 KiB pages
    mixed = hnd[:4] + [FakeCache(layout=0, layer=10 + i) for i in range(4)]
    p = pr(mixed, 100, 100)
    assert p["kernel"] == 0 and p["slot_launches"] == 1 and p["launches"] == 2
    # HND in kernel sub-blocks, or caches of two geometries, stay on the bulk kernel
    assert pr([FakeCache(layout=1, kernel_block_size=4)], 100, 100)["slot_launches"] == 0
    two = [FakeCache(layout=1, layer=0), FakeCache(layout=1, layer=1, head_bytes=128)]
    assert pr(two, 100, 100)["slot_launches"] == 0
    # few pages: a small grid, in window groups (up to 4 x the CTAs the pages fill)
    small = pr(hnd[:2], 10, 10)                  # 40 pages: 3 CTAs, 4 window groups
    assert small["grid"] == 12
    # the dynamic share-out from 64 pages a warp (152 SMs: 304 CTAs)
    assert pr(hnd, 2432, 2432)["dynamic"] == 1          # 155,648 pages
    assert pr(hnd, 2431, 2431)["dynamic"] == 0


def test_group_and_tags_reject_bad_arguments_without_cuda():
    lib = K.load_library()
    arr = K.cache_array([FakeCache(layer=0), FakeCache(layer=1, column=1)])
    reqs = B.kvcs_requests(1, 16, 32, 48, 64)
    outs = B.kvcs_outputs(1, 0, 128, None, None, None, None, None)
    # column 1 with num_columns 1
    assert lib.kvcs_group_checksums(arr, 2, 16, ctypes.byref(reqs), 4,
                                    ctypes.byref(outs), None, None) == K.KVCS_EINVAL
    outs = B.kvcs_outputs(2, 0, 128, None, None, None, 256, None)
    # a mismatch output without expected values
    assert lib.kvcs_group_checksums(arr, 2, 16, ctypes.byref(reqs), 4,
                                    ctypes.byref(outs), None, None) == K.KVCS_EINVAL
    outs = B.kvcs_outputs(65, 0, 128, None, None, None, None, None)
    assert lib.kvcs_group_checksums(arr, 2, 16, ctypes.byref(reqs), 4,
                                    ctypes.byref(outs), None, None) == K.KVCS_EINVAL
    # unknown output flags
    outs = B.kvcs_outputs(2, 2, 128, None, None, None, None, None)
    assert lib.kvcs_group_checksums(arr, 2, 16, ctypes.byref(reqs), 4,
                                    ctypes.byref(outs), None, None) == K.KVCS_EINVAL
    assert lib.kvcs_block_checksum_tags(64, 4, 3, 0, 128, None) == K.KVCS_EINVAL
    assert lib.kvcs_block_checksum_tags(None, 32, 0, 0, None, None) == K.KVCS_OK
