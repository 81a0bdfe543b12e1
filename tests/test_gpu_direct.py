"""Pages that are not all 16-byte aligned, against the oracle through the C
ABI: the direct-load kernel (every layout, pools 0 or 8 bytes past a 16-byte
boundary, rows that are 8 mod 16 bytes, where chunks pair up over two rows,
rows and head runs past a stage, pages whose alignment alternates with the
block) and the bulk kernel's misaligned instances (NHD and latent rows of
whole 16-byte columns, and HND heads without kernel sub-blocks: interiors by
bulk copy, edge words by 8-byte asynchronous copies).  Ragged and empty
positions, first positions past 2^57 (t P wraps 2^64).  Bit-exact uint64
equality."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shifted(wl, shift, block_pad=0):
    """The same bytes at ``shift`` bytes past a 16-byte boundary, each page
    followed by ``block_pad`` spare bytes (block stride = page + pad)."""
    caches, keep = [], []
    for c in wl.caches:
        halves = 1 if c.layout == W.LAYOUT_LATENT else 2
        page = wl.block_size * c.num_heads * c.head_bytes
        stride = page + block_pad
        raw = torch.zeros(halves * c.num_blocks * stride + shift + 16, dtype=torch.uint8,
                          device=DEV)
        pool = raw[shift:shift + halves * c.num_blocks * stride]
        pool.view(halves * c.num_blocks, stride)[:, :page] = \
            c.pool.view(halves * c.num_blocks, page)
        keep.append(raw)
        extra = dict(block_stride=stride, half_stride=c.num_blocks * stride) if block_pad else {}
        caches.append(dataclasses.replace(c, pool=pool, **extra))
    return W.Workload(wl.name, wl.block_size, caches, wl.pos_offsets, wl.first_position,
                      wl.num_tokens, wl.block_ids, wl.info), keep


def _rows_bulk(c, bs):
    """NHD or latent rows of whole 16-byte columns of one head, and HND heads
    of whole 16-byte columns without kernel sub-blocks: the bulk kernel
    stages them even 8 bytes off a boundary."""
    if c.head_bytes % 16:
        return False
    if c.layout in (W.LAYOUT_HND, W.LAYOUT_XSPLIT):
        subs = getattr(c, "kernel_block_size", 0) not in (0, bs)
        return not (subs and c.layout == W.LAYOUT_HND) and c.head_bytes * bs <= 65536
    if c.layout not in (W.LAYOUT_NHD, W.LAYOUT_LATENT):
        return False
    row = c.num_heads * c.head_bytes if c.layout == W.LAYOUT_NHD else c.head_bytes
    return row <= 65536


def _check(wl, kernel=None):
    from gpu_helpers import full_oracle, gpu_checksums
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    if kernel is None:
        kernel = 0 if all(_rows_bulk(c, wl.block_size) for c in wl.caches) else 1
    assert plan["kernel"] == kernel, plan
    got, st = gpu_checksums(wl)
    exp, est = full_oracle(wl)
    assert st == est == 0
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, f"{bad.size} of {got.size} differ, first {bad[:8].tolist()}"


CASES = [
    # (layout, heads, head_bytes, block_size, kernel_block_size)
    (W.LAYOUT_NHD, 8, 256, 16, 0),      # the 8B-shaped row, 128 chunks
    (W.LAYOUT_NHD, 3, 24, 16, 0),       # 72-byte rows: chunks pair over two rows
    (W.LAYOUT_NHD, 1, 8, 5, 0),         # one word per row
    (W.LAYOUT_NHD, 5, 40, 3, 0),        # 200-byte rows
    (W.LAYOUT_LATENT, 1, 72, 16, 0),
    (W.LAYOUT_LATENT, 1, 1152, 64, 0),  # the MLA row
    (W.LAYOUT_HND, 8, 256, 16, 0),
    (W.LAYOUT_HND, 3, 24, 7, 0),        # head runs alternate their alignment
    (W.LAYOUT_HND, 2, 8, 16, 0),
    (W.LAYOUT_HND, 4, 64, 16, 4),       # kernel sub-blocks
    (W.LAYOUT_HND, 3, 24, 12, 3),
    (W.LAYOUT_XSPLIT, 4, 64, 16, 0),
    (W.LAYOUT_XSPLIT, 2, 48, 7, 0),
]


@pytest.mark.parametrize("shift", [0, 8])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"l{c[0]}h{c[1]}b{c[2]}bs{c[3]}k{c[4]}")
def test_direct_kernel_matches_oracle(case, shift):
    layout, heads, hb, bs, kbs = case
    wl = W.random_case(21, DEV, layout=layout, layers=3, heads=heads, head_bytes=hb,
                       block_size=bs, lengths=(70, 33, 5, bs), first_positions=(1, 0, 0, 0),
                       extra_positions=(0, 1, 0, 0))
    if kbs:
        wl = W.Workload(wl.name, bs, [dataclasses.replace(c, kernel_block_size=kbs)
                                      for c in wl.caches], wl.pos_offsets, wl.first_position,
                        wl.num_tokens, wl.block_ids, wl.info)
    aligned16 = hb % 16 == 0 and (layout != W.LAYOUT_NHD or (heads * hb) % 16 == 0)
    if shift == 0 and aligned16:
        # 16-byte geometry: force the direct kernel with blocks 8 mod 16 apart
        wl, keep = _shifted(wl, 0, block_pad=8)
    else:
        wl, keep = _shifted(wl, shift)
    _check(wl)


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND])
def test_rows_and_head_runs_past_a_stage(layout):
    """128 KiB NHD rows (64 heads of 2 KiB) and 128 KiB HND head runs
    (block_size 512): each lane owns several chunk columns."""
    if layout == W.LAYOUT_NHD:
        wl = W.random_case(22, DEV, layout=layout, layers=2, heads=64, head_bytes=2048,
                           block_size=2, lengths=(5, 2))
    else:
        wl = W.random_case(22, DEV, layout=layout, layers=2, heads=2, head_bytes=256,
                           block_size=512, lengths=(700, 3))
    wl, keep = _shifted(wl, 8)
    _check(wl)


def test_many_positions_and_caches_misaligned():
    """Thousands of positions over 16 layers, 8 bytes off: warps' page
    ranges start and end inside positions and inside a position's caches."""
    g = torch.Generator().manual_seed(5)
    lengths = torch.randint(1, 400, (96,), generator=g).tolist()
    wl = W.random_case(23, DEV, layout=W.LAYOUT_NHD, layers=16, heads=2, head_bytes=24,
                       block_size=16, lengths=lengths)
    wl, keep = _shifted(wl, 8)
    _check(wl, kernel=1)


def test_position_past_2_pow_57_misaligned():
    wl = W.random_case(24, DEV, layout=W.LAYOUT_NHD, layers=2, heads=3, head_bytes=24,
                       block_size=16, lengths=((1 << 57) * 16 + 20,),
                       first_positions=(1 << 57,))
    wl, keep = _shifted(wl, 8)
    _check(wl)


def test_bad_block_id_and_columns_misaligned():
    """A bad block id gives 0 and the status bit; replica columns add per
    column; an accumulating call adds onto earlier contents."""
    from gpu_helpers import full_oracle
    wl = W.random_case(25, DEV, layout=W.LAYOUT_NHD, layers=4, heads=2, head_bytes=24,
                       block_size=8, lengths=(40, 17))
    wl, keep = _shifted(wl, 8)
    exp, _ = full_oracle(wl)
    ids = wl.block_ids.clone()
    ids[2] = wl.caches[0].num_blocks + 5
    bad = W.Workload(wl.name, wl.block_size, wl.caches, wl.pos_offsets, wl.first_position,
                     wl.num_tokens, ids, wl.info)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = K.workload_checksums(bad, status=status)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint64)
    want = exp.copy()
    want[2] = 0
    assert int(status.item()) & K.KVCS_STATUS_BAD_BLOCK_ID
    assert np.array_equal(got, want)
    # two columns (layers 0-1 and 2-3), their row sum is the checksum
    cols = [dataclasses.replace(c, column=i // 2) for i, c in enumerate(wl.caches)]
    vals = K.group_checksums(cols, wl.block_size, wl.pos_offsets, wl.first_position,
                             wl.num_tokens, wl.block_ids, 2)
    torch.cuda.synchronize()
    v = vals.cpu().numpy().view(np.uint64)
    assert np.array_equal(v.sum(axis=1, dtype=np.uint64), exp)
    # accumulate the same call onto the values: every word doubles
    K.group_checksums(cols, wl.block_size, wl.pos_offsets, wl.first_position,
                      wl.num_tokens, wl.block_ids, 2, values=vals, accumulate=True)
    torch.cuda.synchronize()
    assert np.array_equal(vals.cpu().numpy().view(np.uint64), v * np.uint64(2))


MIS_ROWS = [
    # (layout, heads, head_bytes, block_size, lengths, first_positions)
    (W.LAYOUT_NHD, 8, 256, 16, (70, 33, 5, 16), (1, 0, 0, 0)),     # 2 KiB rows
    (W.LAYOUT_NHD, 2, 32, 16, (100, 1, 17), (0, 0, 1)),            # 64-byte rows
    (W.LAYOUT_NHD, 8, 128, 16, (60, 37), (0, 0)),                  # fp8-shaped 16 KiB pages, packed
    (W.LAYOUT_LATENT, 1, 1152, 64, (200, 64, 1), (0, 0, 0)),       # the MLA row
    (W.LAYOUT_LATENT, 1, 16, 4, (9, 1, 5), (0, 0, 1)),             # 16-byte rows: edges only at nv 1
    (W.LAYOUT_NHD, 64, 1024, 1, (7, 3), (0, 0)),                   # 64 KiB rows, a unit each
    (W.LAYOUT_NHD, 2, 64, 16, [16 * k + 1 for k in range(40)], list(range(40))),  # one-token blocks
]


@pytest.mark.parametrize("place", ["base8", "stride8", "v_only"])
@pytest.mark.parametrize("case", MIS_ROWS, ids=lambda c: f"l{c[0]}h{c[1]}b{c[2]}bs{c[3]}")
def test_misaligned_rows_bulk_instance(case, place):
    """NHD and latent rows 8 bytes off a 16-byte boundary: every page
    (base8), every other block (stride8), or only the V pages (v_only: the
    half stride is 8 mod 16) go to the bulk kernel's misaligned-rows
    instance and give the oracle's checksums."""
    layout, heads, hb, bs, lengths, fps = case
    if layout == W.LAYOUT_LATENT and place == "v_only":
        pytest.skip("a latent cache has no V pages")
    wl = W.random_case(31, DEV, layout=layout, layers=3, heads=heads, head_bytes=hb,
                       block_size=bs, lengths=lengths, first_positions=fps)
    if place == "base8":
        wl, keep = _shifted(wl, 8)
    elif place == "stride8":
        wl, keep = _shifted(wl, 0, block_pad=8)
    else:
        caches, keep = [], []
        for c in wl.caches:
            page = bs * c.num_heads * c.head_bytes
            raw = torch.zeros(2 * c.num_blocks * page + 8, dtype=torch.uint8, device=DEV)
            v = c.pool.view(2, c.num_blocks * page)
            raw[:c.num_blocks * page] = v[0]
            raw[c.num_blocks * page + 8:] = v[1]
            keep.append(raw)
            caches.append(dataclasses.replace(c, pool=raw, half_stride=c.num_blocks * page + 8))
        wl = W.Workload(wl.name, bs, caches, wl.pos_offsets, wl.first_position,
                        wl.num_tokens, wl.block_ids, wl.info)
    _check(wl, kernel=0)


MIS_HND = [
    # (heads, head_bytes, block_size, lengths, first_positions)
    (8, 256, 16, (70, 33, 5, 16), (1, 0, 0, 0)),       # 32 KiB pages, a unit each
    (8, 128, 16, (60, 37), (0, 0)),                     # fp8-shaped 16 KiB pages, packed
    (2, 32, 16, (100, 1, 17), (0, 0, 1)),               # 1 KiB pages, many to a stage
    (4, 256, 64, (150, 64, 9), (0, 0, 0)),              # 16 KiB heads: two units a page
    (8, 64, 16, [16 * k + 1 for k in range(40)], list(range(40))),  # one-token blocks
]


@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_XSPLIT])
@pytest.mark.parametrize("place", ["base8", "stride8", "v_only"])
@pytest.mark.parametrize("case", MIS_HND, ids=lambda c: f"h{c[0]}b{c[1]}bs{c[2]}")
def test_misaligned_heads_bulk_instances(case, place, layout):
    """HND and x-split heads 8 bytes off a 16-byte boundary: every page
    (base8), every other block (stride8), or only the V pages (v_only) go
    to the bulk kernel's misaligned-heads instances (a unit's heads, all
    their slots, as one run: interior by bulk copy, edge words by 8-byte
    copies) and give the oracle's checksums."""
    heads, hb, bs, lengths, fps = case
    wl = W.random_case(33, DEV, layout=layout, layers=3, heads=heads, head_bytes=hb,
                       block_size=bs, lengths=lengths, first_positions=fps)
    if place == "base8":
        wl, keep = _shifted(wl, 8)
    elif place == "stride8":
        wl, keep = _shifted(wl, 0, block_pad=8)
    else:
        caches, keep = [], []
        for c in wl.caches:
            page = bs * c.num_heads * c.head_bytes
            raw = torch.zeros(2 * c.num_blocks * page + 8, dtype=torch.uint8, device=DEV)
            v = c.pool.view(2, c.num_blocks * page)
            raw[:c.num_blocks * page] = v[0]
            raw[c.num_blocks * page + 8:] = v[1]
            keep.append(raw)
            caches.append(dataclasses.replace(c, pool=raw, half_stride=c.num_blocks * page + 8))
        wl = W.Workload(wl.name, bs, caches, wl.pos_offsets, wl.first_position,
                        wl.num_tokens, wl.block_ids, wl.info)
    _check(wl, kernel=0)


def test_misaligned_rows_whole_positions_and_bad_ids():
    """304 positions (whole-position mode, plain stores) of 8-byte-shifted
    NHD pools, with a bad block id: 0 there and the status bit."""
    from gpu_helpers import full_oracle
    wl = W.random_case(32, DEV, layout=W.LAYOUT_NHD, layers=4, heads=4, head_bytes=64,
                       block_size=16, lengths=[64] * 76)
    wl, keep = _shifted(wl, 8)
    assert wl.num_positions == 304
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0
    exp, _ = full_oracle(wl)
    ids = wl.block_ids.clone()
    ids[100] = -3
    bad = W.Workload(wl.name, wl.block_size, wl.caches, wl.pos_offsets, wl.first_position,
                     wl.num_tokens, ids, wl.info)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = K.workload_checksums(bad, status=status)
    torch.cuda.synchronize()
    want = exp.copy()
    want[100] = 0
    assert int(status.item()) & K.KVCS_STATUS_BAD_BLOCK_ID
    assert np.array_equal(out.cpu().numpy().view(np.uint64), want)
