"""More cache layouts through the C ABI: explicit half/block strides
([num_blocks, 2, ...] pools, separate K and V tensors, padded blocks) and
HND kernel sub-blocks.  Each layout is built from a canonical pool with
torch views (data movement only) and must give the canonical checksums,
which are checked against the oracle."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(wl):
    from gpu_helpers import gpu_checksums
    return gpu_checksums(wl)


def canonical(seed, layout, hb=64, bs=16, heads=4, layers=3, lengths=(70, 33, 5)):
    wl = W.random_case(seed, DEV, layout=layout, layers=layers, heads=heads,
                       head_bytes=hb, block_size=bs, lengths=lengths)
    from gpu_helpers import full_oracle
    exp, _ = full_oracle(wl)
    got, st = run(wl)
    assert st == 0 and np.array_equal(got, exp)
    return wl, exp


def with_caches(wl, caches):
    return W.Workload(wl.name, wl.block_size, caches, wl.pos_offsets, wl.first_position,
                      wl.num_tokens, wl.block_ids)


def page_bytes(wl, c):
    return wl.block_size * c.num_heads * c.head_bytes


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND])
@pytest.mark.parametrize("hb", [64, 24])      # bulk kernel, direct kernel
def test_kv_interleaved_per_block(layout, hb):
    """[num_blocks, 2, page]: half_stride = page, block_stride = 2 page."""
    wl, exp = canonical(1, layout, hb=hb)
    caches = []
    for c in wl.caches:
        pb = page_bytes(wl, c)
        inter = c.pool.view(2, c.num_blocks, pb).transpose(0, 1).contiguous().view(-1)
        caches.append(dataclasses.replace(c, pool=inter, half_stride=pb, block_stride=2 * pb))
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("v_first", [False, True])
def test_separate_k_and_v_tensors(v_first):
    wl, exp = canonical(2, W.LAYOUT_NHD)
    caches = []
    keep = []
    for c in wl.caches:
        pb = page_bytes(wl, c)
        halves = c.pool.view(2, c.num_blocks * pb)
        if v_first:                 # V allocated before K: often a negative stride
            v = halves[1].clone()
            k = halves[0].clone()
        else:
            k = halves[0].clone()
            v = halves[1].clone()
        keep.append((k, v))
        caches.append(dataclasses.replace(c, pool=k, v_pool=v))
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_LATENT])
@pytest.mark.parametrize("pad", [256, 8])     # 16-byte and 8-byte block strides
def test_padded_blocks(layout, pad):
    hb = 1152 if layout == W.LAYOUT_LATENT else 64
    heads = 1 if layout == W.LAYOUT_LATENT else 4
    wl, exp = canonical(3, layout, hb=hb, heads=heads)
    caches = []
    for c in wl.caches:
        pb = page_bytes(wl, c)
        halves = 1 if layout == W.LAYOUT_LATENT else 2
        stride = pb + pad
        buf = torch.zeros(halves * c.num_blocks * stride, dtype=torch.uint8, device=DEV)
        buf.view(halves * c.num_blocks, stride)[:, :pb] = c.pool.view(halves * c.num_blocks, pb)
        caches.append(dataclasses.replace(c, pool=buf, block_stride=stride,
                                          half_stride=c.num_blocks * stride))
    plan = K.plan_for(caches, wl.block_size, wl.num_positions)
    # blocks 8 mod 16 apart: NHD and latent rows and HND heads stay on the
    # bulk kernel (its misaligned instances)
    assert plan["kernel"] == 0
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("bs,kbs", [(16, 1), (16, 4), (16, 8), (16, 16), (48, 12), (48, 6),
                                    (32, 2)])
@pytest.mark.parametrize("hb", [64, 24])
def test_hnd_kernel_sub_blocks(bs, kbs, hb):
    """HND blocks split into block_size / kbs sub-blocks:
    [2, num_blocks, sub, heads, kbs, hb]."""
    heads = 4
    wl, exp = canonical(4, W.LAYOUT_HND, hb=hb, bs=bs, heads=heads)
    r = bs // kbs
    caches = []
    for c in wl.caches:
        v = c.pool.view(2, c.num_blocks, heads, r, kbs, hb).permute(0, 1, 3, 2, 4, 5)
        caches.append(dataclasses.replace(c, pool=v.contiguous().view(-1),
                                          kernel_block_size=kbs))
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


def test_nhd_kernel_block_size_is_the_same_memory():
    wl, exp = canonical(5, W.LAYOUT_NHD)
    caches = [dataclasses.replace(c, kernel_block_size=4) for c in wl.caches]
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("hb,bs", [(64, 16), (256, 16), (32, 5), (16, 1)])
@pytest.mark.parametrize("pad", [0, 8])       # bulk kernel, its misaligned-heads instance
def test_xsplit_layout(hb, bs, pad):
    """[2, num_blocks, heads, head_bytes / 16, block_size, 16]: the x-split
    layout (16-byte x chunks) for K and V pages."""
    heads = 4
    wl, exp = canonical(6, W.LAYOUT_NHD, hb=hb, bs=bs, heads=heads,
                        lengths=(70, 33, 5))
    C = hb // 16
    caches = []
    for c in wl.caches:
        v = c.pool.view(2, c.num_blocks, bs, heads, C, 16).permute(0, 1, 3, 4, 2, 5)
        x = v.contiguous().view(2 * c.num_blocks, -1)
        pb = x.shape[1]
        if pad:
            buf = torch.zeros(2 * c.num_blocks, pb + pad, dtype=torch.uint8, device=DEV)
            buf[:, :pb] = x
            spec = dataclasses.replace(c, pool=buf.view(-1), layout=W.LAYOUT_XSPLIT,
                                       block_stride=pb + pad,
                                       half_stride=c.num_blocks * (pb + pad))
        else:
            spec = dataclasses.replace(c, pool=x.view(-1), layout=W.LAYOUT_XSPLIT)
        caches.append(spec)
    plan = K.plan_for(caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0
    got, st = run(with_caches(wl, caches))
    assert st == 0 and np.array_equal(got, exp)


def _relaid(c, bs, kind):
    """Bytes of canonical pool ``c`` (NHD, or latent) in layout ``kind``."""
    if kind in ("nhd", "latent"):
        return c.pool.clone(), dict()
    v = c.pool.view(2, c.num_blocks, bs, c.num_heads, c.head_bytes)
    if kind == "hnd":
        return v.permute(0, 1, 3, 2, 4).contiguous().view(-1), dict(layout=W.LAYOUT_HND)
    if kind == "hnd_sub4":
        return (v.view(2, c.num_blocks, bs // 4, 4, c.num_heads, c.head_bytes)
                .permute(0, 1, 2, 4, 3, 5).contiguous().view(-1),
                dict(layout=W.LAYOUT_HND, kernel_block_size=4))
    assert kind == "xsplit"
    return (v.view(2, c.num_blocks, bs, c.num_heads, c.head_bytes // 16, 16)
            .permute(0, 1, 3, 4, 2, 5).contiguous().view(-1), dict(layout=W.LAYOUT_XSPLIT))


@pytest.mark.parametrize("kind", ["nhd", "hnd", "hnd_sub4", "xsplit", "latent"])
@pytest.mark.parametrize("heads,hb", [(8, 256), (2, 32)])   # >= and < 256 word columns
def test_misaligned_pools_every_layout(kind, heads, hb):
    """Pools starting 8 bytes past a 16-byte boundary give the canonical
    checksums in every layout."""
    bs = 16
    if kind == "latent":
        heads, hb = 1, hb * 4 + 8
    wl, exp = canonical(9, W.LAYOUT_LATENT if kind == "latent" else W.LAYOUT_NHD, hb=hb,
                        bs=bs, heads=heads, layers=2, lengths=(70, 33, 5))
    caches, keep = [], []
    for c in wl.caches:
        data, extra = _relaid(c, bs, kind)
        raw = torch.zeros(data.numel() + 8, dtype=torch.uint8, device=DEV)
        raw[8:] = data
        keep.append(raw)
        caches.append(dataclasses.replace(c, pool=raw[8:], **extra))
    wl2 = with_caches(wl, caches)
    # NHD rows of whole 16-byte columns, HND heads (no sub-blocks) and x-split
    # heads go to the bulk kernel's misaligned instances; HND sub-blocks (and
    # 8-mod-16 latent rows) to the direct kernel
    expect = 0 if kind in ("nhd", "hnd", "xsplit") else 1
    assert K.plan_for(wl2.caches, bs, wl2.num_positions)["kernel"] == expect
    got, st = run(wl2)
    assert st == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("layout,kbs,hb,bs", [(W.LAYOUT_XSPLIT, 0, 64, 16),
                                              (W.LAYOUT_XSPLIT, 0, 48, 7),
                                              (W.LAYOUT_HND, 4, 64, 16),
                                              (W.LAYOUT_HND, 3, 24, 12),
                                              (W.LAYOUT_HND, 8, 256, 32)])
def test_xsplit_and_sub_blocks_against_the_oracle_directly(layout, kbs, hb, bs):
    """Random pools read as x-split or sub-blocked HND by both the GPU and
    the oracle (which addresses these layouts itself)."""
    from gpu_helpers import full_oracle
    wl = W.random_case(12, DEV, layout=layout, layers=3, heads=4, head_bytes=hb,
                       block_size=bs, lengths=(70, 33, 5))
    wl = with_caches(wl, [dataclasses.replace(c, kernel_block_size=kbs) for c in wl.caches])
    exp, est = full_oracle(wl)
    got, st = run(wl)
    assert st == est == 0 and np.array_equal(got, exp)


@pytest.mark.parametrize("kind", ["interleaved", "separate", "separate_v_first", "padded16",
                                  "padded8"])
@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND])
def test_strided_pools_against_the_oracle_directly(kind, layout):
    """Pages placed by explicit strides or in separate K and V tensors, read
    by the GPU and by the oracle (which takes the strides itself; a separate
    V tensor is appended to the K bytes on the host)."""
    from gpu_helpers import full_oracle
    wl = W.random_case(13, DEV, layout=layout, layers=3, heads=4, head_bytes=64,
                       block_size=16, lengths=(70, 33, 5))
    caches, keep = [], []
    for c in wl.caches:
        pb = page_bytes(wl, c)
        halves = c.pool.view(2, c.num_blocks, pb)
        if kind == "interleaved":
            pool = halves.transpose(0, 1).contiguous().view(-1)
            caches.append(dataclasses.replace(c, pool=pool, half_stride=pb, block_stride=2 * pb))
        elif kind.startswith("separate"):
            if kind == "separate_v_first":
                v = halves[1].clone()
                k = halves[0].clone()
            else:
                k = halves[0].clone()
                v = halves[1].clone()
            keep.append((k, v))
            caches.append(dataclasses.replace(c, pool=k.view(-1), v_pool=v.view(-1)))
        else:
            pad = 16 if kind == "padded16" else 8
            stride = pb + pad
            buf = torch.zeros(2 * c.num_blocks * stride, dtype=torch.uint8, device=DEV)
            buf.view(2 * c.num_blocks, stride)[:, :pb] = halves.reshape(2 * c.num_blocks, pb)
            caches.append(dataclasses.replace(c, pool=buf, block_stride=stride,
                                              half_stride=c.num_blocks * stride))
    wl2 = with_caches(wl, caches)
    exp, est = full_oracle(wl2)
    got, st = run(wl2)
    assert st == est == 0 and np.array_equal(got, exp)
