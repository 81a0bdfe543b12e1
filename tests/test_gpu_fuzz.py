"""Seeded random geometries against the oracle: every position of each case
(one exact value per block position: module docstring item 2 of the
checksum page), so that the planner's choices meet in combinations no
hand-written case names: layout and kernel sub-blocks, pools and strides 0
or 8 bytes off a 16-byte boundary, heads of 8 mod 16 bytes, request shapes
from the newest block of each request to whole prefixes, replica-key
columns, accumulating calls and a caller workspace."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    """One random call: its workload (pools possibly re-placed), the number
    of columns, whether it accumulates and whether it passes a workspace."""
    g = torch.Generator().manual_seed(seed)

    def pick(xs):
        return xs[int(torch.randint(0, len(xs), (1,), generator=g))]

    layout = pick([W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_LATENT, W.LAYOUT_XSPLIT])
    bs = pick([1, 4, 7, 16, 32, 64])
    if layout == W.LAYOUT_LATENT:
        heads, hb = 1, pick([16, 64, 72, 576, 1152])
    elif layout == W.LAYOUT_XSPLIT:
        heads, hb = pick([1, 2, 4, 8]), pick([16, 32, 64, 128, 256])
    else:
        heads, hb = pick([1, 2, 3, 4, 8]), pick([16, 24, 32, 48, 64, 128, 256])
    layers = pick([1, 2, 3, 5])
    n = pick([1, 3, 17, 60, 160])
    shape = pick(["newest", "prefix", "mixed"])
    big = seed % 8 == 7
    if big:
        # enough small units for the dynamic share-out (1024 a SM)
        layout = pick([W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_XSPLIT])
        heads, hb, bs, layers, n, shape = 1, pick([16, 32]), pick([4, 16]), 6, 1200, "prefix"
    lengths, first, extra = [], [], []
    for _ in range(n):
        tokens = int(torch.randint(1, 40 * bs + 1, (1,), generator=g))
        nblk = -(-tokens // bs)
        lengths.append(tokens)
        if shape == "newest":
            first.append(nblk - 1)
            extra.append(0)
        elif shape == "prefix":
            first.append(0)
            extra.append(0)
        else:
            first.append(int(torch.randint(0, nblk, (1,), generator=g)))
            extra.append(int(torch.randint(0, 2, (1,), generator=g)))
    args = dict(layers=layers, block_size=bs, lengths=lengths, first_positions=first,
                extra_positions=extra)
    wl = W.random_case(1000 + seed, DEV, layout=layout, heads=heads, head_bytes=hb, **args)
    if seed % 5 == 3 and not big:
        # a second group of caches with 24-byte heads (the direct-load
        # kernel) in the same call: same requests and block ids, other layers
        other = W.random_case(1000 + seed, DEV, layout=W.LAYOUT_NHD, heads=2, head_bytes=24,
                              layer_numbers=[100 + i for i in range(layers)], **args)
        assert torch.equal(other.block_ids, wl.block_ids)
        wl = W.Workload(wl.name, bs, list(wl.caches) + list(other.caches), wl.pos_offsets,
                        wl.first_position, wl.num_tokens, wl.block_ids, wl.info)
    kbs = 0
    if layout == W.LAYOUT_HND and bs > 1 and pick([False, True]):
        kbs = pick([d for d in (1, 2, 4, 8, 16) if d < bs and bs % d == 0] or [0])
    shift = pick([0, 0, 8])
    pad = pick([0, 0, 8, 16])
    caches, keep = [], []
    for c in wl.caches:
        halves = 1 if c.layout == W.LAYOUT_LATENT else 2
        page = bs * c.num_heads * c.head_bytes
        stride = page + pad
        raw = torch.zeros(halves * c.num_blocks * stride + shift + 16, dtype=torch.uint8,
                          device=DEV)
        pool = raw[shift:shift + halves * c.num_blocks * stride]
        pool.view(halves * c.num_blocks, stride)[:, :page] = \
            c.pool.view(halves * c.num_blocks, page)
        keep.append(raw)
        extra_fields = dict(block_stride=stride, half_stride=c.num_blocks * stride) if pad else {}
        if kbs and c.layout == W.LAYOUT_HND:
            extra_fields["kernel_block_size"] = kbs
        caches.append(dataclasses.replace(c, pool=pool, **extra_fields))
    cols = pick([1, 1, 2, 3]) if len(caches) >= 3 else 1
    caches = [dataclasses.replace(c, column=i % cols) for i, c in enumerate(caches)]
    wl = W.Workload(wl.name, bs, caches, wl.pos_offsets, wl.first_position, wl.num_tokens,
                    wl.block_ids, wl.info)
    return wl, keep, cols, pick([False, True]), pick([False, True])


@pytest.mark.parametrize("block", range(16))
def test_random_geometries_match_oracle(block):
    from gpu_helpers import full_oracle
    for seed in range(block * 25, (block + 1) * 25):
        wl, keep, cols, accumulate, workspace = _case(seed)
        exp, est = full_oracle(wl)
        assert est == 0, seed
        exp = exp.reshape(-1)
        ws = (torch.full((K.KVCS_WORKSPACE_WORDS,), -1, dtype=torch.int64, device=DEV)
              if workspace else None)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        vals = torch.zeros((wl.num_positions, cols), dtype=torch.int64, device=DEV)
        calls = 2 if accumulate else 1
        for _ in range(calls):
            K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                              wl.num_tokens, wl.block_ids, cols, values=vals,
                              accumulate=accumulate, total_positions=wl.num_positions,
                              workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, seed
        got = vals.cpu().numpy().view(np.uint64).sum(axis=1, dtype=np.uint64)
        want = exp * np.uint64(calls)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (seed, bad.size, got.size, bad[:6].tolist())
