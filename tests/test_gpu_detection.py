"""The checksum as a KV-transfer failure detector, on the GPU: stored
(tagged) checksums of a cache are taken, one fault is injected in the host
data (a flipped byte, two swapped tokens, swapped block ids, swapped layer
numbers, swapped heads), and the verifying call flags exactly the block
positions the fault touched.  Faults are made in the data only; nothing
faults the GPU."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make():
    wl = W.random_case(17, DEV, layout=W.LAYOUT_NHD, layers=3, heads=4, head_bytes=64,
                       block_size=16, lengths=(70, 40), spare_blocks=2)
    n = wl.num_positions
    g = torch.Generator(device=DEV).manual_seed(5)
    hashes = torch.randint(0, 256, (n, 32), dtype=torch.uint8, device=DEV, generator=g)
    tags = K.block_checksum_tags(hashes, 0xF00D)
    return wl, tags


def verify(wl, tags, stored=None):
    n = wl.num_positions
    rows = torch.empty(n, dtype=torch.int64, device=DEV)
    extra = {}
    if stored is not None:
        extra = dict(expected=stored, mismatch=torch.empty(n, dtype=torch.uint8, device=DEV),
                     mismatch_count=torch.zeros(1, dtype=torch.int32, device=DEV))
    K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                      wl.num_tokens, wl.block_ids, 1, row_sums=rows, tags=tags,
                      total_positions=n, **extra)
    torch.cuda.synchronize()
    if stored is None:
        return rows
    return (extra["mismatch"].cpu().numpy().nonzero()[0].tolist(),
            int(extra["mismatch_count"].item()))


def pages(c, bs):
    return c.pool.view(2, c.num_blocks, bs, c.num_heads, c.head_bytes)


FAULTS = ["byte", "tokens", "block_ids", "layers", "heads"]


@pytest.mark.parametrize("fault", FAULTS)
def test_injected_fault_is_flagged_where_it_lands(fault):
    wl, tags = make()
    stored = verify(wl, tags)
    assert verify(wl, tags, stored) == ([], 0)
    ids = wl.block_ids.cpu().tolist()
    bs = wl.block_size
    if fault == "byte":                     # one bit of layer 1's V, position 2
        v = pages(wl.caches[1], bs)
        v[1, ids[2], 5, 3, 17] ^= 0x10
        expect = [2]
    elif fault == "tokens":                 # two slots of position 0 swapped in layer 0
        v = pages(wl.caches[0], bs)
        a = v[:, ids[0], 3].clone()
        v[:, ids[0], 3] = v[:, ids[0], 9]
        v[:, ids[0], 9] = a
        expect = [0]
    elif fault == "block_ids":              # the table points positions 1 and 6 at each other's pages
        t = wl.block_ids.clone()
        t[1], t[6] = wl.block_ids[6], wl.block_ids[1]
        wl = dataclasses.replace(wl, block_ids=t)
        expect = [1, 6]
    elif fault == "layers":                 # layers 0 and 2 exchange their numbers
        c = wl.caches
        wl = dataclasses.replace(wl, caches=[dataclasses.replace(c[0], layer=c[2].layer),
                                             c[1], dataclasses.replace(c[2], layer=c[0].layer)])
        expect = list(range(wl.num_positions))
    else:                                   # heads 0 and 3 of layer 2 swapped in position 4
        v = pages(wl.caches[2], bs)
        a = v[:, ids[4], :, 0].clone()
        v[:, ids[4], :, 0] = v[:, ids[4], :, 3]
        v[:, ids[4], :, 3] = a
        expect = [4]
    flagged, count = verify(wl, tags, stored)
    assert flagged == expect and count == len(expect)
