"""Seeded random calls of the KV write fused with the checksum
(kvcs_write_kv), all layers of a call in one launch: the written pools equal
a plain scatter (data movement with torch), and the running word of every
block equals the oracle's checksum of the tokens written to it (the
checksum page, module docstring item 2, over the written pages) -- across
layouts, kernel sub-blocks, head geometry, block sizes, token orders with
padding tokens, and pools 0 or 8 bytes off a 16-byte boundary."""

import numpy as np
import pytest
import torch

from helpers import W, OracleCache, OracleRequests, c_form, host_bytes
from test_gpu_write import to_canonical
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_case(seed):
    g = torch.Generator().manual_seed(seed)

    def pick(xs):
        return xs[int(torch.randint(0, len(xs), (1,), generator=g))]

    layout = pick([W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_XSPLIT, W.LAYOUT_LATENT])
    bs = pick([1, 4, 8, 16, 32])
    if layout == W.LAYOUT_LATENT:
        heads, hb = 1, pick([8, 40, 64, 576, 1152])
    elif layout == W.LAYOUT_XSPLIT:
        heads, hb = pick([1, 2, 4, 8]), pick([16, 32, 64, 256])
    else:
        heads, hb = pick([1, 2, 3, 8]), pick([8, 24, 32, 64, 128, 256])
    kbs = pick([d for d in (1, 2, 4) if d < bs and bs % d == 0] or [0]) \
        if layout == W.LAYOUT_HND and pick([False, True]) else 0
    layers = pick([1, 2, 4])
    shift = pick([0, 0, 8])
    lengths = [int(torch.randint(1, 6 * bs + 2, (1,), generator=g))
               for _ in range(pick([1, 3, 20]))]
    nblk = [-(-n // bs) for n in lengths]
    nb = sum(nblk) + pick([0, 3])
    ids = torch.randperm(nb, generator=g)[:sum(nblk)].tolist()
    tables, k = [], 0
    for c in nblk:
        tables.append(ids[k:k + c])
        k += c
    halves = 1 if layout == W.LAYOUT_LATENT else 2
    page = bs * heads * hb
    caches, keep = [], []
    for li in range(layers):
        raw = torch.zeros(halves * nb * page + shift + 16, dtype=torch.uint8, device=DEV)
        keep.append(raw)
        caches.append(W.CacheSpec(raw[shift:shift + halves * nb * page], nb, layout, li, 0,
                                  heads, hb, kernel_block_size=kbs))
    ref = [torch.zeros(to_canonical(c, bs).shape, dtype=torch.uint8, device=DEV)
           for c in caches]
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    toks = [(r, t) for r, n in enumerate(lengths) for t in range(n)]
    order = torch.randperm(len(toks), generator=g).tolist()
    cuts = sorted(set([0, len(order)] + torch.randint(0, len(order) + 1, (2,),
                                                       generator=g).tolist()))
    for a, b in zip(cuts, cuts[1:]):
        sel = [toks[i] for i in order[a:b]]
        slots = [tables[r][t // bs] * bs + t % bs for r, t in sel] + [-1]
        pos = [t for _, t in sel] + [0]
        n = len(slots)
        slot_t = torch.tensor(slots, dtype=torch.int64, device=DEV)
        pos_t = torch.tensor(pos, dtype=torch.int64, device=DEV)
        keys, vals = [], []
        for _ in caches:
            shape = (n, hb) if layout == W.LAYOUT_LATENT else (n, heads, hb)
            keys.append(torch.randint(0, 256, shape, dtype=torch.uint8, generator=g).to(DEV))
            vals.append(None if layout == W.LAYOUT_LATENT else
                        torch.randint(0, 256, shape, dtype=torch.uint8, generator=g).to(DEV))
        K.write_kv(caches, bs, keys, vals, slot_t, pos_t, block_sums=sums, status=status)
        live = slot_t >= 0
        blk, o = slot_t[live] // bs, slot_t[live] % bs
        for li in range(layers):
            if layout == W.LAYOUT_LATENT:
                ref[li][blk, o] = keys[li][live]
            else:
                ref[li][0, blk, o] = keys[li][live]
                ref[li][1, blk, o] = vals[li][live]
    torch.cuda.synchronize()
    assert int(status.item()) == 0, seed
    for li, c in enumerate(caches):
        assert torch.equal(to_canonical(c, bs).contiguous(), ref[li]), (seed, li)
    ocaches = [OracleCache(host_bytes(r), nb, W.LAYOUT_LATENT if layout == W.LAYOUT_LATENT
                           else W.LAYOUT_NHD, li, 0, heads, hb) for li, r in enumerate(ref)]
    po = [0]
    for tb in tables:
        po.append(po[-1] + len(tb))
    reqs = OracleRequests(po, [0] * len(lengths), lengths, [b for tb in tables for b in tb])
    exp, _ = c_form(ocaches, bs, reqs)
    got = sums.cpu().numpy().view(np.uint64)
    for q, blk in enumerate(reqs.block_ids):
        assert got[blk] == np.uint64(exp[q]), (seed, q, blk)
    for blk in set(range(nb)) - set(reqs.block_ids):
        assert got[blk] == 0, (seed, blk)


@pytest.mark.parametrize("block", range(6))
def test_random_writes_match_scatter_and_oracle(block):
    for seed in range(block * 20, (block + 1) * 20):
        _run_case(seed)
