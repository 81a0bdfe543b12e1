"""The KV write fused with the checksum (kvcs_write_kv) through the C ABI:
the written pools equal a plain scatter (data movement with torch), and the
running word of every block equals the oracle's block checksum of the
tokens written to it, for every layout."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W, OracleCache, OracleRequests, c_form, host_bytes
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def to_canonical(c, bs):
    """A pool in its declared layout -> canonical NHD [2, nb, bs, H, hb] (or
    latent [nb, bs, row]) bytes, via torch views."""
    nb, H, hb = c.num_blocks, c.num_heads, c.head_bytes
    if c.layout == W.LAYOUT_LATENT:
        return c.pool.view(nb, bs, hb)
    if c.layout == W.LAYOUT_NHD:
        return c.pool.view(2, nb, bs, H, hb)
    if c.layout == W.LAYOUT_HND:
        kbs = c.kernel_block_size or bs
        v = c.pool.view(2, nb, bs // kbs, H, kbs, hb).permute(0, 1, 2, 4, 3, 5)
        return v.reshape(2, nb, bs, H, hb)
    v = c.pool.view(2, nb, H, hb // 16, bs, 16).permute(0, 1, 4, 2, 3, 5)
    return v.reshape(2, nb, bs, H, hb)


@pytest.mark.parametrize("layout,hb,kbs", [
    (W.LAYOUT_NHD, 64, 0), (W.LAYOUT_NHD, 24, 0), (W.LAYOUT_HND, 64, 0),
    (W.LAYOUT_HND, 32, 4), (W.LAYOUT_XSPLIT, 64, 0), (W.LAYOUT_LATENT, 1152, 0),
    (W.LAYOUT_LATENT, 40, 0)])
def test_write_matches_scatter_and_oracle(layout, hb, kbs):
    bs, layers = 16, 2
    heads = 1 if layout == W.LAYOUT_LATENT else 4
    lengths = [37, 5, 18]
    g = torch.Generator().manual_seed(11)
    nb = 12
    ids = torch.randperm(nb, generator=g)[:sum(-(-n // bs) for n in lengths)].tolist()
    tables, k = [], 0
    for n in lengths:
        tables.append(ids[k:k + -(-n // bs)])
        k += -(-n // bs)
    halves = 1 if layout == W.LAYOUT_LATENT else 2
    caches = [W.CacheSpec(torch.zeros(halves * nb * bs * heads * hb, dtype=torch.uint8,
                                      device=DEV), nb, layout, li, 0, heads, hb,
                          kernel_block_size=kbs) for li in range(layers)]
    ref = [torch.zeros_like(c.pool).view(*to_canonical(c, bs).shape) for c in caches]
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # tokens (request, position), written in three shuffled calls with
    # padding tokens mixed in
    toks = [(r, t) for r, n in enumerate(lengths) for t in range(n)]
    order = torch.randperm(len(toks), generator=g).tolist()
    for part in (order[:20], order[20:45], order[45:]):
        sel = [toks[i] for i in part]
        slots = [tables[r][t // bs] * bs + t % bs for r, t in sel] + [-1, -5]
        pos = [t for _, t in sel] + [3, 0]
        n = len(slots)
        slot_t = torch.tensor(slots, dtype=torch.int64, device=DEV)
        pos_t = torch.tensor(pos, dtype=torch.int64, device=DEV)
        for li, c in enumerate(caches):
            if layout == W.LAYOUT_LATENT:
                key = torch.randint(0, 256, (n, hb), dtype=torch.uint8, generator=g).to(DEV)
                val = None
            else:
                key = torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8,
                                    generator=g).to(DEV)
                val = torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8,
                                    generator=g).to(DEV)
            K.write_kv(c, bs, key, val, slot_t, pos_t, block_sums=sums, status=status)
            for j, s in enumerate(slots):
                if s < 0:
                    continue
                b, o = s // bs, s % bs
                if layout == W.LAYOUT_LATENT:
                    ref[li][b, o] = key[j]
                else:
                    ref[li][0, b, o] = key[j]
                    ref[li][1, b, o] = val[j]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for li, c in enumerate(caches):
        assert torch.equal(to_canonical(c, bs).contiguous(), ref[li].contiguous()), li
    # every written block's running word is the oracle's block checksum
    ocaches = [OracleCache(host_bytes(r), nb, W.LAYOUT_LATENT if layout == W.LAYOUT_LATENT
                           else W.LAYOUT_NHD, li, 0, heads, hb)
               for li, r in enumerate(ref)]
    po = [0]
    for tb in tables:
        po.append(po[-1] + len(tb))
    reqs = OracleRequests(po, [0] * len(lengths), lengths, [b for tb in tables for b in tb])
    exp, _ = c_form(ocaches, bs, reqs)
    got = u64(sums)
    for q, b in enumerate(reqs.block_ids):
        assert got[b] == np.uint64(exp[q]), (q, b)
    unused = set(range(nb)) - set(reqs.block_ids)
    assert all(got[b] == 0 for b in unused)


def test_write_flags_bad_slots_and_positions():
    nb, bs, heads, hb = 4, 8, 2, 32
    c = W.CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8, device=DEV),
                    nb, W.LAYOUT_NHD, 0, 0, heads, hb)
    key = torch.ones((3, heads, hb), dtype=torch.uint8, device=DEV)
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.write_kv(c, bs, key, key.clone(), torch.tensor([nb * bs + 3, 5, 9], device=DEV),
               torch.tensor([0, -2, 1], device=DEV), block_sums=sums, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & K.KVCS_STATUS_BAD_BLOCK_ID
    assert int(st.item()) & K.KVCS_STATUS_BAD_REQUESTS
    # slot 5 (negative position) was written but not summed; slot 9 both
    pool = c.pool.view(2, nb, bs, heads, hb)
    assert int(pool[0, 0, 5].sum()) == heads * hb and int(pool[0, 1, 1].sum()) == heads * hb
    assert int(sums[0].item()) == 0 and int(sums[1].item()) != 0


def test_all_layers_in_one_call_equals_layer_by_layer():
    bs, nb, heads, hb, layers = 16, 20, 8, 256, 5
    g = torch.Generator().manual_seed(21)
    n = 300
    slots = torch.randperm(nb * bs, generator=g)[:n].to(DEV)
    pos = torch.randint(0, 4096, (n,), generator=g).to(DEV)
    keys = [torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
            for _ in range(layers)]
    vals = [torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
            for _ in range(layers)]

    def fresh():
        return [W.CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8,
                                        device=DEV), nb, W.LAYOUT_NHD, li, 0, heads, hb)
                for li in range(layers)]

    a, b = fresh(), fresh()
    sa = torch.zeros(nb, dtype=torch.int64, device=DEV)
    sb = torch.zeros(nb, dtype=torch.int64, device=DEV)
    K.write_kv(a, bs, keys, vals, slots, pos, block_sums=sa)
    for c, k, v in zip(b, keys, vals):
        K.write_kv(c, bs, k, v, slots, pos, block_sums=sb)
    torch.cuda.synchronize()
    assert torch.equal(sa, sb)
    for ca, cb in zip(a, b):
        assert torch.equal(ca.pool, cb.pool)


def _oracle_sums(caches, refs, bs, tables, lengths):
    """Oracle block checksums of the blocks in `tables` from canonical pools."""
    ocaches = []
    for c, r in zip(caches, refs):
        lay = W.LAYOUT_LATENT if c.layout == W.LAYOUT_LATENT else W.LAYOUT_NHD
        ocaches.append(OracleCache(host_bytes(r), c.num_blocks, lay, c.layer, c.head_offset,
                                   c.num_heads, c.head_bytes))
    po = [0]
    for tb in tables:
        po.append(po[-1] + len(tb))
    reqs = OracleRequests(po, [0] * len(lengths), lengths, [b for tb in tables for b in tb])
    exp, _ = c_form(ocaches, bs, reqs)
    return reqs.block_ids, exp


def test_mixed_layouts_in_one_call():
    """NHD, HND in kernel sub-blocks, x-split and latent caches written by one
    call (one launch per layout family) add into the same running words."""
    bs, nb = 16, 10
    specs = [(W.LAYOUT_NHD, 4, 64, 0), (W.LAYOUT_HND, 4, 32, 4), (W.LAYOUT_XSPLIT, 2, 48, 0),
             (W.LAYOUT_LATENT, 1, 72, 0), (W.LAYOUT_NHD, 2, 16, 0)]
    caches = []
    for li, (lay, heads, hb, kbs) in enumerate(specs):
        halves = 1 if lay == W.LAYOUT_LATENT else 2
        caches.append(W.CacheSpec(torch.zeros(halves * nb * bs * heads * hb, dtype=torch.uint8,
                                              device=DEV), nb, lay, li, 0, heads, hb,
                                  kernel_block_size=kbs))
    lengths = [40, 23]
    g = torch.Generator().manual_seed(5)
    ids = torch.randperm(nb, generator=g).tolist()
    tables = [ids[0:3], ids[3:5]]
    sel = [(r, t) for r, n in enumerate(lengths) for t in range(n)]
    slots = torch.tensor([tables[r][t // bs] * bs + t % bs for r, t in sel], device=DEV)
    pos = torch.tensor([t for _, t in sel], device=DEV)
    n = len(sel)
    keys, vals = [], []
    for c in caches:
        if c.layout == W.LAYOUT_LATENT:
            keys.append(torch.randint(0, 256, (n, c.head_bytes), dtype=torch.uint8,
                                      generator=g).to(DEV))
            vals.append(None)
        else:
            keys.append(torch.randint(0, 256, (n, c.num_heads, c.head_bytes), dtype=torch.uint8,
                                      generator=g).to(DEV))
            vals.append(torch.randint(0, 256, (n, c.num_heads, c.head_bytes),
                                      dtype=torch.uint8, generator=g).to(DEV))
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    K.write_kv(caches, bs, keys, vals, slots, pos, block_sums=sums)
    torch.cuda.synchronize()
    refs = [to_canonical(c, bs).contiguous() for c in caches]
    block_ids, exp = _oracle_sums(caches, refs, bs, tables, lengths)
    got = u64(sums)
    for q, b in enumerate(block_ids):
        assert got[b] == np.uint64(exp[q]), (q, b)
    # the written rows landed where the layouts put them
    sl = slots.cpu()
    for c, k, v, r in zip(caches, keys, vals, refs):
        if c.layout == W.LAYOUT_LATENT:
            assert torch.equal(r[sl // bs, sl % bs].cpu(), k.cpu())
        else:
            assert torch.equal(r[0, sl // bs, sl % bs].cpu(), k.cpu())
            assert torch.equal(r[1, sl // bs, sl % bs].cpu(), v.cpu())


def test_more_caches_than_one_launch_holds():
    """70 caches of one family take two launches; the words still add up."""
    bs, nb, layers, hb = 8, 6, 70, 16
    g = torch.Generator().manual_seed(8)
    caches = [W.CacheSpec(torch.zeros(nb * bs * hb, dtype=torch.uint8, device=DEV), nb,
                          W.LAYOUT_LATENT, li, 0, 1, hb) for li in range(layers)]
    lengths = [13]
    tables = [[4, 1]]
    slots = torch.tensor([tables[0][t // bs] * bs + t % bs for t in range(13)], device=DEV)
    pos = torch.arange(13, device=DEV)
    keys = [torch.randint(0, 256, (13, hb), dtype=torch.uint8, generator=g).to(DEV)
            for _ in range(layers)]
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    l0 = K.launch_count()
    K.write_kv(caches, bs, keys, [None] * layers, slots, pos, block_sums=sums)
    torch.cuda.synchronize()
    assert K.launch_count() - l0 == 2
    refs = [to_canonical(c, bs).contiguous() for c in caches]
    block_ids, exp = _oracle_sums(caches, refs, bs, tables, lengths)
    got = u64(sums)
    for q, b in enumerate(block_ids):
        assert got[b] == np.uint64(exp[q]), (q, b)


def test_prepared_writer_matches_write_kv():
    """KVWriter (arguments marshalled once) writes and sums exactly as
    write_kv, for all prepared tokens and for a leading subset."""
    bs, nb, heads, hb, layers, n = 16, 10, 2, 64, 3, 40
    g = torch.Generator().manual_seed(31)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(DEV)
    pos = torch.randint(0, 300, (n,), generator=g).to(DEV)
    keys = [torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
            for _ in range(layers)]
    vals = [torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
            for _ in range(layers)]

    def fresh():
        return [W.CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8,
                                        device=DEV), nb, W.LAYOUT_HND, li, 0, heads, hb)
                for li in range(layers)]

    for count in (n, 17, 0):
        a, b = fresh(), fresh()
        sa = torch.zeros(nb, dtype=torch.int64, device=DEV)
        sb = torch.zeros(nb, dtype=torch.int64, device=DEV)
        K.KVWriter(a, bs, keys, vals, slots, pos, block_sums=sa)(num_tokens=count)
        K.write_kv(b, bs, [k[:count] for k in keys], [v[:count] for v in vals], slots[:count],
                   pos[:count], block_sums=sb)
        torch.cuda.synchronize()
        assert torch.equal(sa, sb)
        for ca, cb in zip(a, b):
            assert torch.equal(ca.pool, cb.pool)


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_XSPLIT, W.LAYOUT_LATENT])
def test_write_far_positions_wrap(layout):
    """Token positions near 2^61 (t P past 2^64): the running word equals
    the oracle's block checksum, all products taken mod 2^64."""
    bs, nb, heads, hb = 16, 3, 2, 64
    if layout == W.LAYOUT_LATENT:
        heads, hb = 1, 96
    far = 1 << 57
    g = torch.Generator().manual_seed(41)
    halves = 1 if layout == W.LAYOUT_LATENT else 2
    c = W.CacheSpec(torch.zeros(halves * nb * bs * heads * hb, dtype=torch.uint8, device=DEV),
                    nb, layout, 3, 0, heads, hb)
    n = 13
    slots = torch.arange(n, device=DEV) + 2 * bs           # block 2, slots 0..12
    pos = torch.arange(n, device=DEV) + far * bs
    key = torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
    val = None if layout == W.LAYOUT_LATENT else \
        torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
    if layout == W.LAYOUT_LATENT:
        key = key.view(n, hb)
    sums = torch.zeros(nb, dtype=torch.int64, device=DEV)
    K.write_kv(c, bs, key, val, slots, pos, block_sums=sums)
    torch.cuda.synchronize()
    canon = to_canonical(c, bs).contiguous()
    oc = OracleCache(host_bytes(canon), nb, W.LAYOUT_LATENT if layout == W.LAYOUT_LATENT
                     else W.LAYOUT_NHD, 3, 0, heads, hb)
    exp, st = c_form([oc], bs, OracleRequests([0, 1], [far], [far * bs + n], [2]))
    assert st == 0
    assert u64(sums)[2] == np.uint64(exp[0])


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_XSPLIT])
def test_write_with_8_byte_aligned_buffers(layout):
    """Key and value buffers 8 bytes off a 16-byte boundary: the write moves
    8-byte pieces, with the same pools and running words as aligned buffers."""
    bs, nb, heads, hb, n = 16, 6, 2, 64, 37
    g = torch.Generator().manual_seed(51)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(DEV)
    pos = torch.randint(0, 2000, (n,), generator=g).to(DEV)
    key = torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)
    val = torch.randint(0, 256, (n, heads, hb), dtype=torch.uint8, generator=g).to(DEV)

    def offset8(t):
        raw = torch.zeros(t.numel() + 8, dtype=torch.uint8, device=DEV)
        raw[8:] = t.reshape(-1)
        return raw[8:].view(t.shape)

    def cache():
        return W.CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8, device=DEV),
                           nb, layout, 1, 0, heads, hb)

    a, b = cache(), cache()
    sa = torch.zeros(nb, dtype=torch.int64, device=DEV)
    sb = torch.zeros(nb, dtype=torch.int64, device=DEV)
    K.write_kv(a, bs, key, val, slots, pos, block_sums=sa)
    k8, v8 = offset8(key), offset8(val)
    assert k8.data_ptr() % 16 == 8
    K.write_kv(b, bs, k8, v8, slots, pos, block_sums=sb)
    torch.cuda.synchronize()
    assert torch.equal(a.pool, b.pool)
    assert torch.equal(sa, sb)
