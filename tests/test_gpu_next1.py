"""Replica-key columns, offload row sums, block tags and the fused verify,
on the GPU through the C ABI, bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from helpers import W, c_form, oracle_caches, oracle_requests
from oracle import kvcs_oracle as O
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def _columns_case(seed, layers=6, lengths=(70, 33, 5), cols=(0, 1, 2, 0, 1, 2),
                  **kw):
    wl = W.random_case(seed, DEV, layers=layers, heads=2, head_bytes=kw.pop("hb", 64),
                       block_size=kw.pop("bs", 16), lengths=lengths, **kw)
    for c, k in zip(wl.caches, cols):
        c.column = k
    return wl


def _oracle_values(wl, ncols):
    caches = oracle_caches(wl.caches)
    reqs = oracle_requests(wl)
    out = np.zeros((wl.num_positions, ncols), dtype=np.uint64)
    for k in range(ncols):
        sub = [c for c, s in zip(caches, wl.caches) if s.column == k]
        out[:, k] = np.array(c_form(sub, wl.block_size, reqs)[0], dtype=np.uint64)
    return out


def _group(wl, ncols, **kw):
    return K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                             wl.num_tokens, wl.block_ids, ncols,
                             total_positions=wl.num_positions, **kw)


@pytest.mark.parametrize("mode", ["split", "whole", "generic", "consecutive"])
def test_columns_match_oracle(mode):
    if mode == "whole":      # 304 positions: whole positions per CTA
        wl = _columns_case(1, lengths=[32] * 152, hb=16, bs=16)
    elif mode == "generic":  # 24-byte heads: generic kernel
        wl = _columns_case(2, hb=24)
    elif mode == "consecutive":   # two columns of three consecutive layers
        wl = _columns_case(3, cols=(0, 0, 0, 1, 1, 1), hb=32, bs=8)
    else:
        wl = _columns_case(4)
    values = _group(wl, 3 if mode != "consecutive" else 2)
    torch.cuda.synchronize()
    ncols = values.shape[1]
    exp = _oracle_values(wl, ncols)
    assert np.array_equal(u64(values).reshape(-1, ncols), exp)
    # the row sums are the single-column checksum over every cache
    import dataclasses
    one = W.Workload(wl.name, wl.block_size,
                     [dataclasses.replace(c, column=0) for c in wl.caches],
                     wl.pos_offsets, wl.first_position, wl.num_tokens, wl.block_ids)
    full = K.workload_checksums(one)
    torch.cuda.synchronize()
    assert np.array_equal(exp.sum(axis=1, dtype=np.uint64), u64(full))


def test_columns_over_several_launches():
    wl = _columns_case(5, layers=200, cols=[i % 3 for i in range(200)], hb=16, bs=4,
                       lengths=(9, 4))
    values = _group(wl, 3)
    torch.cuda.synchronize()
    assert np.array_equal(u64(values).reshape(-1, 3), _oracle_values(wl, 3))


def test_tags_match_oracle():
    g = torch.Generator(device=DEV).manual_seed(7)
    hashes = torch.randint(0, 256, (1000, 32), dtype=torch.uint8, device=DEV, generator=g)
    fp = 0x9E3779B97F4A7C15
    tags = K.block_checksum_tags(hashes, fp)
    torch.cuda.synchronize()
    exp = O.block_checksum_tags([bytes(r) for r in hashes.cpu().numpy()], fp)
    assert u64(tags).tolist() == exp
    # a strided view (every other 64-byte record) works too
    wide = torch.randint(0, 256, (50, 64), dtype=torch.uint8, device=DEV, generator=g)
    t2 = K.block_checksum_tags(wide[:, :40], 3)
    torch.cuda.synchronize()
    assert u64(t2).tolist() == O.block_checksum_tags(
        [bytes(r[:40]) for r in wide.cpu().numpy()], 3)


def test_verify_detects_moved_blocks_and_changed_bytes():
    wl = _columns_case(6, lengths=(170, 133, 50))
    assert wl.num_positions == 24
    n = wl.num_positions
    g = torch.Generator(device=DEV).manual_seed(8)
    hashes = torch.randint(0, 256, (n, 32), dtype=torch.uint8, device=DEV, generator=g)
    tags = K.block_checksum_tags(hashes, 0x1234)
    # offload: the tagged row sums are stored with the KV
    stored = torch.empty(n, dtype=torch.int64, device=DEV)
    _group(wl, 3, row_sums=stored, tags=tags)
    torch.cuda.synchronize()
    exp_rows = O.row_sums(_oracle_values(wl, 3).tolist(),
                          O.block_checksum_tags([bytes(r) for r in hashes.cpu().numpy()],
                                                0x1234))
    assert u64(stored).tolist() == exp_rows

    def check():
        mm = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
        cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
        _group(wl, 3, tags=tags, expected=stored, mismatch=mm, mismatch_count=cnt)
        torch.cuda.synchronize()
        return mm.cpu().numpy(), int(cnt.item())

    mm, cnt = check()
    assert cnt == 0 and not mm.any()
    # load two blocks into each other's positions
    ids = wl.block_ids.clone()
    wl.block_ids[[3, 10]] = ids[[10, 3]]
    mm, cnt = check()
    assert cnt == 2 and mm.nonzero()[0].tolist() == [3, 10]
    wl.block_ids.copy_(ids)
    # one changed byte in one layer's K of one block
    blk = int(ids[20])
    c = wl.caches[4]
    view = c.pool.view(2, c.num_blocks, wl.block_size, c.num_heads, c.head_bytes)
    view[0, blk, 0, 1, 5] ^= 0x40
    mm, cnt = check()
    assert cnt == 1 and mm.nonzero()[0].tolist() == [20]


@pytest.mark.parametrize("layout,kbs", [(W.LAYOUT_HND, 0), (W.LAYOUT_HND, 4),
                                        (W.LAYOUT_XSPLIT, 0), (W.LAYOUT_LATENT, 0)])
def test_columns_in_every_layout(layout, kbs):
    """Replica-key columns of HND (with and without kernel sub-blocks),
    x-split and latent caches, against the oracle reading those layouts."""
    import dataclasses
    hb = 96 if layout == W.LAYOUT_LATENT else 64
    wl = W.random_case(7, DEV, layout=layout, layers=4, heads=2, head_bytes=hb, block_size=16,
                       lengths=(70, 33, 5))
    caches = [dataclasses.replace(c, column=i % 2, kernel_block_size=kbs)
              for i, c in enumerate(wl.caches)]
    wl = W.Workload(wl.name, wl.block_size, caches, wl.pos_offsets, wl.first_position,
                    wl.num_tokens, wl.block_ids)
    values = _group(wl, 2)
    torch.cuda.synchronize()
    assert np.array_equal(u64(values).reshape(-1, 2), _oracle_values(wl, 2))
