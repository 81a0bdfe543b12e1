"""Accumulating calls (KVCS_OUT_ACCUMULATE) through the C ABI: checksumming
the layers of a workload in groups, each call adding into the same words,
ends with the one-call result and with the oracle's checksums; the words'
earlier contents are kept (added to mod 2^64); a position with a bad block
id adds nothing.  Whole-position and split launches, bulk and generic
kernels are all covered."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
from gpu_helpers import full_oracle
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"
M64 = (1 << 64) - 1


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def checksummer(wl, caches):
    return K.Checksummer(caches, wl.block_size, wl.pos_offsets, wl.first_position,
                         wl.num_tokens, wl.block_ids, wl.num_positions)


def groups_of(caches, sizes):
    out, k = [], 0
    for s in sizes:
        out.append(caches[k:k + s])
        k += s
    assert k == len(caches)
    return out


CASES = {
    # many positions: whole-position bulk launches
    "whole": lambda: W.llama3_8b(seed=3, device=DEV, num_requests=19, min_len=1024,
                                 max_len=1024, layers=6),
    # few positions: split bulk launches
    "split": lambda: W.random_case(4, DEV, layers=5, heads=4, head_bytes=256,
                                   lengths=(70, 33)),
    # head bytes not a multiple of 16: the generic kernel
    "generic": lambda: W.random_case(5, DEV, layers=4, heads=3, head_bytes=24,
                                     lengths=(150, 16, 1)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_groups_add_up_to_the_full_checksum(name):
    wl = CASES[name]()
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    if name == "generic":
        assert plan["kernel"] == 1
    else:
        assert plan["kernel"] == 0 and plan["split"] == (name == "split")
    n = len(wl.caches)
    sizes = [1, n - 3, 2] if n > 3 else [1] * n
    one = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    checksummer(wl, wl.caches)(one)
    acc = torch.zeros(wl.num_positions, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for grp in groups_of(wl.caches, sizes):
        checksummer(wl, grp)(acc, status, accumulate=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(u64(acc), u64(one))
    exp, st = full_oracle(wl)
    assert st == 0
    assert np.array_equal(u64(acc), np.asarray(exp, dtype=np.uint64))


def test_accumulate_keeps_earlier_contents_and_skips_bad_ids():
    wl = W.random_case(6, DEV, layers=3, heads=2, head_bytes=64, lengths=(90, 40))
    g = torch.Generator().manual_seed(9)
    start = torch.randint(-(1 << 62), 1 << 62, (wl.num_positions,), generator=g,
                          dtype=torch.int64)
    # one position points past the pool
    bad = 2
    ids = wl.block_ids.clone()
    ids[bad] = wl.caches[0].num_blocks + 7
    wl_bad = dataclasses.replace(wl, block_ids=ids)
    acc = start.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    checksummer(wl_bad, wl_bad.caches)(acc, status, accumulate=True)
    torch.cuda.synchronize()
    assert int(status.item()) & K.KVCS_STATUS_BAD_BLOCK_ID
    exp, _ = full_oracle(wl_bad)
    want = [(int(s) + int(e)) & M64 for s, e in zip(start.numpy().view(np.uint64), exp)]
    want[bad] = int(start.numpy().view(np.uint64)[bad])
    assert np.array_equal(u64(acc), np.asarray(want, dtype=np.uint64))


def test_group_checksums_accumulate_with_row_sums():
    """Two columns accumulated over two layer groups; the row sums asked for
    on the last call are those of the one-call values."""
    wl = W.random_case(7, DEV, layers=4, heads=2, head_bytes=64, lengths=(64, 50))
    caches = [dataclasses.replace(c, column=i % 2) for i, c in enumerate(wl.caches)]
    args = (wl.block_size, wl.pos_offsets, wl.first_position, wl.num_tokens, wl.block_ids, 2)
    ref_rows = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    ref = K.group_checksums(caches, *args, row_sums=ref_rows,
                            total_positions=wl.num_positions)
    vals = torch.zeros((wl.num_positions, 2), dtype=torch.int64, device=DEV)
    rows = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    K.group_checksums(caches[:2], *args, values=vals, accumulate=True,
                      total_positions=wl.num_positions)
    K.group_checksums(caches[2:], *args, values=vals, row_sums=rows, accumulate=True,
                      total_positions=wl.num_positions)
    torch.cuda.synchronize()
    assert torch.equal(vals, ref)
    assert torch.equal(rows, ref_rows)
