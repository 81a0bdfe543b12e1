"""Mamba state checksums on the GPU through the C ABI, bit-exact against
the oracle: SSM rows staged by the bulk kernel, conv rows of 6 bytes read
by the generic kernel, both in one call, whole-position and split modes."""

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def check(wl, kernel=None):
    from gpu_helpers import full_oracle, gpu_checksums
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    if kernel is not None:
        assert plan["kernel"] == kernel, plan
    got, st = gpu_checksums(wl)
    exp, est = full_oracle(wl)
    assert st == est == 0
    assert np.array_equal(got, exp)
    return got


def small(seed=0, **kw):
    args = dict(num_requests=5, layers=3, ssm_heads=6, head_dim=8, d_state=16,
                conv_dim=50, conv_width=4)
    args.update(kw)
    return W.mamba2(seed, DEV, **args)


def only(wl, pb):
    return W.Workload(wl.name, wl.block_size, [c for c in wl.caches if c.piece_bytes == pb],
                      wl.pos_offsets, wl.first_position, wl.num_tokens, wl.block_ids,
                      wl.info)


def test_mixed_ssm_and_conv_states():
    got = check(small(), kernel=2)
    assert np.count_nonzero(got) == got.size


def test_ssm_rows_bulk_kernel():
    check(only(small(1), 4), kernel=0)
    # 2-byte elements staged by the bulk kernel: 16-byte conv rows
    wl = small(2, conv_width=9)          # 8 bf16 values = 16 B rows
    check(only(wl, 2), kernel=0)


def test_conv_rows_generic_kernel():
    check(only(small(3), 2), kernel=1)


def test_whole_position_mode_and_the_position_rule():
    # 304 requests: whole positions per CTA
    wl = small(4, num_requests=304, layers=2, conv_width=9)
    check(wl, kernel=0)
    # two positions per request, the state block at position 0 only; a
    # request listed from position 1 has no state
    wl = small(5, num_requests=4, positions_per_request=2, first_positions=[0, 1, 0, 1])
    got = check(wl)
    assert got[1] == got[2] == got[3] == got[5] == got[6] == got[7] == 0
    assert got[0] != 0 and got[4] != 0


@pytest.mark.parametrize("row,pb,rows", [
    (6, 2, 64), (6, 2, 8), (2, 2, 40), (12, 4, 4), (20, 4, 36), (62, 2, 24), (4, 4, 100),
    (6, 2, 50), (12, 4, 5), (10, 2, 7), (6, 2, 4096), (12, 4, 2048)])
def test_short_state_rows_generic_kernel(row, pb, rows):
    """Short rows in the generic kernel: blocks whose size is a multiple of
    16 bytes are read as flat 16-byte chunks, others one row per thread."""
    g = torch.Generator(device=DEV).manual_seed(row * 1000 + rows)
    base = small(8, num_requests=5)
    nb = base.caches[0].num_blocks
    caches = [W.CacheSpec(W.fill_bytes(nb * rows * row, W.BITS16, g, torch.device(DEV)), nb,
                          W.LAYOUT_STATE, li, 5, rows, row, piece_bytes=pb) for li in range(3)]
    wl = W.Workload("short", 16, caches, base.pos_offsets, base.first_position,
                    base.num_tokens, base.block_ids)
    check(wl, kernel=1)


def test_unknown_split_is_one_row_per_shard():
    # a whole shard's state (here 96 KiB) as a single row
    g = torch.Generator(device=DEV).manual_seed(6)
    nb, row = 6, 96 * 1024
    caches = [W.CacheSpec(W.fill_bytes(nb * row, W.BITS16, g, torch.device(DEV)), nb,
                          W.LAYOUT_STATE, li, 3, 1, row, piece_bytes=4) for li in range(2)]
    base = small(7, num_requests=4)
    wl = W.Workload("shard", 16, caches, base.pos_offsets, base.first_position,
                    base.num_tokens, base.block_ids)
    check(wl, kernel=1)
