"""Calls whose blocks are mostly partial (at most two positions per request,
such as the newest block of each request): NHD caches on the bulk kernel's
instance in which the whole producer warp issues a unit's copies and the
consumers reduce a packed unit of many pages at once; latent and HND caches
on the valid-slot kernel.  Each case compares every position with the oracle
(one exact value per block position: module docstring item 2 of the checksum
page)."""

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _newest_blocks(seed, n, block_size, full_share=0.0):
    """``n`` requests that each list only their newest block: lengths
    block_size k + nv with nv uniform in [1, block_size - 1] (a share of
    them full, nv = block_size), k in [0, 200]."""
    g = torch.Generator().manual_seed(seed)
    ks = torch.randint(0, 201, (n,), generator=g).tolist()
    nvs = torch.randint(1, block_size, (n,), generator=g).tolist()
    full = (torch.rand(n, generator=g) < full_share).tolist()
    lengths = [k * block_size + (block_size if f else nv) for k, nv, f in zip(ks, nvs, full)]
    first = [k for k in ks]
    return lengths, first


def _check(wl, workspace=False):
    from gpu_helpers import full_oracle
    assert wl.num_positions <= 2 * wl.num_requests      # the mostly-partial path applies
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    ws = (torch.zeros(K.KVCS_WORKSPACE_WORDS, dtype=torch.int64, device=DEV)
          if workspace else None)
    K.workload_checksummer(wl, workspace=ws)(out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    exp, st = full_oracle(wl)
    assert st == 0
    got = out.cpu().numpy().view(np.uint64)
    bad = np.flatnonzero(got != exp.reshape(-1))
    assert bad.size == 0, f"{bad.size} of {got.size} positions differ, first {bad[:8].tolist()}"


# (layout, layers, heads, head_bytes, block_size, requests, full share)
CASES = {
    "nhd_8b_rows": (W.LAYOUT_NHD, 4, 8, 256, 16, 300, 0.0),
    "hnd_8b_heads": (W.LAYOUT_HND, 4, 8, 256, 16, 300, 0.0),
    "hnd_fp8": (W.LAYOUT_HND, 6, 8, 128, 16, 200, 0.2),
    "latent_mla": (W.LAYOUT_LATENT, 5, 1, 1152, 64, 120, 0.1),
    "nhd_some_full": (W.LAYOUT_NHD, 3, 4, 128, 16, 257, 0.5),
    # 80 pages of 16 valid bytes a position: units of more than 32 pages
    "nhd_tiny_rows": (W.LAYOUT_NHD, 40, 1, 16, 16, 170, 0.0),
    "hnd_one_head": (W.LAYOUT_HND, 12, 1, 64, 32, 90, 0.3),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_newest_blocks_match_oracle(case):
    layout, layers, heads, hb, bs, n, full = CASES[case]
    lengths, first = _newest_blocks(sorted(CASES).index(case), n, bs, full)
    wl = W.random_case(11, DEV, layout=layout, layers=layers, heads=heads, head_bytes=hb,
                       block_size=bs, lengths=lengths, first_positions=first)
    assert wl.num_positions == n
    _check(wl)


def test_two_positions_per_request():
    """Each request lists two positions: its last full block and its
    partial newest one, or (every third request) its newest block and one
    past its tokens (a skipped position, whose checksum is 0)."""
    g = torch.Generator().manual_seed(5)
    n = 150
    ks = torch.randint(1, 100, (n,), generator=g).tolist()
    nvs = torch.randint(1, 16, (n,), generator=g).tolist()
    lengths = [k * 16 + nv for k, nv in zip(ks, nvs)]
    past = [i % 3 == 0 for i in range(n)]
    first = [k if p_ else k - 1 for k, p_ in zip(ks, past)]
    extra = [1 if p_ else 0 for p_ in past]
    for seed, layout in ((6, W.LAYOUT_NHD), (7, W.LAYOUT_HND)):
        wl = W.random_case(seed, DEV, layout=layout, layers=3, heads=8, head_bytes=128,
                           block_size=16, lengths=lengths, first_positions=first,
                           extra_positions=extra)
        assert wl.num_positions == 2 * n
        _check(wl)


def test_few_positions_split():
    """Fewer positions than SMs (ranges cut at unit granularity, zeroed
    output, atomics) on the mostly-partial path."""
    lengths, first = _newest_blocks(21, 40, 16)
    for layout in (W.LAYOUT_NHD, W.LAYOUT_HND):
        wl = W.random_case(8, DEV, layout=layout, layers=16, heads=8, head_bytes=256,
                           block_size=16, lengths=lengths, first_positions=first)
        plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
        assert plan["split"] == 1
        _check(wl)


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND])
def test_decode_with_workspace(layout):
    """The decode-shaped benchmark workload's recipe (one one-token block per
    request, 8B geometry) at 4096 requests, as the benchmark runs it: with a
    workspace (the dynamic share-out applies to its 262,144 units), every
    position against the oracle."""
    wl = W.llama3_8b_decode(0, DEV, num_requests=4096, layout=layout)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert K.plan_for(wl.caches, wl.block_size, wl.num_positions, num_sms=sms)["dynamic"] == 1
    _check(wl, workspace=True)
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND])
def test_accumulating_calls(layout):
    """An accumulating call (every result added into the caller's words)
    through the mostly-partial path, twice onto the same words: twice the
    oracle's checksums, mod 2^64."""
    from gpu_helpers import full_oracle
    lengths, first = _newest_blocks(31, 200, 16)
    wl = W.random_case(12, DEV, layout=layout, layers=4, heads=8, head_bytes=256, block_size=16,
                       lengths=lengths, first_positions=first)
    exp, st = full_oracle(wl)
    assert st == 0
    vals = torch.zeros((wl.num_positions, 1), dtype=torch.int64, device=DEV)
    for _ in range(2):
        K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                          wl.num_tokens, wl.block_ids, 1, values=vals, accumulate=True,
                          total_positions=wl.num_positions)
    torch.cuda.synchronize()
    got = vals.cpu().numpy().view(np.uint64).reshape(-1)
    assert np.array_equal(got, exp.reshape(-1) * np.uint64(2))
