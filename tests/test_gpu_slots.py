"""The valid-slot kernel (calls of at most two positions per request over
latent or HND caches, or NHD caches of pages up to 8 KiB: the newest block
of each request, and the like):
every position against the oracle (one exact value per block position:
module docstring item 2 of the checksum page), in its fixed and dynamic
share-outs, with replica-key columns and accumulating calls, bad block ids,
skipped positions, more caches than one launch holds, NHD caches of the
same call on the bulk kernel, and positions whose t P passes 2^64."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _newest(seed, n, bs, full_share=0.0, one_token=False, kmax=200):
    """``n`` requests listing only their newest block: lengths bs k + nv,
    nv uniform in [1, bs - 1] (1 with ``one_token``; bs for a share of
    them), k uniform in [0, kmax]."""
    g = torch.Generator().manual_seed(seed)
    ks = torch.randint(0, kmax + 1, (n,), generator=g).tolist()
    nvs = [1] * n if one_token else torch.randint(1, bs, (n,), generator=g).tolist()
    full = (torch.rand(n, generator=g) < full_share).tolist()
    return [k * bs + (bs if f else nv) for k, nv, f in zip(ks, nvs, full)], ks


def _plan(wl, **kw):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return K.plan_for(wl.caches, wl.block_size, wl.num_positions, num_sms=sms,
                      num_requests=wl.num_requests, **kw)


def _check(wl, workspace=False, exp=None):
    from gpu_helpers import full_oracle
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((wl.num_positions,), -1, dtype=torch.int64, device=DEV)
    ws = (torch.full((K.KVCS_WORKSPACE_WORDS,), -1, dtype=torch.int64, device=DEV)
          if workspace else None)
    K.workload_checksummer(wl, workspace=ws)(out, status)
    torch.cuda.synchronize()
    if exp is None:
        exp, st = full_oracle(wl)
        assert st == 0
    got = out.cpu().numpy().view(np.uint64)
    bad = np.flatnonzero(got != np.asarray(exp).reshape(-1))
    assert bad.size == 0, f"{bad.size} of {got.size} positions differ, first {bad[:8].tolist()}"
    return int(status.item()), exp


# (layout, layers, heads, head_bytes, block_size, requests, one token, full share)
CASES = {
    "hnd_8b": (W.LAYOUT_HND, 6, 8, 256, 16, 400, False, 0.1),
    "hnd_8b_one_token": (W.LAYOUT_HND, 6, 8, 256, 16, 400, True, 0.0),
    "hnd_fp8_one_head": (W.LAYOUT_HND, 10, 1, 128, 32, 300, False, 0.2),
    "hnd_3_heads_48": (W.LAYOUT_HND, 4, 3, 48, 16, 250, False, 0.0),
    "latent_mla": (W.LAYOUT_LATENT, 5, 1, 1152, 64, 150, False, 0.1),
    "latent_mla_one_token": (W.LAYOUT_LATENT, 7, 1, 1152, 64, 150, True, 0.0),
    "latent_odd_row": (W.LAYOUT_LATENT, 9, 1, 80, 8, 333, False, 0.0),
    "hnd_block_1": (W.LAYOUT_HND, 3, 4, 64, 1, 200, False, 1.0),
    "few_positions": (W.LAYOUT_HND, 16, 8, 256, 16, 3, False, 0.0),
    "nhd_8k_pages": (W.LAYOUT_NHD, 6, 8, 128, 8, 300, False, 0.1),
    "nhd_8k_pages_one_token": (W.LAYOUT_NHD, 6, 8, 256, 4, 300, True, 0.0),
    "nhd_4k_pages_3_heads": (W.LAYOUT_NHD, 5, 3, 80, 16, 200, False, 0.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("workspace", [False, True])
def test_newest_blocks_match_oracle(case, workspace):
    layout, layers, heads, hb, bs, n, one, full = CASES[case]
    if bs == 1:
        lengths, first = [k + 1 for k in range(n)], list(range(n))
    else:
        lengths, first = _newest(sorted(CASES).index(case), n, bs, full, one)
    wl = W.random_case(31, DEV, layout=layout, layers=layers, heads=heads, head_bytes=hb,
                       block_size=bs, lengths=lengths, first_positions=first)
    plan = _plan(wl)
    assert plan["kernel"] == 3 and plan["slot_launches"] == 1
    st, _ = _check(wl, workspace)
    assert st == 0


@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_LATENT])
def test_dynamic_share_out(layout):
    """A call large enough for the dynamic share-out (64 pages a warp and a
    workspace): the same words with and without the workspace, twice in a
    row on the same workspace, every position against the oracle."""
    if layout == W.LAYOUT_HND:
        lengths, first = _newest(5, 2600, 16, kmax=60)
        wl = W.random_case(41, DEV, layout=layout, layers=32, heads=8, head_bytes=64,
                           block_size=16, lengths=lengths, first_positions=first)
    else:
        lengths, first = _newest(6, 2800, 64, kmax=8)
        wl = W.random_case(42, DEV, layout=layout, layers=61, heads=1, head_bytes=144,
                           block_size=64, lengths=lengths, first_positions=first)
    assert _plan(wl)["kernel"] == 3 and _plan(wl)["dynamic"] == 1
    _, exp = _check(wl, workspace=False)
    ws = torch.zeros(K.KVCS_WORKSPACE_WORDS, dtype=torch.int64, device=DEV)
    outs = [torch.empty(wl.num_positions, dtype=torch.int64, device=DEV) for _ in range(2)]
    ck = K.workload_checksummer(wl, workspace=ws)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for o in outs:
        ck(o, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for o in outs:
        assert np.array_equal(o.cpu().numpy().view(np.uint64), np.asarray(exp).reshape(-1))
    del wl
    torch.cuda.empty_cache()


def test_columns_and_accumulate():
    """Replica-key columns (caches alternate between three columns, sorted
    by the library) and an accumulating call made twice: each column is the
    oracle's checksum over its caches, twice, mod 2^64."""
    from gpu_helpers import full_oracle
    lengths, first = _newest(7, 180, 16)
    wl = W.random_case(43, DEV, layout=W.LAYOUT_HND, layers=9, heads=4, head_bytes=128,
                       block_size=16, lengths=lengths, first_positions=first)
    cols = 3
    caches = [dataclasses.replace(c, column=i % cols) for i, c in enumerate(wl.caches)]
    vals = torch.zeros((wl.num_positions, cols), dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        K.group_checksums(caches, wl.block_size, wl.pos_offsets, wl.first_position,
                          wl.num_tokens, wl.block_ids, cols, values=vals, accumulate=True,
                          total_positions=wl.num_positions, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = vals.cpu().numpy().view(np.uint64)
    for c in range(cols):
        sub = W.Workload(wl.name, wl.block_size, [x for i, x in enumerate(wl.caches)
                                                  if i % cols == c],
                         wl.pos_offsets, wl.first_position, wl.num_tokens, wl.block_ids,
                         wl.info)
        exp, est = full_oracle(sub)
        assert est == 0
        assert np.array_equal(got[:, c], np.asarray(exp).reshape(-1) * np.uint64(2)), c


def test_bad_block_ids_and_skipped_positions():
    """A block id past the pools flags KVCS_STATUS_BAD_BLOCK_ID and its
    position reads 0; positions past a request's tokens read 0; the rest
    equal the oracle's."""
    from gpu_helpers import full_oracle
    g = torch.Generator().manual_seed(8)
    n = 120
    ks = torch.randint(1, 50, (n,), generator=g).tolist()
    nvs = torch.randint(1, 16, (n,), generator=g).tolist()
    lengths = [16 * k + nv for k, nv in zip(ks, nvs)]
    extra = [1 if i % 4 == 0 else 0 for i in range(n)]   # one position past the tokens
    wl = W.random_case(44, DEV, layout=W.LAYOUT_HND, layers=4, heads=8, head_bytes=64,
                       block_size=16, lengths=lengths, first_positions=ks,
                       extra_positions=extra)
    assert wl.num_positions <= 2 * n and _plan(wl)["kernel"] == 3
    exp, est = full_oracle(wl)
    assert est == 0
    exp = np.asarray(exp).reshape(-1).copy()
    assert (exp == 0).sum() >= sum(extra)
    bad = [3, 77]
    ids = wl.block_ids.clone()
    for b in bad:
        ids[b] = wl.caches[0].num_blocks + 5
        exp[b] = 0
    wl2 = dataclasses.replace(wl, block_ids=ids)
    st, _ = _check(wl2, exp=exp)
    assert st & K.KVCS_STATUS_BAD_BLOCK_ID
    assert not st & K.KVCS_STATUS_BAD_REQUESTS


def test_more_caches_than_one_launch():
    """130 latent caches: two valid-slot launches adding into one output."""
    lengths, first = _newest(9, 60, 8)
    wl = W.random_case(45, DEV, layout=W.LAYOUT_LATENT, layers=130, heads=1, head_bytes=64,
                       block_size=8, lengths=lengths, first_positions=first)
    plan = _plan(wl)
    assert plan["slot_launches"] == 2 and plan["memsets"] == 1
    st, _ = _check(wl)
    assert st == 0


def test_mixed_with_nhd_caches():
    """HND and NHD caches of other layers in one call: the HND caches on the
    valid-slot kernel, the NHD ones on the bulk kernel, both adding into the
    same zeroed output."""
    lengths, first = _newest(10, 200, 16)
    a = W.random_case(46, DEV, layout=W.LAYOUT_HND, layers=3, heads=8, head_bytes=128,
                      block_size=16, lengths=lengths, first_positions=first)
    b = W.random_case(46, DEV, layout=W.LAYOUT_NHD, layers=3, heads=8, head_bytes=128,
                      block_size=16, lengths=lengths, first_positions=first,
                      layer_numbers=[10, 11, 12])
    assert torch.equal(a.block_ids, b.block_ids)
    wl = W.Workload("mixed", 16, list(a.caches) + list(b.caches), a.pos_offsets,
                    a.first_position, a.num_tokens, a.block_ids, a.info)
    plan = _plan(wl)
    assert plan["slot_launches"] == 1 and plan["launches"] == 2 and plan["kernel"] != 3
    st, _ = _check(wl, workspace=True)
    assert st == 0


def test_far_positions_wrap():
    """Block positions near 2^57 (t P past 2^64): every product mod 2^64."""
    far = 1 << 57
    n = 40
    g = torch.Generator().manual_seed(11)
    nvs = torch.randint(1, 16, (n,), generator=g).tolist()
    firsts = [far + i for i in range(n)]
    lengths = [16 * f + nv for f, nv in zip(firsts, nvs)]
    wl = W.random_case(47, DEV, layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=64,
                       block_size=16, lengths=lengths, first_positions=firsts)
    assert _plan(wl)["kernel"] == 3
    st, _ = _check(wl)
    assert st == 0


def _random_call(seed):
    """One random call of mostly partial blocks over latent or HND caches:
    its workload (columns assigned), the number of columns, whether it
    accumulates and whether it passes a workspace."""
    g = torch.Generator().manual_seed(seed)

    def pick(xs):
        return xs[int(torch.randint(0, len(xs), (1,), generator=g))]

    layout = pick([W.LAYOUT_HND, W.LAYOUT_LATENT, W.LAYOUT_NHD])
    bs = pick([1, 2, 4, 8, 16, 32, 64])
    if layout == W.LAYOUT_LATENT:
        heads, hb = 1, pick([16, 48, 80, 576, 1152])
    elif layout == W.LAYOUT_NHD:
        # pages of at most 8 KiB (larger NHD pages stay on the bulk kernel)
        heads, hb, bs = pick([(8, 128, 8), (2, 128, 16), (8, 256, 4), (1, 64, 64),
                              (4, 32, 16), (3, 48, 8), (1, 16, 1)])
    else:
        heads, hb = pick([1, 2, 3, 4, 8]), pick([16, 32, 48, 128, 256])
    layers = pick([1, 2, 5, 8])
    n = pick([1, 2, 7, 40, 150, 600])
    shape = pick(["one_token", "random", "some_full", "two_positions"])
    lengths, first, extra = [], [], []
    for _ in range(n):
        k = int(torch.randint(0, 100, (1,), generator=g))
        if shape == "one_token" or bs == 1:
            nv = 1
        elif shape == "some_full" and float(torch.rand(1, generator=g)) < 0.3:
            nv = bs
        else:
            nv = int(torch.randint(1, bs, (1,), generator=g))
        lengths.append(k * bs + nv)
        if shape == "two_positions" and k > 0:
            first.append(k - 1)                 # the last full block and the newest
        else:
            first.append(k)
        extra.append(1 if shape == "two_positions" and k == 0 else 0)
    wl = W.random_case(2000 + seed, DEV, layout=layout, layers=layers, heads=heads,
                       head_bytes=hb, block_size=bs, lengths=lengths, first_positions=first,
                       extra_positions=extra)
    cols = pick([1, 1, 2, 3]) if layers >= 3 else 1
    caches = [dataclasses.replace(c, column=i % cols) for i, c in enumerate(wl.caches)]
    wl = dataclasses.replace(wl, caches=caches)
    return wl, cols, pick([False, True]), pick([False, True])


@pytest.mark.parametrize("block", range(6))
def test_random_calls_match_oracle(block):
    from gpu_helpers import full_oracle
    for seed in range(block * 20, (block + 1) * 20):
        wl, cols, accumulate, workspace = _random_call(seed)
        assert wl.num_positions <= 2 * wl.num_requests
        assert _plan(wl)["slot_launches"] >= 1, seed
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
        got = vals.cpu().numpy().view(np.uint64)
        for c in range(cols):
            sub = dataclasses.replace(wl, caches=[x for x in wl.caches if x.column == c])
            exp, est = full_oracle(sub)
            assert est == 0
            want = np.asarray(exp).reshape(-1) * np.uint64(calls)
            bad = np.flatnonzero(got[:, c] != want)
            assert bad.size == 0, (seed, c, bad.size, bad[:6].tolist())
