"""The full-size workloads in the launch configuration the benchmark times
(one call over every cache and request): sampled positions against the
oracle, plus properties that hold at any size."""

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sample(wl, n=48, seed=0):
    g = np.random.default_rng(seed)
    P = wl.num_positions
    po = wl.pos_offsets.cpu().numpy()
    last = po[1:] - 1                       # partial last blocks
    pick = set(g.choice(P, size=min(n, P), replace=False).tolist())
    pick |= set(last[:8].tolist()) | {0, P - 1}
    return sorted(pick)


def _check(wl, n=48):
    from gpu_helpers import gpu_checksums, oracle_sampled
    got, st = gpu_checksums(wl)
    assert st == 0
    pos, exp, est = oracle_sampled(wl, _sample(wl, n))
    assert est == 0
    assert np.array_equal(got[pos], exp)
    return got


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_llama3_8b_full():
    wl = W.llama3_8b(0, DEV)
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0 and plan["launches"] == 1
    got = _check(wl)
    assert np.count_nonzero(got) == got.size
    del wl
    _free()


def test_mla_full():
    wl = W.mla(0, DEV)
    _check(wl, n=24)
    del wl
    _free()


def test_llama3_70b_full_and_sweep():
    wl = W.llama3_70b(0, DEV)
    from gpu_helpers import gpu_checksums
    full = _check(wl, n=24)
    # request-count sweep: the first n requests alone give the same values
    for n in (1, 2, 8, 32):
        sub = W.Workload(wl.name, wl.block_size, wl.caches, wl.pos_offsets[:n + 1],
                         wl.first_position[:n], wl.num_tokens[:n],
                         wl.block_ids[:int(wl.pos_offsets[n])])
        got, st = gpu_checksums(sub)
        assert st == 0
        assert np.array_equal(got, full[:got.size])
    del wl
    _free()


def test_invariance_full():
    """16 requests of 3000 tokens, 8B-shaped: producer bs16 NHD, consumer
    bs64 HND, two TP shards; per-token-range sums match bit for bit."""
    from gpu_helpers import gpu_checksums, oracle_sampled
    prod, cons, s0, s1 = W.invariance(0, DEV)
    a, _ = gpu_checksums(prod)
    b, _ = gpu_checksums(cons)
    c0, _ = gpu_checksums(s0)
    c1, _ = gpu_checksums(s1)
    assert np.array_equal(c0 + c1, a)
    pa = a.reshape(16, 188)
    pb = b.reshape(16, 47)
    sums = np.add.reduceat(pa, np.arange(0, 188, 4), axis=1, dtype=np.uint64)
    assert np.array_equal(sums, pb)
    pos, exp, _ = oracle_sampled(cons, list(range(0, 752, 37)) + [46, 751])
    assert np.array_equal(b[pos], exp)
    del prod, cons, s0, s1
    _free()


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_fused_write_full_size(kind):
    """The benchmark's write steps (32 layers; 32 x 512 new tokens, or 256
    requests x 1 token) through the prepared call it times: every written
    block's running word equals a checksum pass over the written pools, and
    sampled blocks equal the oracle."""
    from gpu_helpers import oracle_sampled
    wb = W.llama3_8b_write(0, DEV, kind=kind)
    sums = torch.zeros(wb.num_blocks, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.KVWriter(wb.caches, wb.block_size, wb.keys, wb.values, wb.slot_mapping, wb.positions,
               block_sums=sums, status=status)()
    wl = wb.checksum_workload()
    npos = int(wb.block_ids.numel())
    out = torch.empty(npos, dtype=torch.int64, device=DEV)
    K.Checksummer(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position, wl.num_tokens,
                  wl.block_ids, npos)(out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ids = wb.block_ids.long()
    words = sums[ids]
    assert torch.equal(words, out)
    pos, exp, _ = oracle_sampled(wl, _sample(wl, 24))
    assert np.array_equal(words.cpu().numpy().view(np.uint64)[pos], exp)
    del wb, wl
    _free()
