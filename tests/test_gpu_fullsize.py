"""The full-size workloads in the launch configuration the benchmark times
(one call over every cache and request), compared with the oracle at every
block position: one exact 64-bit value per position (page
"vllm.distributed.kv_transfer.kv_checksum.checksum", module docstring
item 2), so the whole output must be equal bit for bit."""

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_all(wl, workspace=False):
    """Library output of one call over ``wl`` equals the oracle at every
    position; returns the output.  With ``workspace`` the call passes one
    (the benchmark's launch configuration: the dynamic share-out)."""
    from gpu_helpers import gpu_checksums, oracle_every_position
    if workspace:
        ws = torch.zeros(K.KVCS_WORKSPACE_WORDS, dtype=torch.int64, device=DEV)
        out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        K.workload_checksummer(wl, workspace=ws)(out, status)
        torch.cuda.synchronize()
        got, st = out.cpu().numpy().view(np.uint64), int(status.item())
    else:
        got, st = gpu_checksums(wl)
    assert st == 0
    exp, est = oracle_every_position(wl)
    assert est == 0
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, f"{bad.size} of {got.size} positions differ, first {bad[:8].tolist()}"
    return got


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_llama3_8b_full():
    wl = W.llama3_8b(0, DEV)
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0 and plan["launches"] == 1
    got = _check_all(wl)
    assert np.count_nonzero(got) == got.size
    del wl
    _free()


@pytest.mark.parametrize("seed", [1, 2])
def test_llama3_8b_full_other_seeds(seed):
    """The 8B-shaped workload's other two seeds (other lengths, block ids and
    values), in the benchmark's launch configuration."""
    wl = W.llama3_8b(seed, DEV)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert K.plan_for(wl.caches, wl.block_size, wl.num_positions, num_sms=sms)["dynamic"] == 1
    got = _check_all(wl, workspace=True)
    assert np.count_nonzero(got) == got.size
    del wl
    _free()


@pytest.mark.parametrize("name", ["mla", "llama3_70b"])
def test_dynamic_share_out_full(name):
    """MLA and 70B at full size as the benchmark times them (with a
    workspace: the dynamic share-out), every position against the oracle."""
    wl = W.mla(0, DEV) if name == "mla" else W.llama3_70b(0, DEV)
    _check_all(wl, workspace=True)
    del wl
    _free()


def test_mla_full():
    wl = W.mla(0, DEV)
    _check_all(wl)
    del wl
    _free()


def test_llama3_70b_full_and_sweep():
    """Every position of the 43 GB workload, and the request-count sweep
    (the first n requests alone, in the launch mode the sweep times: split
    at unit granularity for few requests) equal to the prefix of the
    oracle-checked full result."""
    wl = W.llama3_70b(0, DEV)
    from gpu_helpers import gpu_checksums
    full = _check_all(wl)
    for n in (1, 2, 4, 8, 16, 32, 64):
        sub = W.Workload(wl.name, wl.block_size, wl.caches, wl.pos_offsets[:n + 1],
                         wl.first_position[:n], wl.num_tokens[:n],
                         wl.block_ids[:int(wl.pos_offsets[n])])
        got, st = gpu_checksums(sub)
        assert st == 0
        assert np.array_equal(got, full[:got.size]), n
    del wl
    _free()


def test_invariance_full():
    """16 requests of 3000 tokens, 8B-shaped: producer bs16 NHD, consumer
    bs64 HND, two TP shards.  Each variant equals the oracle at every
    position, and per-token-range sums match bit for bit."""
    from gpu_helpers import gpu_checksums
    prod, cons, s0, s1 = W.invariance(0, DEV)
    a = _check_all(prod)
    b = _check_all(cons)
    c0 = _check_all(s0)
    c1 = _check_all(s1)
    assert np.array_equal(c0 + c1, a)
    pa = a.reshape(16, 188)
    pb = b.reshape(16, 47)
    sums = np.add.reduceat(pa, np.arange(0, 188, 4), axis=1, dtype=np.uint64)
    assert np.array_equal(sums, pb)
    del prod, cons, s0, s1
    _free()


def test_mamba2_full():
    """The Mamba2-shaped states (SSM rows on the bulk kernel, conv rows on
    the generic kernel, one call), every position against the oracle."""
    wl = W.mamba2(0, DEV, num_requests=64)
    _check_all(wl)
    del wl
    _free()


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_fused_write_full_size(kind):
    """The benchmark's write steps (32 layers; 32 x 512 new tokens, or 256
    requests x 1 token) through the prepared call it times: every written
    block's running word equals a checksum pass over the written pools and
    the oracle over the written pages."""
    from gpu_helpers import oracle_every_position
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
    exp, est = oracle_every_position(wl)
    assert est == 0
    assert np.array_equal(words.cpu().numpy().view(np.uint64), exp)
    del wb, wl
    _free()
