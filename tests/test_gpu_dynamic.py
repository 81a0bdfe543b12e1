"""Calls with a workspace (KVCS_OUT_WORKSPACE): the bulk kernel reads a
fixed share of each launch's units per CTA and hands the rest out in chunks
from a counter in the workspace.  The result is the same exact checksum
(module docstring item 2 of the checksum page: one value per block
position), so every case compares every position with the oracle, or with
the static call where the oracle already checked that."""

import dataclasses

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ws():
    return torch.full((K.KVCS_WORKSPACE_WORDS,), -1, dtype=torch.int64, device=DEV)


def _u(t):
    return t.cpu().numpy().view(np.uint64)


def _dynamic(wl, ws, columns=1, accumulate=False, values=None, status=None):
    vals = K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                             wl.num_tokens, wl.block_ids, columns, values=values,
                             total_positions=wl.num_positions, accumulate=accumulate,
                             workspace=ws, status=status)
    torch.cuda.synchronize()
    return vals


def _oracle(wl):
    from gpu_helpers import full_oracle
    exp, st = full_oracle(wl)
    assert st == 0
    return exp


def _assert_dynamic(wl):
    """The call is large enough for the dynamic share-out (1024 units a SM)."""
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan["units"] >= 1024 * sms
    return plan


def _ragged(seed, n=48, layers=32, **kw):
    g = torch.Generator().manual_seed(seed)
    lengths = torch.randint(1, 4000, (n,), generator=g).tolist()
    args = dict(layers=layers, heads=2, head_bytes=32, block_size=16)
    args.update(kw)
    return W.random_case(seed, DEV, lengths=lengths, **args)


@pytest.mark.parametrize("seed", [0, 1])
def test_dynamic_matches_oracle(seed):
    """Ragged requests (partial last blocks), enough units for the dynamic
    share-out; every position against the oracle."""
    wl = _ragged(seed)
    _assert_dynamic(wl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _u(_dynamic(wl, _ws(), status=status)).reshape(-1)
    assert int(status.item()) == 0
    assert np.array_equal(got, _oracle(wl))


def test_dynamic_packed_pages_and_misaligned_rows():
    """fp8-shaped 16 KiB pages packed three to a stage, and the same pools 8
    bytes off a 16-byte boundary (the misaligned-rows instance)."""
    wl = _ragged(3, n=40, layers=18, heads=8, head_bytes=128)
    _assert_dynamic(wl)
    exp = _oracle(wl)
    assert np.array_equal(_u(_dynamic(wl, _ws())).reshape(-1), exp)
    caches, keep = [], []
    for c in wl.caches:
        raw = torch.zeros(c.pool.numel() + 8, dtype=torch.uint8, device=DEV)
        raw[8:] = c.pool
        keep.append(raw)
        caches.append(dataclasses.replace(c, pool=raw[8:]))
    mis = W.Workload(wl.name, wl.block_size, caches, wl.pos_offsets, wl.first_position,
                     wl.num_tokens, wl.block_ids, wl.info)
    assert np.array_equal(_u(_dynamic(mis, _ws())).reshape(-1), exp)


def test_dynamic_several_launches():
    """Two layout families (NHD and HND: two bulk launches, two counters)
    and a cache the bulk kernel cannot stage (a direct-load launch) in one
    call."""
    wl = _ragged(4, layers=16)
    hnd = _ragged(4, layers=16, layout=W.LAYOUT_HND)
    odd = _ragged(4, layers=1, head_bytes=24)
    caches = (list(wl.caches)
              + [dataclasses.replace(c, layer=c.layer + 16) for c in hnd.caches]
              + [dataclasses.replace(c, layer=99) for c in odd.caches])
    mixed = W.Workload("mixed", wl.block_size, caches, wl.pos_offsets, wl.first_position,
                       wl.num_tokens, wl.block_ids)
    plan = _assert_dynamic(mixed)
    assert plan["kernel"] == 2 and plan["launches"] == 3
    assert np.array_equal(_u(_dynamic(mixed, _ws())).reshape(-1), _oracle(mixed))


def test_dynamic_more_caches_than_a_launch():
    """200 caches of one family: two bulk launches, two counters."""
    wl = _ragged(5, n=24, layers=200, heads=1, head_bytes=16)
    plan = _assert_dynamic(wl)
    assert plan["launches"] == 2
    assert np.array_equal(_u(_dynamic(wl, _ws())).reshape(-1), _oracle(wl))


def test_dynamic_columns_accumulate_and_reuse():
    """Replica columns; an accumulating call (only the counters are zeroed,
    the values keep their contents); the same workspace used by calls back
    to back on one stream."""
    wl = _ragged(6)
    _assert_dynamic(wl)
    exp = _oracle(wl)
    ws = _ws()
    cols = [dataclasses.replace(c, column=i % 2) for i, c in enumerate(wl.caches)]
    cw = W.Workload(wl.name, wl.block_size, cols, wl.pos_offsets, wl.first_position,
                    wl.num_tokens, wl.block_ids, wl.info)
    vals = _dynamic(cw, ws, columns=2)
    v = _u(vals)
    assert np.array_equal(v.sum(axis=1, dtype=np.uint64), exp)
    _dynamic(cw, ws, columns=2, accumulate=True, values=vals)
    assert np.array_equal(_u(vals), v * np.uint64(2))
    # ten calls back to back, no synchronisation between them
    outs = [torch.empty(wl.num_positions, dtype=torch.int64, device=DEV) for _ in range(10)]
    ck = K.workload_checksummer(wl, workspace=ws)
    for o in outs:
        ck(o)
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(_u(o), exp)


def test_dynamic_small_call_stays_static():
    """Below the threshold the workspace is not used: a few positions still
    come out right."""
    wl = W.random_case(7, DEV, layers=2, heads=2, head_bytes=64, block_size=16,
                       lengths=(70, 33, 5))
    assert np.array_equal(_u(_dynamic(wl, _ws())).reshape(-1), _oracle(wl))


def test_dynamic_in_a_cuda_graph():
    """The workspace call captured in a CUDA graph and replayed after the
    pools change equals a direct (static) call."""
    wl = _ragged(8)
    _assert_dynamic(wl)
    ws = _ws()
    ck = K.workload_checksummer(wl, workspace=ws)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ck(out, None, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ck(out, None, s.cuda_stream)
    gen = torch.Generator(device=DEV).manual_seed(977)  # not the fill's own seed
    prev = K.workload_checksums(wl)
    for _ in range(2):
        for c in wl.caches:
            c.pool.copy_(torch.randint(0, 256, c.pool.shape, dtype=torch.uint8, device=DEV,
                                       generator=gen))
        g.replay()
        torch.cuda.synchronize()
        ref = K.workload_checksums(wl)
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and not torch.equal(ref, prev)
        prev = ref


def test_dynamic_full_size_llama3_8b():
    """The benchmark's call: the 8B-shaped workload (10,013 positions, 21 GB)
    through the workspace path, every position against the oracle."""
    from gpu_helpers import oracle_every_position
    wl = W.llama3_8b(0, DEV)
    ws = _ws()
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.workload_checksummer(wl, workspace=ws)(out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    exp, est = oracle_every_position(wl)
    assert est == 0
    assert np.array_equal(_u(out), exp)
    del wl
    torch.cuda.empty_cache()
