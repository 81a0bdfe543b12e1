"""kvcs_block_checksums_noalloc, called through the C ABI, against
kvcs_block_checksums on the same inputs.

The entry point is for callers that cannot allocate device memory: its
scratch (the bulk kernel's work counters) is the library's module-scope
array, shared by every call on a device and left holding the last call's
counters.  So the cases here make two calls in a row on one stream, with no
synchronisation between them, each large enough to use the counters, and
check both results.  The file is collected last and also passes alone in a
fresh process, where its first call is the one that looks the array up."""

import ctypes

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ragged(seed, n, layers, layout=W.LAYOUT_NHD):
    g = torch.Generator().manual_seed(seed)
    lengths = torch.randint(1, 4000, (n,), generator=g).tolist()
    return W.random_case(seed, DEV, lengths=lengths, layers=layers, heads=2, head_bytes=32,
                         block_size=16, layout=layout)


def _abi_args(wl):
    arr = K.cache_array(wl.caches)
    reqs = K.kvcs_requests(wl.num_requests, wl.pos_offsets.data_ptr(),
                           wl.first_position.data_ptr(), wl.num_tokens.data_ptr(),
                           wl.block_ids.data_ptr())
    return arr, reqs


def _noalloc(wl, out, status, stream):
    arr, reqs = _abi_args(wl)
    return K.load_library().kvcs_block_checksums_noalloc(
        arr, len(wl.caches), wl.block_size, ctypes.byref(reqs), wl.num_positions,
        out.data_ptr(), status.data_ptr(), stream)


def _existing(wl, stream):
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    arr, reqs = _abi_args(wl)
    K.kvcs_block_checksums(arr, len(wl.caches), wl.block_size, reqs, wl.num_positions,
                           out.data_ptr(), None, stream)
    return out


def _uses_counters(wl):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions, num_sms=sms)
    return plan["dynamic"] == 1


def test_two_calls_in_a_row_match_block_checksums():
    """Two calls back to back: NHD (5749 positions, ragged) then HND of
    another size (one bulk launch each, both through the shared counters).
    The second call finds the first one's counters in the array."""
    a = _ragged(0, 48, 32)
    b = _ragged(1, 40, 24, layout=W.LAYOUT_HND)
    assert _uses_counters(a) and _uses_counters(b)
    s = torch.cuda.Stream()
    outs = [torch.full((wl.num_positions,), -1, dtype=torch.int64, device=DEV)
            for wl in (a, b)]
    stats = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    for wl, out, st in zip((a, b), outs, stats):
        assert _noalloc(wl, out, st, s.cuda_stream) == K.KVCS_OK
    with torch.cuda.stream(s):
        refs = [_existing(wl, s.cuda_stream) for wl in (a, b)]
    torch.cuda.synchronize()
    for out, ref, st in zip(outs, refs, stats):
        assert int(st.item()) == 0
        assert torch.equal(out, ref)


def test_repeated_calls_on_the_same_workload():
    """The same workload twice in a row into two outputs, and a third time
    after its pools changed: each result equals the existing entry's."""
    wl = _ragged(2, 48, 32)
    assert _uses_counters(wl)
    s = torch.cuda.Stream()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o1 = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    o2 = torch.empty_like(o1)
    torch.cuda.synchronize()
    assert _noalloc(wl, o1, st, s.cuda_stream) == K.KVCS_OK
    assert _noalloc(wl, o2, st, s.cuda_stream) == K.KVCS_OK
    with torch.cuda.stream(s):
        ref = _existing(wl, s.cuda_stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1, ref) and torch.equal(o2, ref)
    gen = torch.Generator(device=DEV).manual_seed(991)  # not the fill's own seed
    for c in wl.caches:
        c.pool.copy_(torch.randint(0, 256, c.pool.shape, dtype=torch.uint8, device=DEV,
                                   generator=gen))
    torch.cuda.synchronize()
    assert _noalloc(wl, o1, st, s.cuda_stream) == K.KVCS_OK
    with torch.cuda.stream(s):
        ref2 = _existing(wl, s.cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(o1, ref2) and not torch.equal(ref2, ref)


def test_two_decode_shaped_calls_in_a_row():
    """The newest block of each of 4096 requests (one valid token each), NHD
    then HND: calls of mostly partial blocks (the wide rows instance, then
    the valid-slot kernel), back to back through the shared counters."""
    calls = [W.llama3_8b_decode(s, DEV, num_requests=4096, layout=lay)
             for s, lay in ((3, W.LAYOUT_NHD), (4, W.LAYOUT_HND))]
    for wl in calls:
        assert wl.num_positions == wl.num_requests and _uses_counters(wl)
    s = torch.cuda.Stream()
    outs = [torch.empty(wl.num_positions, dtype=torch.int64, device=DEV) for wl in calls]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    for wl, out in zip(calls, outs):
        assert _noalloc(wl, out, st, s.cuda_stream) == K.KVCS_OK
    with torch.cuda.stream(s):
        refs = [_existing(wl, s.cuda_stream) for wl in calls]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for out, ref in zip(outs, refs):
        assert torch.equal(out, ref)
    del calls
    torch.cuda.empty_cache()


def test_small_call_and_limits():
    """A call too small for the counters (fixed split) still equals the
    existing entry; more than KVCS_NOALLOC_MAX_CACHES caches is refused
    with KVCS_ETOOLARGE before any launch; no positions is a no-op."""
    wl = W.random_case(4, DEV, layers=2, heads=2, head_bytes=64, block_size=16,
                       lengths=(70, 33, 5))
    assert not _uses_counters(wl)
    s = torch.cuda.Stream()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    assert _noalloc(wl, out, st, s.cuda_stream) == K.KVCS_OK
    with torch.cuda.stream(s):
        ref = _existing(wl, s.cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and int(st.item()) == 0

    big = W.random_case(5, DEV, layers=K.KVCS_NOALLOC_MAX_CACHES + 1, heads=1,
                        head_bytes=16, block_size=16, lengths=(20,))
    before = K.launch_count()
    out2 = torch.empty(big.num_positions, dtype=torch.int64, device=DEV)
    assert _noalloc(big, out2, st, s.cuda_stream) == K.KVCS_ETOOLARGE
    assert K.launch_count() == before
    assert "1024" in K.strerror(K.KVCS_ETOOLARGE)
    arr, reqs = _abi_args(wl)
    assert K.load_library().kvcs_block_checksums_noalloc(
        arr, len(wl.caches), wl.block_size, ctypes.byref(reqs), 0, None, None,
        s.cuda_stream) == K.KVCS_OK


def test_torch_front_end_allocates_nothing():
    """The binding's front end with a caller output: no torch allocation
    during the call, and the same result as the existing entry."""
    wl = _ragged(6, 48, 32)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    n0 = torch.cuda.memory_stats()["allocation.all.allocated"]
    K.block_checksums_noalloc(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                              wl.num_tokens, wl.block_ids, out, wl.num_positions, st)
    n1 = torch.cuda.memory_stats()["allocation.all.allocated"]
    assert n1 == n0
    ref = K.workload_checksums(wl)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and int(st.item()) == 0
    assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())
