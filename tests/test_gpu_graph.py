"""The library's calls inside CUDA graphs: they allocate nothing and never
synchronise, so a serving engine can capture them with its step.  A captured
call replayed after the pools change gives the direct call's result."""

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("lengths", [(70, 33, 5), (1024,) * 19])
def test_captured_checksums_match_direct_calls(lengths):
    wl = W.random_case(11, DEV, layers=3, heads=4, head_bytes=64, lengths=lengths)
    ck = K.Checksummer(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                       wl.num_tokens, wl.block_ids, wl.num_positions)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    acc = torch.zeros(wl.num_positions, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):           # warm up outside the capture
        ck(out, status, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ck(out, status, s.cuda_stream)
        ck(acc, status, s.cuda_stream, accumulate=True)
    gen = torch.Generator(device=DEV).manual_seed(3)
    for _ in range(3):
        for c in wl.caches:              # new KV in place, then replay
            c.pool.copy_(torch.randint(0, 256, c.pool.shape, dtype=torch.uint8,
                                       device=DEV, generator=gen))
        before = acc.clone()
        g.replay()
        torch.cuda.synchronize()
        ref = torch.empty_like(out)
        K.workload_checksums(wl, out=ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        u = lambda t: t.cpu().numpy().view(np.uint64)
        assert np.array_equal(u(acc), u(before) + u(ref))    # wraps mod 2^64
    assert int(status.item()) == 0


def test_captured_write_matches_direct_write():
    bs, nb, heads, hb, layers, n = 16, 12, 4, 64, 3, 50
    g0 = torch.Generator().manual_seed(4)
    slots = torch.randperm(nb * bs, generator=g0)[:n].to(DEV)
    pos = torch.randint(0, 500, (n,), generator=g0).to(DEV)
    keys = [torch.empty((n, heads, hb), dtype=torch.uint8, device=DEV) for _ in range(layers)]
    vals = [torch.empty((n, heads, hb), dtype=torch.uint8, device=DEV) for _ in range(layers)]

    def caches():
        return [W.CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8,
                                        device=DEV), nb, W.LAYOUT_NHD, li, 0, heads, hb)
                for li in range(layers)]

    a, b = caches(), caches()
    sa = torch.zeros(nb, dtype=torch.int64, device=DEV)
    sb = torch.zeros(nb, dtype=torch.int64, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.write_kv(a, bs, keys, vals, slots, pos, block_sums=sa, stream=s.cuda_stream)
    torch.cuda.synchronize()
    sa.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        K.write_kv(a, bs, keys, vals, slots, pos, block_sums=sa, stream=s.cuda_stream)
    gen = torch.Generator(device=DEV).manual_seed(5)
    for _ in range(2):
        for t in keys + vals:
            t.copy_(torch.randint(0, 256, t.shape, dtype=torch.uint8, device=DEV,
                                  generator=gen))
        g.replay()
        K.write_kv(b, bs, keys, vals, slots, pos, block_sums=sb)
        torch.cuda.synchronize()
        assert torch.equal(sa, sb)
        for ca, cb in zip(a, b):
            assert torch.equal(ca.pool, cb.pool)


def test_concurrent_calls_on_several_streams():
    """Calls enqueued on four streams at once (their kernels may overlap)
    give the results of the same calls made one at a time."""
    wls = [W.random_case(20 + k, DEV, layers=3, heads=4, head_bytes=64,
                         lengths=(300, 41, 77), layout=(W.LAYOUT_NHD, W.LAYOUT_HND)[k % 2])
           for k in range(4)]
    ref = []
    for wl in wls:
        out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
        K.workload_checksums(wl, out=out)
        ref.append(out)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in wls]
    cks = [K.Checksummer(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                         wl.num_tokens, wl.block_ids, wl.num_positions) for wl in wls]
    outs = [torch.zeros_like(r) for r in ref]
    for _ in range(5):
        for ck, out, s in zip(cks, outs, streams):
            ck(out, None, s.cuda_stream)
    torch.cuda.synchronize()
    for out, r in zip(outs, ref):
        assert torch.equal(out, r)
