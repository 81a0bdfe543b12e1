"""Parity of the CUDA library with the oracle, through the C ABI.

Bit-exact uint64 equality everywhere: the checksum is exact integer
arithmetic mod 2**64, so there is exactly one correct answer."""

import numpy as np
import pytest
import torch

from helpers import W, oracle_inputs, py_form
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu

DEV = "cuda"


def gpu(wl, stream=None):
    from gpu_helpers import gpu_checksums
    return gpu_checksums(wl, stream)


def oracle(wl):
    from gpu_helpers import full_oracle
    return full_oracle(wl)


def assert_equal(got, exp):
    got = np.asarray(got, dtype=np.uint64)
    exp = np.asarray(exp, dtype=np.uint64)
    assert got.shape == exp.shape
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:8].tolist()}"


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_bit_exact(seed):
    wl = W.tiny(seed, DEV)
    got, st = gpu(wl)
    caches, reqs = oracle_inputs(wl)
    exp, est = py_form(caches, wl.block_size, reqs)
    assert st == 0 and est == 0
    assert_equal(got, exp)
    assert K.plan_for(wl.caches, wl.block_size, wl.num_positions)["kernel"] == 0


# Bulk-kernel geometries: every layout, units per page > 1, HND heads per
# unit < heads, ragged lengths, first positions > 0, positions past the
# tokens, large layer numbers and head offsets.
BULK = [
    dict(layout=W.LAYOUT_NHD, layers=3, heads=8, head_bytes=256, block_size=16,
         lengths=(100, 37, 1, 64)),
    dict(layout=W.LAYOUT_NHD, layers=2, heads=4, head_bytes=128, block_size=80,
         lengths=(300, 81, 79)),                      # 2 units per page
    dict(layout=W.LAYOUT_NHD, layers=2, heads=2, head_bytes=16, block_size=1,
         lengths=(9, 3)),
    dict(layout=W.LAYOUT_NHD, layers=2, heads=3, head_bytes=48, block_size=7,
         lengths=(50, 20), first_positions=(2, 0), extra_positions=(1, 3)),
    dict(layout=W.LAYOUT_HND, layers=2, heads=8, head_bytes=256, block_size=64,
         lengths=(200, 64, 65)),                      # 4 heads per unit
    dict(layout=W.LAYOUT_HND, layers=3, heads=5, head_bytes=32, block_size=16,
         lengths=(47, 16, 3), first_positions=(1, 0, 0)),
    dict(layout=W.LAYOUT_HND, layers=1, heads=3, head_bytes=4096, block_size=8,
         lengths=(30,)),                              # 1 head per unit, 256 cols
    dict(layout=W.LAYOUT_LATENT, layers=3, heads=1, head_bytes=1152, block_size=64,
         lengths=(200, 64, 1)),                       # 3 units per page
    dict(layout=W.LAYOUT_LATENT, layers=2, heads=1, head_bytes=16, block_size=5,
         lengths=(23,), extra_positions=(2,)),
    dict(layout=W.LAYOUT_NHD, layers=2, heads=64, head_bytes=512, block_size=4,
         lengths=(9,)),                               # 32 KiB rows, 2048 cols
    dict(layout=W.LAYOUT_NHD, layers=2, heads=1, head_bytes=16, block_size=4,
         lengths=[8] * 152),                          # whole-position mode
    dict(layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=16, block_size=4,
         lengths=(4,), layer_numbers=(32767, 9), head_offset=65534),
    dict(layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=256, block_size=256,
         lengths=(300, 256)),                         # 64 KiB units, 3 stages
    dict(layout=W.LAYOUT_NHD, layers=3, heads=8, head_bytes=128, block_size=16,
         lengths=[37] * 40, first_positions=[1] * 40),  # fp8-shaped, 16 KiB pages
    dict(layout=W.LAYOUT_HND, layers=5, heads=2, head_bytes=64, block_size=16,
         lengths=(70, 9, 16)),                        # 2 KiB pages, 10 per unit
    dict(layout=W.LAYOUT_LATENT, layers=7, heads=1, head_bytes=64, block_size=16,
         lengths=(33, 100), extra_positions=(1, 0)),  # 1 KiB pages, 7 per unit
    dict(layout=W.LAYOUT_NHD, layers=6, heads=4, head_bytes=1024, block_size=2,
         lengths=(11, 4)),                            # 8 KiB pages, 4 per unit
    dict(layout=W.LAYOUT_NHD, layers=2, heads=2, head_bytes=64, block_size=16,
         lengths=((1 << 57) * 16 + 37,), first_positions=(1 << 57,)),  # t P wraps 2^64
    # decode-shaped HND: each request lists only its newest block, holding
    # 1, 2 or 15 tokens (only those slots are copied), plus full blocks
    dict(layout=W.LAYOUT_HND, layers=3, heads=8, head_bytes=256, block_size=16,
         lengths=[16 * k + 1 for k in range(40)] + [16 * 7 + 2, 16 * 3 + 15, 64],
         first_positions=list(range(40)) + [7, 3, 0]),
    dict(layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=64, block_size=16,
         lengths=[16 * (k % 9) + 1 + (k % 3) for k in range(304)],
         first_positions=[k % 9 for k in range(304)]),  # whole-position mode
]


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("case", range(len(BULK)))
def test_bulk_kernel_matches_oracle(case, seed):
    wl = W.random_case(seed, DEV, **BULK[case])
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0
    got, st = gpu(wl)
    exp, est = oracle(wl)
    assert st == est == 0
    assert_equal(got, exp)


def test_whole_position_mode_is_used():
    wl = W.random_case(0, DEV, **BULK[10])
    assert wl.num_positions == 304
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if wl.num_positions >= sms and (wl.num_positions % sms == 0):
        assert plan["split"] == 0 and plan["memsets"] == 0


# Generic-kernel geometries: per-head bytes not a multiple of 16, rows
# bigger than a stage.
GENERIC = [
    dict(layout=W.LAYOUT_NHD, layers=2, heads=3, head_bytes=24, block_size=16,
         lengths=(70, 5)),
    dict(layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=8, block_size=3,
         lengths=(10,), first_positions=(1,)),
    dict(layout=W.LAYOUT_LATENT, layers=2, heads=1, head_bytes=72, block_size=16,
         lengths=(40,), extra_positions=(1,)),
    dict(layout=W.LAYOUT_HND, layers=1, heads=2, head_bytes=256, block_size=512,
         lengths=(600,)),                             # head run > 64 KiB
    dict(layout=W.LAYOUT_NHD, layers=2, heads=3, head_bytes=24, block_size=16,
         lengths=((1 << 57) * 16 + 20,), first_positions=(1 << 57,)),  # t P wraps 2^64
]


@pytest.mark.parametrize("case", range(len(GENERIC)))
def test_generic_kernel_matches_oracle(case):
    wl = W.random_case(3, DEV, **GENERIC[case])
    assert K.plan_for(wl.caches, wl.block_size, wl.num_positions)["kernel"] == 1
    got, st = gpu(wl)
    exp, est = oracle(wl)
    assert st == est == 0
    assert_equal(got, exp)


@pytest.mark.parametrize("layout,kernel", [(W.LAYOUT_NHD, 0), (W.LAYOUT_HND, 0)])
def test_misaligned_base(layout, kernel):
    """Pools 8 bytes past a 16-byte boundary: NHD rows and HND heads go to
    the bulk kernel's misaligned instances."""
    wl = W.random_case(4, DEV, layout=layout, layers=2, heads=2, head_bytes=32, block_size=4,
                       lengths=(13,))
    for c in wl.caches:
        raw = torch.zeros(c.pool.numel() + 8, dtype=torch.uint8, device=DEV)
        raw[8:] = c.pool
        c.pool = raw[8:]
    assert K.plan_for(wl.caches, wl.block_size, wl.num_positions)["kernel"] == kernel
    got, st = gpu(wl)
    exp, _ = oracle(wl)
    assert st == 0
    assert_equal(got, exp)


@pytest.mark.parametrize("layers", [129, 300])
def test_many_caches_split_over_launches(layers):
    wl = W.random_case(5, DEV, layers=layers, heads=1, head_bytes=16, block_size=2,
                       lengths=(7, 2))
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["launches"] == -(-layers // 128) and plan["memsets"] == 1
    before = K.launch_count()
    got, st = gpu(wl)
    # the checksum launches and the kernel that zeroes the output first
    assert K.launch_count() - before == plan["launches"] + plan["memsets"]
    exp, _ = oracle(wl)
    assert_equal(got, exp)


def test_bad_block_ids_flagged_and_zeroed():
    wl = W.random_case(6, DEV, layers=2, heads=2, head_bytes=32, block_size=4,
                       lengths=(30, 9), spare_blocks=0)
    good, st = gpu(wl)
    assert st == 0
    ids = wl.block_ids.clone()
    ids[1] = wl.caches[0].num_blocks
    ids[4] = -7
    wl.block_ids = ids
    got, st = gpu(wl)
    assert st & K.KVCS_STATUS_BAD_BLOCK_ID
    exp = good.copy()
    exp[[1, 4]] = 0
    assert_equal(got, exp)


def test_bad_request_table_flagged():
    wl = W.random_case(7, DEV, layers=1, heads=1, head_bytes=16, block_size=4,
                       lengths=(16,))
    total = wl.num_positions
    po = wl.pos_offsets.clone()
    po[-1] -= 1          # the last position now belongs to no request
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = K.block_checksums(wl.caches, wl.block_size, po, wl.first_position,
                            wl.num_tokens, wl.block_ids, status=status,
                            total_positions=total)
    torch.cuda.synchronize()
    assert int(status.item()) & K.KVCS_STATUS_BAD_REQUESTS
    assert int(out[-1].item()) == 0


def test_empty_and_zero_token_requests():
    wl = W.random_case(8, DEV, layers=2, heads=2, head_bytes=16, block_size=4,
                       lengths=(0, 5, 0), extra_positions=(2, 0, 1))
    got, st = gpu(wl)
    exp, _ = oracle(wl)
    assert st == 0
    assert_equal(got, exp)
    assert got[0] == got[1] == got[-1] == 0
    # no positions at all: nothing is launched
    before = K.launch_count()
    empty = K.block_checksums(wl.caches, 4, torch.zeros(1, dtype=torch.int64, device=DEV),
                              torch.zeros(0, dtype=torch.int64, device=DEV),
                              torch.zeros(0, dtype=torch.int64, device=DEV),
                              torch.zeros(0, dtype=torch.int32, device=DEV))
    assert empty.numel() == 0 and K.launch_count() == before


def test_shared_block_ids_and_nondefault_stream():
    wl = W.random_case(9, DEV, layers=2, heads=4, head_bytes=64, block_size=8,
                       lengths=(40, 40), spare_blocks=0)
    ids = wl.block_ids.clone()
    half = ids.numel() // 2
    ids[half:2 * half] = ids[:half]        # second request shares the prefix
    wl.block_ids = ids
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got, st = gpu(wl, stream=s)
    exp, _ = oracle(wl)
    assert st == 0
    assert_equal(got, exp)


def test_invariance_small():
    """Producer bs16 NHD, consumer bs64 HND, and two TP shards, on one GPU:
    every 4 producer positions sum to a consumer position, and the shards'
    partials sum to the producer's checksums."""
    prod, cons, s0, s1 = W.invariance(0, DEV, num_requests=3, tokens=300, layers=4)
    a, _ = gpu(prod)
    b, _ = gpu(cons)
    c0, _ = gpu(s0)
    c1, _ = gpu(s1)
    assert_equal(c0 + c1, a)
    for r in range(3):
        pa = a[int(prod.pos_offsets[r]):int(prod.pos_offsets[r + 1])]
        pb = b[int(cons.pos_offsets[r]):int(cons.pos_offsets[r + 1])]
        for k in range(len(pb)):
            assert pb[k] == pa[4 * k:4 * k + 4].sum(dtype=np.uint64)
    exp, _ = oracle(cons)
    assert_equal(b, exp)


def test_mixed_geometry_caches():
    """Caches of different shapes in one call: an attention cache and an
    indexer cache of layer 0 (consecutive head numbers), an HND layer and a
    latent layer, all addressed by one block table."""
    g = torch.Generator(device=DEV).manual_seed(11)
    base = W.random_case(11, DEV, layers=1, heads=4, head_bytes=128, block_size=16,
                         lengths=(70, 33, 5))
    nb = base.caches[0].num_blocks
    specs = [(W.LAYOUT_NHD, 0, 0, 4, 128), (W.LAYOUT_NHD, 0, 4, 1, 64),
             (W.LAYOUT_HND, 1, 0, 2, 256), (W.LAYOUT_LATENT, 2, 0, 1, 576),
             (W.LAYOUT_NHD, 3, 2, 3, 32)]
    caches = []
    for layout, layer, off, heads, hb in specs:
        nbytes = W.pool_bytes(layout, nb, 16, heads, hb)
        caches.append(W.CacheSpec(W.fill_bytes(nbytes, W.BYTES, g, torch.device(DEV)),
                                  nb, layout, layer, off, heads, hb))
    wl = W.Workload("mixed", 16, caches, base.pos_offsets, base.first_position,
                    base.num_tokens, base.block_ids)
    plan = K.plan_for(wl.caches, wl.block_size, wl.num_positions)
    assert plan["kernel"] == 0
    got, st = gpu(wl)
    exp, est = oracle(wl)
    assert st == est == 0
    assert_equal(got, exp)


def test_prepared_call_matches_and_follows_refilled_tables():
    wl = W.random_case(12, DEV, layers=3, heads=2, head_bytes=64, block_size=8,
                       lengths=(50, 17), spare_blocks=4)
    ck = K.workload_checksummer(wl)
    out = torch.empty(wl.num_positions, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ck(out, st, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    exp, _ = oracle(wl)
    assert_equal(out.cpu().numpy().view(np.uint64), exp)
    # refill the block table in place (same addresses): the prepared call
    # reads the new ids
    perm = torch.randperm(wl.caches[0].num_blocks, generator=torch.Generator().manual_seed(3))
    wl.block_ids.copy_(perm[:wl.num_positions].to(torch.int32).to(DEV))
    ck(out, st, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    exp2, _ = oracle(wl)
    assert int(st.item()) == 0
    assert_equal(out.cpu().numpy().view(np.uint64), exp2)
