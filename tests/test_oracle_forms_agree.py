"""The C form equals the pure-Python form on seeded random cases of every
layout, including ragged lengths, first positions, extra positions and
unusual geometries; and on the tiny workload."""

import pytest

from helpers import W, c_form, oracle_inputs, py_form

CASES = [
    dict(layout=W.LAYOUT_NHD, layers=3, heads=2, head_bytes=16, block_size=4,
         lengths=(13, 1, 8)),
    dict(layout=W.LAYOUT_HND, layers=2, heads=3, head_bytes=24, block_size=5,
         lengths=(7, 11), first_positions=(0, 1)),
    dict(layout=W.LAYOUT_LATENT, layers=2, heads=1, head_bytes=40, block_size=3,
         lengths=(10,), extra_positions=(2,)),
    dict(layout=W.LAYOUT_NHD, layers=1, heads=1, head_bytes=8, block_size=1,
         lengths=(5, 0, 2), extra_positions=(0, 2, 1)),
    dict(layout=W.LAYOUT_HND, layers=2, heads=2, head_bytes=8, block_size=7,
         lengths=(20,), layer_numbers=(60, 7), head_offset=65530),
]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_c_equals_python(case, seed):
    wl = W.random_case(seed, "cpu", **CASES[case])
    caches, reqs = oracle_inputs(wl)
    assert c_form(caches, wl.block_size, reqs) == py_form(caches, wl.block_size, reqs)


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("layout,kbs,hb,bs", [(W.LAYOUT_XSPLIT, 0, 32, 5),
                                              (W.LAYOUT_XSPLIT, 0, 16, 1),
                                              (W.LAYOUT_HND, 2, 24, 6),
                                              (W.LAYOUT_HND, 1, 8, 3)])
def test_c_equals_python_xsplit_and_sub_blocks(seed, layout, kbs, hb, bs):
    import dataclasses
    wl = W.random_case(seed, "cpu", layout=layout, layers=2, heads=2, head_bytes=hb,
                       block_size=bs, lengths=(13, 4), first_positions=(1, 0))
    wl = dataclasses.replace(wl, caches=[dataclasses.replace(c, kernel_block_size=kbs)
                                         for c in wl.caches])
    caches, reqs = oracle_inputs(wl)
    assert c_form(caches, wl.block_size, reqs) == py_form(caches, wl.block_size, reqs)


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_workload(seed):
    wl = W.tiny(seed)
    caches, reqs = oracle_inputs(wl)
    a = py_form(caches, wl.block_size, reqs)
    assert a == c_form(caches, wl.block_size, reqs, threads=3)
    assert len(a[0]) == 7 and a[1] == 0 and all(v != 0 for v in a[0])


def test_threads_do_not_change_results():
    wl = W.random_case(5, "cpu", layers=2, heads=4, head_bytes=16, block_size=4,
                       lengths=(33, 17, 2, 40))
    caches, reqs = oracle_inputs(wl)
    one = c_form(caches, wl.block_size, reqs, threads=1)
    for t in (2, 3, 7, 64):
        assert c_form(caches, wl.block_size, reqs, threads=t) == one


@pytest.mark.parametrize("layout", [W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_LATENT, W.LAYOUT_XSPLIT])
def test_c_equals_python_with_strides(layout):
    """Pages placed by explicit strides: K and V interleaved per block with
    padding."""
    import dataclasses
    import numpy as np
    hb = 32
    heads = 1 if layout == W.LAYOUT_LATENT else 2
    wl = W.random_case(3, "cpu", layout=layout, layers=2, heads=heads, head_bytes=hb,
                       block_size=4, lengths=(11, 6))
    caches, reqs = oracle_inputs(wl)
    page = 4 * heads * hb
    halves = 1 if layout == W.LAYOUT_LATENT else 2
    strided = []
    for c in caches:
        buf = np.zeros((c.num_blocks, halves, page + 16), dtype=np.uint8)
        buf[:, :, :page] = c.data.reshape(halves, c.num_blocks, page).transpose(1, 0, 2)
        strided.append(dataclasses.replace(c, data=buf.reshape(-1), half_stride=page + 16,
                                           block_stride=halves * (page + 16)))
    a = py_form(caches, 4, reqs)
    assert c_form(strided, 4, reqs) == py_form(strided, 4, reqs) == a
