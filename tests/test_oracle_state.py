"""Pins for the oracle's Mamba state checksums (page
"vllm.distributed.kv_transfer.kv_checksum.checksum", paragraph on Mamba
state): the block at position 0 is the running state, one slice per global
row along the TP-split dimension, pieces are 2- or 4-byte unsigned
elements."""

import json
import random

import numpy as np
import pytest

from helpers import FORMS
from oracle import kvcs_oracle as O
from oracle.kvcs_oracle import OracleCache, OracleRequests
from pins import GOLDEN

H = 1 << 16


def state_cache(data, num_blocks, layer, head_offset, rows, row_elements, piece_bytes):
    return OracleCache(data, num_blocks, O.LAYOUT_STATE, layer, head_offset, rows,
                       row_elements * piece_bytes, piece_bytes)


def golden_states():
    return json.loads(GOLDEN.read_text())["states"]


def build(ex):
    pb = ex["piece_bytes"]
    data = np.zeros(ex["num_blocks"] * ex["rows"] * ex["row_elements"] * pb, dtype=np.uint8)
    view = data.reshape(ex["num_blocks"], ex["rows"], ex["row_elements"], pb)
    for blk, row, e, val in ex["elements"]:
        view[blk, row, e] = np.frombuffer(int(val).to_bytes(pb, "little"), dtype=np.uint8)
    cache = state_cache(data, ex["num_blocks"], ex["layer"], ex["head_offset"], ex["rows"],
                        ex["row_elements"], pb)
    ids = ex["block_ids"]
    reqs = OracleRequests([0, len(ids)], [ex["first_position"]], [ex["num_tokens"]], ids)
    return cache, reqs


@pytest.mark.parametrize("form", sorted(FORMS))
def test_state_hand_worked(form):
    for ex in golden_states():
        cache, reqs = build(ex)
        vals, st = FORMS[form]([cache], 16, reqs)
        assert st == 0
        assert [int(v) for v in vals] == [int(e) for e in ex["expected"]], ex["name"]


def random_state(seed, nb=5, rows=3, elems=7, pb=2, layer=4, off=10):
    rng = np.random.default_rng(seed)
    data = rng.integers(0, 256, nb * rows * elems * pb, dtype=np.uint8)
    return state_cache(data, nb, layer, off, rows, elems, pb)


@pytest.mark.parametrize("form", sorted(FORMS))
@pytest.mark.parametrize("pb", [2, 4])
def test_state_closed_forms(form, pb):
    rows, elems = 3, 9
    k = 0xBEEF if pb == 2 else 0xDEADBEEF
    one = np.frombuffer(k.to_bytes(pb, "little"), dtype=np.uint8)
    data = np.tile(one, 2 * rows * elems)
    cache = state_cache(data, 2, 7, 100, rows, elems, pb)
    reqs = OracleRequests([0, 2], [0], [5], [1, 0])
    vals, _ = FORMS[form]([cache], 16, reqs)
    msum = sum(2 * (7 * H + 100 + r) + 1 for r in range(rows))
    assert [int(v) for v in vals] == [(k * elems * elems * msum) % (1 << 64), 0]
    # a single nonzero element: x * m * (2p + 1)
    rng = random.Random(pb)
    for _ in range(10):
        r, p, x = rng.randrange(rows), rng.randrange(elems), rng.randrange(1, 1 << (8 * pb))
        data = np.zeros(2 * rows * elems * pb, dtype=np.uint8)
        data.reshape(2, rows, elems, pb)[1, r, p] = np.frombuffer(x.to_bytes(pb, "little"),
                                                                  dtype=np.uint8)
        vals, _ = FORMS[form]([state_cache(data, 2, 7, 100, rows, elems, pb)], 16, reqs)
        assert int(vals[0]) == (x * (2 * (7 * H + 100 + r) + 1) * (2 * p + 1)) % (1 << 64)


@pytest.mark.parametrize("form", sorted(FORMS))
def test_state_only_at_position_zero_and_sensitive(form):
    cache = random_state(3)
    f = FORMS[form]
    base, _ = f([cache], 16, OracleRequests([0, 3], [0], [100], [2, 0, 4]))
    assert int(base[0]) != 0 and int(base[1]) == 0 and int(base[2]) == 0
    later, _ = f([cache], 16, OracleRequests([0, 1], [1], [100], [2]))
    assert [int(v) for v in later] == [0]
    # every single-element change of block 2 changes c
    for row in range(3):
        for e in range(7):
            data = cache.data.copy()
            v = data.reshape(5, 3, 7, 2)
            v[2, row, e, 0] ^= 1
            mod = OracleCache(data, 5, O.LAYOUT_STATE, 4, 10, 3, 14, 2)
            got, _ = f([mod], 16, OracleRequests([0, 1], [0], [100], [2]))
            assert int(got[0]) != int(base[0]), (row, e)
    # swapping two rows changes c
    data = cache.data.copy()
    v = data.reshape(5, 3, 14)
    v[2, [0, 1]] = v[2, [1, 0]]
    got, _ = f([OracleCache(data, 5, O.LAYOUT_STATE, 4, 10, 3, 14, 2)], 16,
               OracleRequests([0, 1], [0], [100], [2]))
    assert int(got[0]) != int(base[0])


def test_state_forms_agree_and_widths_differ():
    for seed in range(4):
        for pb in (2, 4):
            c = random_state(seed, pb=pb, elems=5 + seed)
            reqs = OracleRequests([0, 3, 4], [0, 0], [10, 3], [4, 1, 3, 0])
            a = FORMS["python"]([c], 16, reqs)
            assert a == FORMS["c"]([c], 16, reqs)
    # the same bytes read as 2- or as 4-byte elements give different sums
    c2 = random_state(9, pb=2, elems=8)
    c4 = OracleCache(c2.data, c2.num_blocks, O.LAYOUT_STATE, c2.layer, c2.head_offset,
                     c2.num_heads, c2.head_bytes, 4)
    reqs = OracleRequests([0, 1], [0], [1], [0])
    assert FORMS["python"]([c2], 16, reqs)[0] != FORMS["python"]([c4], 16, reqs)[0]


STATE_MUTANTS = {
    "eight_byte_pieces": ("state_piece", lambda c, b, r, p: int.from_bytes(
        bytes(c.data[(b * c.num_heads + r) * c.head_bytes + 8 * p:
                     (b * c.num_heads + r) * c.head_bytes + 8 * p + 8]), "little")),
    "index_from_one": ("state_slice_checksum", lambda c, b, r: sum(
        O.state_piece(c, b, r, p) * (2 * (p + 1) + 1)
        for p in range(c.head_bytes // c.piece_bytes)) & O.MASK64),
    "signed_elements": ("state_piece", lambda c, b, r, p: int.from_bytes(
        bytes(c.data[(b * c.num_heads + r) * c.head_bytes + c.piece_bytes * p:
                     (b * c.num_heads + r) * c.head_bytes + c.piece_bytes * (p + 1)]),
        "little", signed=True) & O.MASK64),
}


@pytest.mark.parametrize("name", sorted(STATE_MUTANTS))
def test_state_mutant_is_caught(name, monkeypatch):
    attr, fn = STATE_MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    with pytest.raises(AssertionError):
        test_state_hand_worked("python")
        test_state_closed_forms("python", 2)
        test_state_closed_forms("python", 4)
        test_state_only_at_position_zero_and_sensitive("python")


def test_state_at_every_position_is_caught(monkeypatch):
    orig = O.block_checksum

    def every_position(caches, bs, block, position, nt):
        return orig(caches, bs, block, 0, nt)

    monkeypatch.setattr(O, "block_checksum", every_position)
    with pytest.raises(AssertionError):
        test_state_hand_worked("python")
