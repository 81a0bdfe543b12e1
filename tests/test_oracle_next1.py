"""Pins for the oracle's replica-key columns, offload row sums and block
tags (page "vllm.distributed.kv_transfer.kv_checksum.checksum": paragraph on
replicated KV, dataclass KVChecksumGroup, function block_checksum_tags)."""

import json
import random

import numpy as np
import pytest

from helpers import W, OracleCache, c_form, oracle_inputs, py_form
from oracle import kvcs_oracle as O
from pins import GOLDEN


def _tag_golden():
    return json.loads(GOLDEN.read_text())["tags"]


def test_tags_hand_worked():
    for ex in _tag_golden():
        hashes = [bytes.fromhex(h) for h in ex["hashes_hex"]]
        assert O.block_checksum_tags(hashes, int(ex["fingerprint"])) == \
            [int(v) for v in ex["expected"]]


def test_tags_properties():
    rng = random.Random(3)
    hashes = [bytes(rng.getrandbits(8) for _ in range(32)) for _ in range(20)]
    fp = rng.getrandbits(64)
    tags = O.block_checksum_tags(hashes, fp)
    # only the first eight bytes matter
    other = [h[:8] + bytes(rng.getrandbits(8) for _ in range(24)) for h in hashes]
    assert O.block_checksum_tags(other, fp) == tags
    # XOR with the fingerprint: fingerprint 0 gives the raw words, and
    # tagging twice with one fingerprint cancels
    raw = O.block_checksum_tags(hashes, 0)
    assert [t ^ fp for t in raw] == tags
    assert [int.from_bytes(h[:8], "little") for h in hashes] == raw
    # little-endian: byte k weighs 256**k
    assert O.block_checksum_tags([bytes([0, 1] + [0] * 6)], 0) == [256]


def _column_case(seed):
    wl = W.random_case(seed, "cpu", layers=5, heads=2, head_bytes=16, block_size=4,
                       lengths=(14, 5), layer_numbers=[0, 1, 2, 3, 4])
    caches, reqs = oracle_inputs(wl)
    columns = [0, 1, 0, 2, 1]
    return caches, reqs, columns


@pytest.mark.parametrize("seed", [0, 1])
def test_columns_sum_to_the_whole_checksum(seed):
    caches, reqs, columns = _column_case(seed)
    values, st = O.column_checksums(caches, columns, 3, 4, reqs)
    full, _ = py_form(caches, 4, reqs)
    assert st == 0
    assert O.row_sums(values) == full
    # each column is the checksum of its own caches alone
    for k in range(3):
        sub = [c for c, col in zip(caches, columns) if col == k]
        assert [row[k] for row in values] == py_form(sub, 4, reqs)[0]
        assert [row[k] for row in values] == c_form(sub, 4, reqs)[0]


def test_column_of_zero_caches_is_zero():
    caches, reqs, columns = _column_case(2)
    zeroed = [OracleCache(np.zeros_like(c.data), c.num_blocks, c.layout, c.layer,
                          c.head_offset, c.num_heads, c.head_bytes)
              if col == 1 else c for c, col in zip(caches, columns)]
    values, _ = O.column_checksums(zeroed, columns, 3, 4, reqs)
    assert all(row[1] == 0 for row in values)
    assert all(row[0] != 0 for row in values[:2])


def test_tagged_row_sums_detect_wrong_blocks_and_tags():
    caches, reqs, columns = _column_case(4)
    values, _ = O.column_checksums(caches, columns, 3, 4, reqs)
    rng = random.Random(5)
    hashes = [bytes(rng.getrandbits(8) for _ in range(32)) for _ in values]
    tags = O.block_checksum_tags(hashes, 0x1234)
    stored = O.row_sums(values, tags)
    # the same KV under the same tags matches
    assert O.row_sums(values, tags) == stored
    # a block loaded into the wrong position mismatches
    ids = list(reqs.block_ids)
    ids[0], ids[1] = ids[1], ids[0]
    moved = O.OracleRequests(reqs.pos_offsets, reqs.first_position, reqs.num_tokens, ids)
    v2, _ = O.column_checksums(caches, columns, 3, 4, moved)
    fresh = O.row_sums(v2, tags)
    assert fresh[0] != stored[0] and fresh[1] != stored[1]
    assert fresh[2:] == stored[2:]
    # the right KV checked against another block's tag mismatches
    other = O.block_checksum_tags([hashes[1]] + hashes[1:], 0x1234)
    assert O.row_sums(values, other)[0] != stored[0]
