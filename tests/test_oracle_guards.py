"""What the oracle refuses, and the rule that combines partials, pinned in
both forms.

Page "vllm.distributed.kv_transfer.kv_checksum.checksum":

* attribute ``MAX_KV_HEADS_PER_LAYER``: a group whose layers have more KV
  heads than H is left out of checksumming, so a head range reaching past
  H is refused;
* module docstring item 1: pieces are whole 8-byte words of a token's
  slice, so per-head bytes that are not a multiple of 8 are refused; a
  latent row is one slice (one head); x-split heads are whole 16-byte
  chunks, and kernel sub-blocks split a block evenly (the KV-cache page,
  "reshape kv_cache");
* the paragraph on TP ranks and PP stages: partials from every shard add
  up, mod 2**64, to the unsharded checksum (``combine_partials``).

A pool smaller than the pages its geometry addresses is refused by both
forms as well, so a bad test descriptor cannot read past the host array.
"""

import dataclasses

import numpy as np
import pytest

from helpers import FORMS, W, OracleCache, OracleRequests
from oracle import kvcs_oracle as O
from pins import pool_view, random_pool_case

M64 = (1 << 64) - 1


def _kv_case(layout=W.LAYOUT_NHD, heads=2, hb=16, bs=4):
    _, caches, r = random_pool_case(61, layout, layers=2, heads=heads, hb=hb, bs=bs,
                                    lengths=[9], spare=1)
    return caches, r, bs


def _zeros_cache(layout, nb, bs, heads, hb, **kw):
    halves = 1 if layout == W.LAYOUT_LATENT else 2
    return OracleCache(np.zeros(halves * nb * bs * heads * hb, dtype=np.uint8), nb, layout,
                       0, 0, heads, hb, **kw)


def _state_case(rows=3, row_bytes=8, piece_bytes=2, nb=2):
    data = np.arange(nb * rows * row_bytes, dtype=np.uint8)
    c = OracleCache(data, nb, W.LAYOUT_STATE, 0, 0, rows, row_bytes, piece_bytes)
    return [c], OracleRequests([0, 1], [0], [5], [1]), 16


def _refused():
    """(name, caches, requests, block_size) cases both forms must refuse."""
    caches, r, bs = _kv_case()
    c0 = caches[0]
    out = [
        # head range past H = 65536 (attribute MAX_KV_HEADS_PER_LAYER)
        ("heads_past_H", [dataclasses.replace(c0, head_offset=65535)], r, bs),
        ("negative_head_offset", [dataclasses.replace(c0, head_offset=-1)], r, bs),
        # per-head bytes not whole 8-byte pieces (item 1)
        ("head_bytes_12", [_zeros_cache(W.LAYOUT_NHD, c0.num_blocks, bs, 2, 12)], r, bs),
        # a latent row is one slice: exactly one head
        ("latent_two_heads", [_zeros_cache(W.LAYOUT_LATENT, c0.num_blocks, bs, 2, 16)], r, bs),
        # x-split heads are whole 16-byte chunks
        ("xsplit_head_bytes_8", [_zeros_cache(W.LAYOUT_XSPLIT, c0.num_blocks, bs, 2, 8)], r, bs),
        # kernel sub-blocks split an HND block evenly
        ("kernel_block_3_of_4", [_zeros_cache(W.LAYOUT_HND, c0.num_blocks, bs, 2, 16,
                                              kernel_block_size=3)], r, bs),
        # pools smaller than their geometry
        ("pool_short_by_one", [dataclasses.replace(c0, data=c0.data[:-1])], r, bs),
        ("pool_short_strided", [dataclasses.replace(c0, block_stride=2 * bs * 2 * 16)], r, bs),
        ("negative_stride", [dataclasses.replace(c0, half_stride=-8)], r, bs),
    ]
    sc, sr, sbs = _state_case()
    s0 = sc[0]
    out += [
        ("state_piece_bytes_8", [dataclasses.replace(s0, piece_bytes=8)], sr, sbs),
        ("state_row_not_whole_elements", [dataclasses.replace(s0, head_bytes=7,
                                                              data=s0.data[:2 * 3 * 7])], sr, sbs),
        ("state_rows_past_H", [dataclasses.replace(s0, head_offset=65534)], sr, sbs),
        ("state_pool_short", [dataclasses.replace(s0, data=s0.data[:-1])], sr, sbs),
    ]
    return out


REFUSED = _refused()


@pytest.mark.parametrize("form", sorted(FORMS))
@pytest.mark.parametrize("case", REFUSED, ids=[c[0] for c in REFUSED])
def test_refused(case, form):
    _, caches, r, bs = case
    with pytest.raises(ValueError):
        FORMS[form](caches, bs, r)


@pytest.mark.parametrize("form", sorted(FORMS))
def test_accepted_at_the_limits(form):
    """The boundaries themselves are accepted: a head range ending at H
    exactly, a pool of exactly the bytes its geometry needs, and a state
    whose last row ends at H."""
    caches, r, bs = _kv_case()
    c0 = caches[0]
    last = dataclasses.replace(c0, head_offset=65534)         # heads 65534, 65535
    vals, st = FORMS[form]([last], bs, r)
    assert st == 0 and len(vals) == len(r.block_ids)
    # a strided pool holding exactly up to the end of its last page
    page = bs * 2 * 16
    nb = c0.num_blocks
    tight = np.zeros(nb * 2 * page, dtype=np.uint8)           # [block][K page, V page]
    v = tight.reshape(nb, 2, page)
    v[:, 0] = c0.data.reshape(2, nb, page)[0]
    v[:, 1] = c0.data.reshape(2, nb, page)[1]
    strided = dataclasses.replace(c0, data=tight, half_stride=page, block_stride=2 * page)
    a, _ = FORMS[form]([c0], bs, r)
    b, _ = FORMS[form]([strided], bs, r)
    assert [int(x) for x in a] == [int(x) for x in b]
    sc, sr, sbs = _state_case()
    top = dataclasses.replace(sc[0], head_offset=65536 - 3)
    vals, st = FORMS[form]([top], sbs, sr)
    assert st == 0 and int(vals[0]) != 0


# ---------------------------------------------------------------------------
# combine_partials
# ---------------------------------------------------------------------------

def _shard_partials(form):
    """Real partials of one request set: two TP head shards of every layer,
    and two PP stages (layers 0-1 and 2-3), with the unsharded checksums."""
    bs = 3
    _, caches, r = random_pool_case(67, W.LAYOUT_NHD, layers=4, heads=4, hb=8, bs=bs,
                                    lengths=[13, 7], layer_numbers=[0, 1, 2, 3])
    full = [int(x) for x in form(caches, bs, r)[0]]
    tp = []
    for lo, hi in ((0, 3), (3, 4)):
        part = []
        for c in caches:
            v = pool_view(c.data, c.layout, c.num_blocks, bs, c.num_heads, c.head_bytes)
            sub = np.ascontiguousarray(v[:, :, :, lo:hi, :]).reshape(-1)
            part.append(OracleCache(sub, c.num_blocks, c.layout, c.layer, c.head_offset + lo,
                                    hi - lo, c.head_bytes))
        tp.append([int(x) for x in form(part, bs, r)[0]])
    pp = [[int(x) for x in form(caches[:2], bs, r)[0]],
          [int(x) for x in form(caches[2:], bs, r)[0]]]
    return full, tp, pp


def check_combine(combine, form):
    """``combine`` must turn the shards' partials back into the unsharded
    checksums, for TP shards, PP stages and both at once, where the plain
    integer sums run past 2**64."""
    full, tp, pp = _shard_partials(form)
    assert any(sum(col) > M64 for col in zip(*tp)), "the case must wrap"
    assert [int(x) for x in combine(tp)] == full
    assert [int(x) for x in combine(pp)] == full
    # all four partials at once count every slice twice: 2c mod 2**64
    assert [int(x) for x in combine(tp + pp)] == [(2 * c) & M64 for c in full]
    # one shard alone, and a shard that contributes nothing
    assert [int(x) for x in combine([full])] == full
    assert [int(x) for x in combine([full, [0] * len(full)])] == full


@pytest.mark.parametrize("form", sorted(FORMS))
def test_combine_partials(form):
    check_combine(O.combine_partials, FORMS[form])


@pytest.mark.parametrize("mutant", [
    lambda parts: [sum(col) for col in zip(*parts)],                  # no mod 2**64
    lambda parts: [sum(col) & ((1 << 63) - 1) for col in zip(*parts)],  # 63-bit mask
    lambda parts: [max(col) for col in zip(*parts)],                  # not a sum
    lambda parts: [(col[0] - sum(col[1:])) & M64 for col in zip(*parts)],  # wrong sign
    lambda parts: [col[0] ^ col[-1] for col in zip(*parts)],          # XOR instead
], ids=["no_mask", "mask63", "max", "minus", "xor"])
def test_combine_pin_catches(mutant):
    """Planted mistakes in the combining rule (on the CPU) fail the pin."""
    with pytest.raises(AssertionError):
        check_combine(mutant, FORMS["python"])
