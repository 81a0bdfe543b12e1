"""Plant plausible mistakes in the pure-Python oracle (on the CPU only) and
check that the pins catch every one: a dropped term, a wrong sign or index, a
transposed operand, a missing truncation or reduction."""

import pytest

from helpers import py_form
from oracle import kvcs_oracle as O
from pins import ALL_PINS


def _nhd_transposed(cache, bs, block, slot, head, p):
    hb = cache.head_bytes
    byte = 8 * p
    kv = 0
    if byte >= hb:
        kv, byte = 1, byte - hb
    page = kv * cache.num_blocks + block
    if cache.layout == O.LAYOUT_NHD:  # head and slot axes swapped
        return ((page * cache.num_heads + head) * bs + slot) * hb + byte
    return ORIG["piece_byte_offset"](cache, bs, block, slot, head, p)


def _v_then_k(cache, bs, block, slot, head, p):
    if cache.layout == O.LAYOUT_LATENT:
        return ORIG["piece_byte_offset"](cache, bs, block, slot, head, p)
    half = cache.head_bytes // 8
    q = p + half if p < half else p - half
    return ORIG["piece_byte_offset"](cache, bs, block, slot, head, q)


def _block_ignored(cache, bs, block, slot, head, p):
    return ORIG["piece_byte_offset"](cache, bs, 0, slot, head, p)


def _xsplit_axes_swapped(cache, bs, block, slot, head, p):
    if cache.layout != O.LAYOUT_XSPLIT:
        return ORIG["piece_byte_offset"](cache, bs, block, slot, head, p)
    hb = cache.head_bytes
    byte = 8 * p
    kv = 0
    if byte >= hb:
        kv, byte = 1, byte - hb
    page = kv * cache.num_blocks + block
    chunk, inner = divmod(byte, 16)   # slot and chunk axes swapped
    return (((page * cache.num_heads + head) * bs + slot) * (hb // 16) + chunk) * 16 + inner


def _sub_blocks_ignored(cache, bs, block, slot, head, p):
    import dataclasses
    return ORIG["piece_byte_offset"](dataclasses.replace(cache, kernel_block_size=0), bs,
                                     block, slot, head, p)


ORIG = {name: getattr(O, name) for name in (
    "piece_byte_offset", "piece_weight", "piece_index", "token_position",
    "slice_factor", "num_valid_tokens", "pieces_per_token", "read_piece")}

MUTANTS = {
    "even_weight_2j": ("piece_weight", lambda j: 2 * j),
    "weight_j_plus_1": ("piece_weight", lambda j: j + 1),
    "weight_2j_minus_1": ("piece_weight", lambda j: 2 * j - 1),
    "index_drops_p": ("piece_index", lambda t, P, p: t * P),
    "index_transposed": ("piece_index", lambda t, P, p: p * P + t),
    "index_pieces_from_block_start": ("token_position",
                                      lambda pos, bs, slot: slot),
    "position_off_by_one": ("token_position",
                            lambda pos, bs, slot: pos * bs + slot + 1),
    "even_factor": ("slice_factor", lambda l, g: 2 * (l * O.MAX_KV_HEADS_PER_LAYER + g)),
    "factor_wrong_H": ("slice_factor", lambda l, g: 2 * (l * 1024 + g) + 1),
    "factor_layer_ignored": ("slice_factor", lambda l, g: 2 * g + 1),
    "factor_head_ignored": ("slice_factor",
                            lambda l, g: 2 * l * O.MAX_KV_HEADS_PER_LAYER + 1),
    "no_truncation": ("num_valid_tokens", lambda pos, bs, n: bs),
    "truncation_off_by_one": ("num_valid_tokens",
                              lambda pos, bs, n: min(bs, max(0, n + 1 - pos * bs))),
    "k_only_pieces": ("pieces_per_token",
                      lambda c: c.head_bytes // 8),
    "nhd_transposed": ("piece_byte_offset", _nhd_transposed),
    "v_then_k": ("piece_byte_offset", _v_then_k),
    "block_id_ignored": ("piece_byte_offset", _block_ignored),
    "xsplit_axes_swapped": ("piece_byte_offset", _xsplit_axes_swapped),
    "sub_blocks_ignored": ("piece_byte_offset", _sub_blocks_ignored),
    "strides_ignored": ("page_start", lambda c, bs, kv, block:
                        (kv * c.num_blocks + block) * O.page_bytes(c, bs)),
    "big_endian": ("read_piece", lambda c, off: int.from_bytes(
        bytes(c.data[off:off + 8]), "big")),
}


def _fails_some_pin():
    for pin in ALL_PINS:
        try:
            pin(py_form)
        except (AssertionError, IndexError, ValueError):
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = _fails_some_pin()
    assert caught is not None, f"mutant {name} passed every pin"


def test_unmutated_passes_all_pins():
    assert _fails_some_pin() is None


def test_missing_mod_reduction_is_caught(monkeypatch):
    orig = O.block_checksum

    def no_mask(caches, bs, block, position, num_tokens):
        nv = O.num_valid_tokens(position, bs, num_tokens)
        c = 0
        for cache in caches:
            for h in range(cache.num_heads):
                s = O.slice_checksum(cache, bs, block, position, nv, h)
                c += O.slice_factor(cache.layer, cache.head_offset + h) * s
        return c

    monkeypatch.setattr(O, "block_checksum", no_mask)
    assert _fails_some_pin() is not None
    monkeypatch.setattr(O, "block_checksum", orig)


TAG_MUTANTS = {
    "tag_big_endian": lambda hs, fp: [int.from_bytes(h[:8], "big") ^ fp for h in hs],
    "tag_last_bytes": lambda hs, fp: [int.from_bytes(h[-8:], "little") ^ fp for h in hs],
    "tag_no_fingerprint": lambda hs, fp: [int.from_bytes(h[:8], "little") for h in hs],
    "tag_four_bytes": lambda hs, fp: [int.from_bytes(h[:4], "little") ^ fp for h in hs],
}


@pytest.mark.parametrize("name", sorted(TAG_MUTANTS))
def test_tag_mutant_is_caught(name, monkeypatch):
    import test_oracle_next1 as T
    monkeypatch.setattr(O, "block_checksum_tags", TAG_MUTANTS[name])
    with pytest.raises(AssertionError):
        T.test_tags_hand_worked()
