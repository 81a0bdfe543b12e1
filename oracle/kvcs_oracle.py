"""Pure-Python oracle for the connector-agnostic KV-cache block checksum.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library (no headers, helpers or tables).

It is written straight from the definition on the page
"vllm.distributed.kv_transfer.kv_checksum.checksum" (vLLM API docs), module
docstring items 1 and 2, the attributes ``MAX_KV_HEADS_PER_LAYER`` and
``BLOCK_CHECKSUM_BYTES``, the dataclass ``KVChecksumBlocks`` and the function
``num_valid_tokens`` described there.  Every integer is an exact Python int,
reduced mod 2**64 only where the definition says "mod 2**64", so this form is
the slow, obviously-correct ground truth for small inputs.

Definition restated in this module's words (same page, module docstring):

* For each (layer, KV head) pair, a block holds one *slice*.  Its bytes are,
  for each token of the block in turn, that head's K bytes followed by its V
  bytes.  Reading them as consecutive little-endian 64-bit words gives the
  pieces; the word ``p`` of the token at request position ``t`` has index
  ``j = t*P + p``, with ``P`` words per token.
* ``s = sum_j x_j * (2*j + 1) mod 2**64``  (item 1).
* ``c = sum_{layer, head} m * s mod 2**64`` with
  ``m = 2*(layer*H + head) + 1`` and ``H = MAX_KV_HEADS_PER_LAYER = 1 << 16``
  (item 2; the attribute list of the same page).
* A slot whose token index is ``num_tokens`` or more contributes nothing
  (dataclass ``KVChecksumBlocks``, field ``num_tokens``).

Readings where the page is silent:

* Latent (MLA) caches hold one row per token and count as a single KV head
  (global head ``head_offset``) whose token slice is the whole row: there is
  no K/V split, so ``P = row_bytes / 8``.
* A block id outside ``[0, num_blocks)`` of any cache makes that position's
  checksum 0 and sets bit ``STATUS_BAD_BLOCK_ID`` in the returned status.
* Per-token bytes that are not a multiple of 8, and layers with more than
  ``H`` KV heads, are rejected (the page excludes such groups from
  checksumming).
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

import numpy as np

MASK64 = (1 << 64) - 1

# H in the slice factor (attribute MAX_KV_HEADS_PER_LAYER = 1 << 16).
MAX_KV_HEADS_PER_LAYER = 1 << 16

# Bytes of one block's checksum (attribute BLOCK_CHECKSUM_BYTES = 8).
BLOCK_CHECKSUM_BYTES = 8

LAYOUT_NHD = 0     # pool [2, num_blocks, block_size, num_heads, head_bytes]
LAYOUT_HND = 1     # pool [2, num_blocks, num_heads, block_size, head_bytes], or with
                   # kernel sub-blocks [2, num_blocks, block_size / kbs, num_heads, kbs,
                   # head_bytes]
LAYOUT_LATENT = 2  # pool [num_blocks, block_size, row_bytes]
LAYOUT_XSPLIT = 3  # pool [2, num_blocks, num_heads, head_bytes / 16, block_size, 16]
LAYOUT_STATE = 4   # pool [num_blocks, rows, row_bytes]: Mamba running state

STATUS_BAD_BLOCK_ID = 1


@dataclass(frozen=True)
class OracleCache:
    """One layer's paged KV pool on the host, as raw bytes.

    ``data`` is a C-contiguous uint8 array holding the whole pool in the order
    given by ``layout``.  ``head_bytes`` is the bytes of one head's K (equal to
    its V) for one token; for ``LAYOUT_LATENT`` it is the bytes of one token's
    latent row and ``num_heads`` must be 1.

    ``LAYOUT_STATE`` holds a Mamba layer's running state, one block per
    request: ``num_heads`` local rows (the TP-split dimension) of
    ``head_bytes`` bytes, whose pieces are ``piece_bytes``-byte elements
    (2 or 4); ``head_offset`` is the global index of local row 0.  A state
    whose split is unknown is one row per TP shard (``head_offset`` = the
    shard index).
    """

    data: np.ndarray
    num_blocks: int
    layout: int
    layer: int
    head_offset: int
    num_heads: int
    head_bytes: int
    piece_bytes: int = 8
    kernel_block_size: int = 0   # HND: slots per kernel sub-block (0: none)
    half_stride: int = 0         # bytes from a block's K page to its V page (0: packed)
    block_stride: int = 0        # bytes between blocks' pages (0: packed)


@dataclass(frozen=True)
class OracleRequests:
    """Requests in CSR form.

    Request ``r`` owns global position indices
    ``pos_offsets[r] <= i < pos_offsets[r+1]``; index ``i`` is block position
    ``first_position[r] + (i - pos_offsets[r])`` of the request and holds block
    ``block_ids[i]``.  This is the page's dataclass ``KVChecksumBlocks`` for
    one KV cache group, flattened over requests.
    """

    pos_offsets: Sequence[int]
    first_position: Sequence[int]
    num_tokens: Sequence[int]
    block_ids: Sequence[int]


def num_valid_tokens(position: int, block_size: int, num_tokens: int) -> int:
    """Count of the block's slots that carry a token (function
    ``num_valid_tokens``): slot ``slot`` of block ``position`` is token
    ``position*block_size + slot``, and only tokens below ``num_tokens``
    exist."""
    return sum(1 for slot in range(block_size)
               if token_position(position, block_size, slot) < num_tokens)


def pieces_per_token(cache: OracleCache) -> int:
    """``P``: a token's slice is its K bytes then its V bytes for one head
    (module docstring, item 1), or its latent row."""
    if cache.layout == LAYOUT_LATENT:
        return cache.head_bytes // 8
    return 2 * cache.head_bytes // 8


def piece_byte_offset(cache: OracleCache, block_size: int, block: int,
                      slot: int, head: int, p: int) -> int:
    """Byte offset in ``cache.data`` of piece ``p`` of slot ``slot``'s slice
    for local head ``head`` in physical block ``block``.

    The logical order (K bytes then V bytes of the head, token by token) is
    fixed by the definition; the memory order comes from the declared layout
    (page "【vLLM 源码解析】KV Cache": section "reshape kv_cache" for the
    block-size split into kernel blocks, section on reshape_and_cache for the
    key layout with x elements of 16 bytes, here read for K and V alike).
    """
    hb = cache.head_bytes
    byte = 8 * p
    kv = 0
    if cache.layout != LAYOUT_LATENT and byte >= hb:
        kv, byte = 1, byte - hb
    base = page_start(cache, block_size, kv, block)
    if cache.layout == LAYOUT_LATENT:
        return base + slot * hb + byte
    if cache.layout == LAYOUT_NHD:
        return base + (slot * cache.num_heads + head) * hb + byte
    if cache.layout == LAYOUT_HND:
        kbs = cache.kernel_block_size or block_size
        sub, within = divmod(slot, kbs)
        return base + ((sub * cache.num_heads + head) * kbs + within) * hb + byte
    if cache.layout == LAYOUT_XSPLIT:
        chunk, inner = divmod(byte, 16)
        return base + ((head * (hb // 16) + chunk) * block_size + slot) * 16 + inner
    raise ValueError(f"unknown layout {cache.layout}")


def page_bytes(cache: OracleCache, block_size: int) -> int:
    """Bytes of one page: one block's K, its V, or its latent rows."""
    return block_size * cache.num_heads * cache.head_bytes


def page_start(cache: OracleCache, block_size: int, kv: int, block: int) -> int:
    """Byte offset of the page holding half ``kv`` (0: K, 1: V) of ``block``:
    by default the pool is all K pages then all V pages; explicit strides
    place a block's pages anywhere (e.g. K and V interleaved per block, or
    padded blocks)."""
    page = page_bytes(cache, block_size)
    half = cache.half_stride or cache.num_blocks * page
    stride = cache.block_stride or page
    return kv * half + block * stride


def read_piece(cache: OracleCache, offset: int) -> int:
    """Little-endian unsigned 8-byte piece at ``offset``."""
    return int.from_bytes(bytes(cache.data[offset:offset + 8]), "little")


def token_position(position: int, block_size: int, slot: int) -> int:
    """``t``: the token's position in the request; block ``position`` holds
    tokens ``position*block_size`` onwards (function ``num_valid_tokens``)."""
    return position * block_size + slot


def piece_index(t: int, P: int, p: int) -> int:
    """``j = t*P + p`` (module docstring, item 1)."""
    return t * P + p


def piece_weight(j: int) -> int:
    """The odd weight ``2*j + 1`` of piece ``j`` (item 1)."""
    return 2 * j + 1


def slice_checksum(cache: OracleCache, block_size: int, block: int,
                   position: int, nv: int, head: int) -> int:
    """``s = sum_j x_j*(2j+1) mod 2**64`` over the first ``nv`` slots of the
    block for one (layer, local head) slice (item 1)."""
    P = pieces_per_token(cache)
    s = 0
    for slot in range(nv):
        t = token_position(position, block_size, slot)
        for p in range(P):
            x = read_piece(cache, piece_byte_offset(cache, block_size, block,
                                                    slot, head, p))
            s += x * piece_weight(piece_index(t, P, p))
    return s & MASK64


def slice_factor(layer: int, global_head: int) -> int:
    """``m = 2*(layer*H + head) + 1`` (item 2)."""
    return 2 * (layer * MAX_KV_HEADS_PER_LAYER + global_head) + 1


def check_cache(cache: OracleCache, block_size: int) -> None:
    """Reject what the definition does not cover (see module docstring)."""
    if cache.layout == LAYOUT_STATE:
        if cache.piece_bytes not in (2, 4) or cache.head_bytes <= 0 or \
                cache.head_bytes % cache.piece_bytes:
            raise ValueError("state rows are whole 2- or 4-byte elements")
        if cache.head_offset < 0 or cache.num_heads < 1 or \
                cache.head_offset + cache.num_heads > MAX_KV_HEADS_PER_LAYER:
            raise ValueError("bad row range")
        if cache.block_stride < 0:
            raise ValueError("strides are byte offsets within the one pool array")
        state = cache.num_heads * cache.head_bytes
        need = 0
        if cache.num_blocks > 0:
            need = (cache.num_blocks - 1) * (cache.block_stride or state) + state
        if cache.data.size < need:
            raise ValueError("pool smaller than its declared geometry")
        return
    if cache.head_bytes <= 0 or cache.head_bytes % 8:
        raise ValueError("per-token bytes must be a positive multiple of 8")
    if cache.layout == LAYOUT_LATENT and cache.num_heads != 1:
        raise ValueError("a latent cache has exactly one head")
    if cache.layout == LAYOUT_XSPLIT and cache.head_bytes % 16:
        raise ValueError("x-split heads are whole 16-byte chunks")
    if cache.kernel_block_size and (cache.layout != LAYOUT_HND or
                                    cache.kernel_block_size < 0 or
                                    block_size % cache.kernel_block_size):
        raise ValueError("kernel blocks split an HND block evenly")
    if cache.layout not in (LAYOUT_NHD, LAYOUT_HND, LAYOUT_LATENT, LAYOUT_XSPLIT):
        raise ValueError(f"unknown layout {cache.layout}")
    if cache.head_offset < 0 or cache.num_heads < 1:
        raise ValueError("bad head range")
    if cache.head_offset + cache.num_heads > MAX_KV_HEADS_PER_LAYER:
        raise ValueError("a layer with more than H KV heads is excluded")
    if cache.half_stride < 0 or cache.block_stride < 0:
        raise ValueError("strides are byte offsets within the one pool array")
    halves = 1 if cache.layout == LAYOUT_LATENT else 2
    need = 0
    if cache.num_blocks > 0:
        need = page_start(cache, block_size, halves - 1, cache.num_blocks - 1) + \
            page_bytes(cache, block_size)
    if cache.data.size < need:
        raise ValueError("pool smaller than its declared geometry")


def state_piece(cache: OracleCache, block: int, row: int, p: int) -> int:
    """Element ``p`` of local row ``row`` of a state block, read unsigned."""
    w = cache.piece_bytes
    stride = cache.block_stride or cache.num_heads * cache.head_bytes
    off = block * stride + row * cache.head_bytes + w * p
    return int.from_bytes(bytes(cache.data[off:off + w]), "little")


def state_slice_checksum(cache: OracleCache, block: int, row: int) -> int:
    """``s`` of one global row of a Mamba state (paragraph on Mamba state):
    the row's elements are its pieces; the state is not per token, so the
    piece index is the element index."""
    s = 0
    for p in range(cache.head_bytes // cache.piece_bytes):
        s += state_piece(cache, block, row, p) * piece_weight(p)
    return s & MASK64


def block_checksum(caches: Sequence[OracleCache], block_size: int, block: int,
                   position: int, num_tokens: int) -> int:
    """``c = sum_{layer, head} m*s mod 2**64`` for block ``block`` at block
    position ``position`` of a request with ``num_tokens`` tokens (item 2).
    A Mamba state block lives at position 0 only (paragraph on Mamba state);
    its rows are its slices."""
    nv = num_valid_tokens(position, block_size, num_tokens)
    c = 0
    for cache in caches:
        if cache.layout == LAYOUT_STATE:
            if position != 0:
                continue
            for r in range(cache.num_heads):
                s = state_slice_checksum(cache, block, r)
                c += slice_factor(cache.layer, cache.head_offset + r) * s
            continue
        for h in range(cache.num_heads):
            s = slice_checksum(cache, block_size, block, position, nv, h)
            c += slice_factor(cache.layer, cache.head_offset + h) * s
    return c & MASK64


def block_checksums(caches: Sequence[OracleCache], block_size: int,
                    requests: OracleRequests) -> tuple[list[int], int]:
    """One uint64 per global position index, plus a status word.

    Positions whose block id is outside ``[0, num_blocks)`` of some cache give
    0 and set ``STATUS_BAD_BLOCK_ID``.
    """
    if block_size <= 0:
        raise ValueError("block_size must be positive")
    for cache in caches:
        check_cache(cache, block_size)
    po = list(requests.pos_offsets)
    total = po[-1] if po else 0
    if not po or po[0] != 0 or any(b < a for a, b in zip(po, po[1:])):
        raise ValueError("pos_offsets must start at 0 and not decrease")
    if len(requests.block_ids) < total:
        raise ValueError("fewer block ids than positions")
    out = [0] * total
    status = 0
    for r in range(len(po) - 1):
        for i in range(po[r], po[r + 1]):
            position = requests.first_position[r] + (i - po[r])
            block = int(requests.block_ids[i])
            if any(block < 0 or block >= c.num_blocks for c in caches):
                status |= STATUS_BAD_BLOCK_ID
                continue
            out[i] = block_checksum(caches, block_size, block, position,
                                    requests.num_tokens[r])
    return out, status


def combine_partials(parts: Sequence[Sequence[int]]) -> list[int]:
    """Partials from TP ranks and PP stages sum to ``c`` (module docstring,
    the paragraph on TP ranks and PP stages): element-wise sum mod 2**64."""
    return [sum(col) & MASK64 for col in zip(*parts)]


# ---------------------------------------------------------------------------
# Replica-key columns, offload row sums and block tags
# ---------------------------------------------------------------------------

def column_checksums(caches: Sequence[OracleCache], columns: Sequence[int],
                     num_columns: int, block_size: int,
                     requests: OracleRequests) -> tuple[list[list[int]], int]:
    """``values[i][k]``: the partial checksum of position ``i`` over the
    caches whose replica-key column is ``k`` (paragraph on replicated KV:
    one partial per key of the layers it covers; dataclass
    ``KVChecksumGroup``, field ``values``)."""
    total = requests.pos_offsets[-1] if requests.pos_offsets else 0
    values = [[0] * num_columns for _ in range(total)]
    status = 0
    for k in range(num_columns):
        sub = [c for c, col in zip(caches, columns) if col == k]
        vals, st = block_checksums(sub, block_size, requests)
        status |= st
        for i, v in enumerate(vals):
            values[i][k] = v
    return values, status


def row_sums(values: Sequence[Sequence[int]], tags: Sequence[int] | None = None) -> list[int]:
    """A row's partial checksums summed mod 2**64 (dataclass
    ``KVChecksumGroup``, field ``stored``), XORed with the block's tag when
    one is given (function ``block_checksum_tags``)."""
    out = []
    for i, row in enumerate(values):
        r = sum(row) & MASK64
        if tags is not None:
            r ^= tags[i]
        out.append(r)
    return out


def block_checksum_tags(block_hashes: Sequence[bytes], fingerprint: int) -> list[int]:
    """Per block, the 64-bit word an offloaded checksum is XORed with
    (function ``block_checksum_tags``): the first eight bytes of the block's
    hash read as a little-endian unsigned integer, XOR the group's
    fingerprint."""
    tags = []
    for h in block_hashes:
        word = 0
        for k in range(8):
            word += h[k] * (256 ** k)
        tags.append(word ^ (fingerprint & MASK64))
    return tags
