"""Pins that tie an oracle form to the definition, not to itself.

Each ``pin_*`` takes ``form(caches, block_size, requests) -> (values,
status)`` and raises ``AssertionError`` when the form disagrees with what the
page "vllm.distributed.kv_transfer.kv_checksum.checksum" and plain arithmetic
fix:

* hand-worked examples (``tests/golden/hand_examples.json``);
* closed forms (constant pieces; a single nonzero piece; all zero);
* brute force from the *logical* token stream: the request-wide slice is
  built as one byte string per (layer, head) and cut into 8-byte pieces,
  so ``j`` is a byte offset / 8 -- a different formulation from the paged
  per-piece indexing the oracle uses;
* the invariants the page states (additivity over block sizes, layout
  independence, TP/PP partials summing to c, sensitivity to a changed piece
  and to data moved to another token, block, head or layer), plus the
  readings for truncation, first positions and bad block ids.

Nothing here calls the oracle's helpers; the expected values are computed
with independent code so a bug shared by a form and a pin is unlikely.
"""

from __future__ import annotations

import dataclasses
import json
import random
from pathlib import Path

import numpy as np
import torch

from helpers import W, OracleCache, OracleRequests, oracle_caches  # noqa: F401

M64 = (1 << 64) - 1
H = 1 << 16
GOLDEN = Path(__file__).resolve().parent / "golden" / "hand_examples.json"
LAYOUTS = {"NHD": W.LAYOUT_NHD, "HND": W.LAYOUT_HND, "LATENT": W.LAYOUT_LATENT}


# ---------------------------------------------------------------------------
# construction helpers (views, not address arithmetic)
# ---------------------------------------------------------------------------

def pool_view(data: np.ndarray, layout: int, nb: int, bs: int, heads: int,
              hb: int) -> np.ndarray:
    """A named-axis view ``[kv, block, slot, head, byte]`` of a pool."""
    if layout == W.LAYOUT_NHD:
        return data.reshape(2, nb, bs, heads, hb)
    if layout == W.LAYOUT_HND:
        return data.reshape(2, nb, heads, bs, hb).transpose(0, 1, 3, 2, 4)
    return data.reshape(1, nb, bs, 1, hb)


def put_piece(view: np.ndarray, half: int, block: int, slot: int, head: int,
              piece: int, value: int) -> None:
    view[half, block, slot, head, 8 * piece:8 * piece + 8] = np.frombuffer(
        int(value).to_bytes(8, "little"), dtype=np.uint8)


def reqs(first_positions, num_tokens, block_id_lists) -> OracleRequests:
    po = [0]
    ids = []
    for b in block_id_lists:
        po.append(po[-1] + len(b))
        ids.extend(b)
    return OracleRequests(po, list(first_positions), list(num_tokens), ids)


def golden_case(ex):
    caches = []
    for c in ex["caches"]:
        layout = LAYOUTS[c["layout"]]
        nb, hb, nh = c["num_blocks"], c["head_bytes"], c["num_heads"]
        halves = 1 if layout == W.LAYOUT_LATENT else 2
        data = np.zeros(halves * nb * ex["block_size"] * nh * hb, dtype=np.uint8)
        v = pool_view(data, layout, nb, ex["block_size"], nh, hb)
        for half, blk, slot, head, piece, value in c["pieces"]:
            put_piece(v, {"K": 0, "V": 1, "row": 0}[half], blk, slot, head,
                      piece, int(value))
        caches.append(OracleCache(data, nb, layout, c["layer"], c["head_offset"],
                                  nh, hb))
    r = ex["requests"]
    return caches, reqs([q["first_position"] for q in r],
                        [q["num_tokens"] for q in r],
                        [q["block_ids"] for q in r])


def random_pool_case(seed, layout, layers=2, heads=2, hb=16, bs=4,
                     lengths=(11,), first_positions=None, extra=None,
                     spare=2, kind=W.BYTES, head_offset=0, layer_numbers=None):
    wl = W.random_case(seed, "cpu", layout=layout, layers=layers, heads=heads,
                       head_bytes=hb, block_size=bs, lengths=list(lengths),
                       first_positions=first_positions, extra_positions=extra,
                       spare_blocks=spare, kind=kind, head_offset=head_offset,
                       layer_numbers=layer_numbers)
    caches = oracle_caches(wl.caches)
    r = OracleRequests(wl.pos_offsets.tolist(), wl.first_position.tolist(),
                       wl.num_tokens.tolist(), wl.block_ids.tolist())
    return wl, caches, r


def logical_case(seed, layouts, layers, heads, hb, bs_list, lengths,
                 latent=False, head_split=None):
    """Random logical KV (per layer ``[T, 2, heads, hb]`` or ``[T, row]``) and
    paged pools of it for every ``(layout, block_size)`` asked for."""
    g = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    tok_off = [0]
    for n in lengths:
        tok_off.append(tok_off[-1] + n)
    if latent:
        logical = [torch.randint(0, 256, (T, hb), dtype=torch.uint8, generator=g)
                   for _ in range(layers)]
    else:
        logical = [torch.randint(0, 256, (T, 2, heads, hb), dtype=torch.uint8,
                                 generator=g) for _ in range(layers)]
    out = {}
    for layout, bs in zip(layouts, bs_list):
        po, fp, nt, bids, nb = W.make_requests(lengths, bs, g, num_blocks=None)
        nb += 1  # one spare block stays zero
        bids = torch.randperm(nb, generator=g)[: int(po[-1])].to(torch.int32)
        caches = []
        for li, lg in enumerate(logical):
            pool = W.scatter_pool(lg, tok_off, bs, layout, bids, po.tolist(), nb)
            nh = 1 if latent else heads
            caches.append(OracleCache(pool.numpy(), nb, layout, li, 0, nh, hb))
        out[(layout, bs)] = (caches, OracleRequests(po.tolist(), fp.tolist(),
                                                    nt.tolist(), bids.tolist()))
    return logical, tok_off, out


def brute_force_stream(logical, tok_off, lengths, bs, latent=False,
                       layer_numbers=None, head_offset=0):
    """c per block position, from each (layer, head)'s request-wide byte
    stream: token by token, K bytes then V bytes (or the latent row)."""
    res = []
    for r, n in enumerate(lengths):
        streams = []
        for li, lg in enumerate(logical):
            rows = lg[tok_off[r]:tok_off[r] + n].numpy()
            lnum = li if layer_numbers is None else layer_numbers[li]
            if latent:
                streams.append((lnum, head_offset, rows.reshape(n, -1).tobytes()))
            else:
                for h in range(rows.shape[2]):
                    per_tok = np.concatenate([rows[:, 0, h, :], rows[:, 1, h, :]], axis=1)
                    streams.append((lnum, head_offset + h, per_tok.tobytes()))
        npos = -(-n // bs)
        for q in range(npos):
            c = 0
            for lnum, g, stream in streams:
                per_token = len(stream) // n
                lo = q * bs * per_token
                hi = min((q + 1) * bs, n) * per_token
                s = 0
                for off in range(lo, hi, 8):
                    j = off // 8
                    s += int.from_bytes(stream[off:off + 8], "little") * (2 * j + 1)
                c += (2 * (lnum * H + g) + 1) * (s % (1 << 64))
            res.append(c % (1 << 64))
    return res


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_hand_examples(form):
    data = json.loads(GOLDEN.read_text())
    for ex in data["examples"]:
        caches, r = golden_case(ex)
        vals, status = form(caches, ex["block_size"], r)
        assert status == 0, ex["name"]
        assert [int(v) for v in vals] == [int(e) for e in ex["expected"]], ex["name"]


def pin_zero(form):
    for layout in (W.LAYOUT_NHD, W.LAYOUT_HND, W.LAYOUT_LATENT):
        _, caches, r = random_pool_case(1, layout, hb=24, lengths=(9, 5))
        zero = [OracleCache(np.zeros_like(c.data), c.num_blocks, c.layout, c.layer,
                            c.head_offset, c.num_heads, c.head_bytes) for c in caches]
        vals, _ = form(zero, 4, r)
        assert all(v == 0 for v in vals)


def pin_constant_pieces(form):
    """Every piece = k: s = k * sum_{j=t0 P}^{t1 P - 1} (2j+1) = k*((t1 P)^2 -
    (t0 P)^2) and c = s * sum m."""
    rng = random.Random(7)
    for layout, hb, heads, bs in ((W.LAYOUT_NHD, 16, 3, 4), (W.LAYOUT_HND, 8, 2, 5),
                                  (W.LAYOUT_LATENT, 24, 1, 3)):
        k = rng.getrandbits(64)
        lengths = [13, 7]
        fps = [0, 1]
        _, caches, r = random_pool_case(2, layout, heads=heads, hb=hb, bs=bs,
                                        lengths=lengths, first_positions=fps,
                                        layer_numbers=[5, 9], head_offset=2)
        piece = np.frombuffer(k.to_bytes(8, "little"), dtype=np.uint8)
        const = [OracleCache(np.tile(piece, c.data.size // 8), c.num_blocks,
                             c.layout, c.layer, c.head_offset, c.num_heads,
                             c.head_bytes) for c in caches]
        vals, _ = form(const, bs, r)
        P = hb // 8 if layout == W.LAYOUT_LATENT else hb // 4
        msum = sum(2 * (c.layer * H + c.head_offset + h) + 1
                   for c in const for h in range(c.num_heads))
        exp = []
        for ri, (n, f) in enumerate(zip(lengths, fps)):
            for i in range(r.pos_offsets[ri + 1] - r.pos_offsets[ri]):
                q = f + i
                t0 = q * bs
                t1 = min(n, t0 + bs)
                t1 = max(t1, t0)
                s = k * ((t1 * P) ** 2 - (t0 * P) ** 2)
                exp.append((s * msum) % (1 << 64))
        assert [int(v) for v in vals] == exp


def pin_single_piece(form):
    """One nonzero piece x at (layer l, global head g, token t, piece p):
    c = x * m(l, g) * (2(tP + p) + 1) at its position, 0 elsewhere; and 0 at
    every position when the piece's slot is at or past num_tokens."""
    rng = random.Random(11)
    for layout, hb, heads in ((W.LAYOUT_NHD, 16, 3), (W.LAYOUT_HND, 24, 2),
                              (W.LAYOUT_LATENT, 32, 1)):
        bs = 4
        n = 14
        _, caches, r = random_pool_case(3, layout, heads=heads, hb=hb, bs=bs,
                                        lengths=[n], layers=2, layer_numbers=[4, 1],
                                        head_offset=5)
        P = hb // 8 if layout == W.LAYOUT_LATENT else hb // 4
        for _ in range(25):
            ci = rng.randrange(2)
            q = rng.randrange(len(r.block_ids))
            slot = rng.randrange(bs)
            h = rng.randrange(heads)
            p = rng.randrange(P)
            x = rng.getrandbits(64) | 1
            zeroed = [OracleCache(np.zeros_like(c.data), c.num_blocks, c.layout,
                                  c.layer, c.head_offset, c.num_heads, c.head_bytes)
                      for c in caches]
            c0 = zeroed[ci]
            v = pool_view(c0.data, layout, c0.num_blocks, bs, c0.num_heads, hb)
            half, piece = (0, p) if (layout == W.LAYOUT_LATENT or p < hb // 8) \
                else (1, p - hb // 8)
            put_piece(v, half, r.block_ids[q], slot, h, piece, x)
            vals, _ = form(zeroed, bs, r)
            t = q * bs + slot
            exp = [0] * len(vals)
            if t < n:
                m = 2 * (c0.layer * H + c0.head_offset + h) + 1
                exp[q] = (x * m * (2 * (t * P + p) + 1)) % (1 << 64)
            assert [int(a) for a in vals] == exp, (layout, ci, q, slot, h, p)


def pin_single_piece_far_position(form):
    """The single-piece closed form at block positions so far into the
    request (first position 2^60 + 3) that t P passes 2^64: the weight
    2(tP + p) + 1 is taken mod 2^64, like every other product."""
    rng = random.Random(12)
    far = (1 << 60) + 3
    for layout, hb, heads in ((W.LAYOUT_NHD, 16, 2), (W.LAYOUT_HND, 24, 2),
                              (W.LAYOUT_LATENT, 32, 1)):
        bs, n = 4, 14
        _, caches, r = random_pool_case(4, layout, heads=heads, hb=hb, bs=bs, lengths=[n],
                                        layers=1, layer_numbers=[7], head_offset=1)
        rf = OracleRequests(r.pos_offsets, [far], [far * bs + n], r.block_ids)
        P = hb // 8 if layout == W.LAYOUT_LATENT else hb // 4
        for _ in range(10):
            q = rng.randrange(len(r.block_ids))
            slot = rng.randrange(bs)
            h = rng.randrange(heads)
            p = rng.randrange(P)
            x = rng.getrandbits(64) | 1
            c0 = OracleCache(np.zeros_like(caches[0].data), caches[0].num_blocks,
                             caches[0].layout, caches[0].layer, caches[0].head_offset,
                             caches[0].num_heads, caches[0].head_bytes)
            v = pool_view(c0.data, layout, c0.num_blocks, bs, c0.num_heads, hb)
            half, piece = (0, p) if (layout == W.LAYOUT_LATENT or p < hb // 8) \
                else (1, p - hb // 8)
            put_piece(v, half, r.block_ids[q], slot, h, piece, x)
            vals, _ = form([c0], bs, rf)
            t = (far + q) * bs + slot
            assert t * P > 1 << 64
            exp = [0] * len(vals)
            if q * bs + slot < n:
                m = 2 * (c0.layer * H + c0.head_offset + h) + 1
                exp[q] = (x * m * (2 * (t * P + p) + 1)) % (1 << 64)
            assert [int(a) for a in vals] == exp, (layout, q, slot, h, p)


def pin_brute_force_stream(form):
    for latent, layouts in ((False, (W.LAYOUT_NHD, W.LAYOUT_HND)), (True, (W.LAYOUT_LATENT,))):
        lengths = [9, 1, 16]
        for bs in (1, 4, 5):
            hb = 24 if latent else 16
            logical, tok_off, cases = logical_case(
                17 + bs, layouts, layers=2, heads=1 if latent else 3, hb=hb,
                bs_list=[bs] * len(layouts), lengths=lengths, latent=latent)
            exp = brute_force_stream(logical, tok_off, lengths, bs, latent=latent)
            for key, (caches, r) in cases.items():
                vals, status = form(caches, bs, r)
                assert status == 0
                assert [int(v) for v in vals] == exp, (key, bs)


def pin_additivity(form):
    """Consecutive blocks' checksums sum to that of the tokens they hold: a
    producer with block_size b and a consumer with 4b agree on every 4 blocks
    (truncated last block included)."""
    lengths = [29, 8, 33]
    logical, tok_off, cases = logical_case(
        23, (W.LAYOUT_NHD, W.LAYOUT_NHD), layers=2, heads=2, hb=8,
        bs_list=(2, 8), lengths=lengths)
    small, _ = form(*_swap(cases[(W.LAYOUT_NHD, 2)], 2))
    big, _ = form(*_swap(cases[(W.LAYOUT_NHD, 8)], 8))
    rs = cases[(W.LAYOUT_NHD, 2)][1]
    rb = cases[(W.LAYOUT_NHD, 8)][1]
    for r in range(len(lengths)):
        sp = [int(v) for v in small[rs.pos_offsets[r]:rs.pos_offsets[r + 1]]]
        bp = [int(v) for v in big[rb.pos_offsets[r]:rb.pos_offsets[r + 1]]]
        for k, v in enumerate(bp):
            assert v == sum(sp[4 * k:4 * k + 4]) % (1 << 64), (r, k)


def _swap(case, bs):
    caches, r = case
    return caches, bs, r


def pin_layout_invariance(form):
    """The same KV in every memory layout gives the same checksums (the
    paragraph on TP ranks and layouts): NHD, HND, HND in kernel sub-blocks of
    1 and 2 slots, x-split ([heads][head_bytes/16][block_size][16]), and NHD
    pages placed by explicit strides (K and V interleaved per block; padded
    blocks).  The other layouts are the NHD pool rearranged by numpy, each
    written from the layout's shape."""
    lengths = [10, 3]
    bs, heads, hb = 4, 3, 32
    _, _, cases = logical_case(29, (W.LAYOUT_NHD,), layers=2, heads=heads, hb=hb,
                               bs_list=(bs,), lengths=lengths)
    caches_n, rn = cases[(W.LAYOUT_NHD, bs)]
    a, _ = form(caches_n, bs, rn)
    assert any(int(x) for x in a)

    def relaid(layout, perm_of, kbs=0):
        out = []
        for c in caches_n:
            v = c.data.reshape(2, c.num_blocks, bs, heads, hb)     # [kv, block, slot, head, byte]
            out.append(OracleCache(np.ascontiguousarray(perm_of(v)).reshape(-1), c.num_blocks,
                                   layout, c.layer, c.head_offset, heads, hb,
                                   kernel_block_size=kbs))
        return out

    variants = [
        relaid(W.LAYOUT_HND, lambda v: v.transpose(0, 1, 3, 2, 4)),
        relaid(W.LAYOUT_XSPLIT, lambda v: v.reshape(2, v.shape[1], bs, heads, hb // 16, 16)
               .transpose(0, 1, 3, 4, 2, 5)),
    ]
    for kbs in (1, 2):
        variants.append(relaid(
            W.LAYOUT_HND, lambda v, k=kbs: v.reshape(2, v.shape[1], bs // k, k, heads, hb)
            .transpose(0, 1, 2, 4, 3, 5), kbs=kbs))
    # explicit strides: K and V interleaved per block ([block][kv][page]),
    # and blocks padded by 24 bytes
    page = bs * heads * hb
    inter = []
    for c in caches_n:
        v = c.data.reshape(2, c.num_blocks, page).transpose(1, 0, 2)
        inter.append(dataclasses.replace(c, data=np.ascontiguousarray(v).reshape(-1),
                                         half_stride=page, block_stride=2 * page))
    variants.append(inter)
    padded = []
    for c in caches_n:
        buf = np.zeros((2, c.num_blocks, page + 24), dtype=np.uint8)
        buf[:, :, :page] = c.data.reshape(2, c.num_blocks, page)
        padded.append(dataclasses.replace(c, data=buf.reshape(-1),
                                          half_stride=c.num_blocks * (page + 24),
                                          block_stride=page + 24))
    variants.append(padded)
    for caches in variants:
        b, _ = form(caches, bs, rn)
        assert [int(x) for x in a] == [int(x) for x in b], caches[0].layout


def pin_tp_pp_partials(form):
    """Partials from TP head shards and PP layer stages sum to c."""
    _, caches, r = random_pool_case(31, W.LAYOUT_NHD, layers=4, heads=4, hb=8,
                                    bs=3, lengths=[10, 4], layer_numbers=[0, 1, 2, 3])
    full, _ = form(caches, 3, r)
    shards = []
    for lo, hi in ((0, 1), (1, 4)):
        part = []
        for c in caches:
            v = pool_view(c.data, c.layout, c.num_blocks, 3, c.num_heads, c.head_bytes)
            sub = np.ascontiguousarray(v[:, :, :, lo:hi, :]).reshape(-1)
            part.append(OracleCache(sub, c.num_blocks, c.layout, c.layer,
                                    c.head_offset + lo, hi - lo, c.head_bytes))
        shards.append([int(x) for x in form(part, 3, r)[0]])
    tp = [(a + b) % (1 << 64) for a, b in zip(*shards)]
    assert tp == [int(x) for x in full]
    pp = [form(caches[:1], 3, r)[0], form(caches[1:], 3, r)[0]]
    assert [(int(a) + int(b)) % (1 << 64) for a, b in zip(*pp)] == [int(x) for x in full]


def pin_first_position(form):
    """A request described from block position f onwards gives the same
    checksums for those positions as the whole request."""
    _, caches, r = random_pool_case(37, W.LAYOUT_HND, layers=2, heads=2, hb=16,
                                    bs=4, lengths=[19])
    full, _ = form(caches, 4, r)
    for f in (1, 3, 4):
        sub = OracleRequests([0, len(r.block_ids) - f], [f], r.num_tokens,
                             r.block_ids[f:])
        part, _ = form(caches, 4, sub)
        assert [int(x) for x in part] == [int(x) for x in full[f:]]


def pin_past_num_tokens(form):
    """Positions wholly at or past num_tokens give 0, even on real data;
    a request with num_tokens 0 gives 0 everywhere."""
    _, caches, r = random_pool_case(41, W.LAYOUT_NHD, layers=1, heads=2, hb=8,
                                    bs=4, lengths=[6, 0], extra=[2, 3], spare=0)
    vals, _ = form(caches, 4, r)
    assert [int(x) for x in vals[2:]] == [0] * (len(vals) - 2)
    assert all(int(x) != 0 for x in vals[:2])


def pin_bad_block_id(form):
    _, caches, r = random_pool_case(43, W.LAYOUT_NHD, layers=2, heads=1, hb=8,
                                    bs=2, lengths=[7], spare=0)
    good, st = form(caches, 2, r)
    assert st == 0
    ids = list(r.block_ids)
    ids[1] = caches[0].num_blocks      # one past the pool
    ids[2] = -1
    bad = OracleRequests(r.pos_offsets, r.first_position, r.num_tokens, ids)
    vals, st = form(caches, 2, bad)
    assert st & 1
    exp = [int(x) for x in good]
    exp[1] = exp[2] = 0
    assert [int(x) for x in vals] == exp


def pin_sensitivity(form):
    """Changing one piece by any nonzero amount changes c (the weights are
    odd); swapped tokens, blocks, heads and layers of unequal data change it
    (the factors are distinct)."""
    bs, hb, heads = 2, 16, 2
    _, caches, r = random_pool_case(47, W.LAYOUT_NHD, layers=2, heads=heads,
                                    hb=hb, bs=bs, lengths=[3], spare=0,
                                    layer_numbers=[0, 1])
    base = [int(x) for x in form(caches, bs, r)[0]]
    P = hb // 4
    valid = [(q, s) for q in range(len(r.block_ids)) for s in range(bs)
             if q * bs + s < 3]
    for ci in range(len(caches)):
        for q, slot in valid:
            for h in range(heads):
                for p in range(P):
                    for delta in (1, 1 << 63, 0x9E3779B97F4A7C15):
                        data = caches[ci].data.copy()
                        v = pool_view(data, W.LAYOUT_NHD, caches[ci].num_blocks,
                                      bs, heads, hb)
                        half, piece = (0, p) if p < hb // 8 else (1, p - hb // 8)
                        blk = r.block_ids[q]
                        old = int.from_bytes(
                            v[half, blk, slot, h, 8 * piece:8 * piece + 8].tobytes(), "little")
                        put_piece(v, half, blk, slot, h, piece, (old + delta) % (1 << 64))
                        mod = list(caches)
                        c = caches[ci]
                        mod[ci] = OracleCache(data, c.num_blocks, c.layout, c.layer,
                                              c.head_offset, c.num_heads, c.head_bytes)
                        vals = [int(x) for x in form(mod, bs, r)[0]]
                        assert vals[q] != base[q], (ci, q, slot, h, p, delta)
                        assert vals[:q] + vals[q + 1:] == base[:q] + base[q + 1:]
    # swapped tokens (slots 0 and 1 of block position 0, all heads of cache 0)
    data = caches[0].data.copy()
    v = pool_view(data, W.LAYOUT_NHD, caches[0].num_blocks, bs, heads, hb)
    b0 = r.block_ids[0]
    v[:, b0, [0, 1]] = v[:, b0, [1, 0]]
    c = caches[0]
    mod = [OracleCache(data, c.num_blocks, c.layout, c.layer, c.head_offset,
                       c.num_heads, c.head_bytes), caches[1]]
    assert int(form(mod, bs, r)[0][0]) != base[0]
    # swapped blocks
    ids = list(r.block_ids)
    ids[0], ids[1] = ids[1], ids[0]
    sw = [int(x) for x in form(caches, bs, OracleRequests(
        r.pos_offsets, r.first_position, r.num_tokens, ids))[0]]
    assert sw[0] != base[0] and sw[1] != base[1]
    # swapped heads
    data = caches[0].data.copy()
    v = pool_view(data, W.LAYOUT_NHD, caches[0].num_blocks, bs, heads, hb)
    v[:, :, :, [0, 1]] = v[:, :, :, [1, 0]]
    mod = [OracleCache(data, c.num_blocks, c.layout, c.layer, c.head_offset,
                       c.num_heads, c.head_bytes), caches[1]]
    sw = [int(x) for x in form(mod, bs, r)[0]]
    assert all(a != b for a, b in zip(sw, base))
    # swapped layers (each cache's data now carries the other layer number)
    c0, c1 = caches
    mod = [OracleCache(c0.data, c0.num_blocks, c0.layout, c1.layer, c0.head_offset,
                       c0.num_heads, c0.head_bytes),
           OracleCache(c1.data, c1.num_blocks, c1.layout, c0.layer, c1.head_offset,
                       c1.num_heads, c1.head_bytes)]
    sw = [int(x) for x in form(mod, bs, r)[0]]
    assert all(a != b for a, b in zip(sw, base))


def pin_token_additivity(form):
    """A block's checksum grows token by token: c with num_tokens = n minus c
    with n - 1 equals c of the same block when only token n - 1's bytes are
    kept (j = t*P + p runs over tokens), for every layout."""
    for layout, hb in ((W.LAYOUT_NHD, 16), (W.LAYOUT_HND, 8), (W.LAYOUT_LATENT, 24)):
        bs = 4
        _, caches, r = random_pool_case(53, layout, layers=2, heads=2 if layout != 2 else 1,
                                        hb=hb, bs=bs, lengths=[11], spare=0)
        for n in range(1, 12):
            q = (n - 1) // bs                       # block position of token n-1
            blk = r.block_ids[q]
            one = OracleRequests([0, 1], [q], [n], [blk])
            prev = OracleRequests([0, 1], [q], [n - 1], [blk])
            cn = int(form(caches, bs, one)[0][0])
            cp = int(form(caches, bs, prev)[0][0])
            kept = []
            for c in caches:
                d = np.zeros_like(c.data)
                v_src = pool_view(c.data, c.layout, c.num_blocks, bs, c.num_heads, c.head_bytes)
                v_dst = pool_view(d, c.layout, c.num_blocks, bs, c.num_heads, c.head_bytes)
                v_dst[:, blk, (n - 1) % bs] = v_src[:, blk, (n - 1) % bs]
                kept.append(OracleCache(d, c.num_blocks, c.layout, c.layer, c.head_offset,
                                        c.num_heads, c.head_bytes))
            ct = int(form(kept, bs, one)[0][0])
            assert (cn - cp) % (1 << 64) == ct, (layout, n)


ALL_PINS = [pin_hand_examples, pin_zero, pin_constant_pieces, pin_single_piece,
            pin_single_piece_far_position, pin_brute_force_stream, pin_additivity, pin_layout_invariance,
            pin_tp_pp_partials, pin_first_position, pin_past_num_tokens,
            pin_bad_block_id, pin_sensitivity, pin_token_additivity]
