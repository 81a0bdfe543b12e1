"""Seeded synthetic paged-KV workloads.

This module builds inputs only: raw paged KV pools and per-request block
tables.  It holds none of the checksum's arithmetic, so both the CUDA path
(through the binding) and the CPU oracle (in the tests and the benchmark's
CPU baseline) can consume the same inputs.

Paged layout (page "【vLLM 源码解析】KV Cache", sections "地址划分" and
"reshape kv_cache"): one contiguous byte pool per layer, viewed as
``[2 (K/V), num_blocks, block_size, num_kv_heads, head_size]`` (NHD), with
each request's blocks scattered through the pool by its block table.  HND
swaps the two middle axes; a latent (MLA) pool is
``[num_blocks, block_size, row]`` with no K/V axis.

Randomness: the structure (request lengths, block-id permutations) always
comes from a CPU ``torch.Generator`` seeded with ``seed``, so it is identical
whatever device the pools live on; the pool bytes come from a generator on the
pool's device seeded with ``seed + 1``.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Sequence

import torch

LAYOUT_NHD = 0
LAYOUT_HND = 1
LAYOUT_LATENT = 2
LAYOUT_XSPLIT = 3   # [2, num_blocks, heads, head_bytes / 16, block_size, 16]
LAYOUT_STATE = 4    # [num_blocks, rows, row_bytes]: Mamba running state

# Value recipes for pool bytes.  Every one produces raw bits that are only
# ever read back as bytes.
BF16_NORMAL = "bf16_normal"   # torch.randn in bfloat16
BITS16 = "bits16"             # uniform random 16-bit patterns
BYTES = "bytes"               # uniform random bytes (fp8 e4m3 storage)


@dataclass
class CacheSpec:
    """One layer's pool: raw bytes plus the geometry the checksum needs."""

    pool: torch.Tensor      # uint8, contiguous, the whole pool
    num_blocks: int
    layout: int
    layer: int
    head_offset: int
    num_heads: int
    head_bytes: int         # K (= V) bytes per head per token; latent: row bytes
    column: int = 0         # replica-key column (several-key outputs only)
    half_stride: int = 0    # bytes from a block's K page to its V page (0: packed)
    block_stride: int = 0   # bytes between blocks' pages (0: packed)
    kernel_block_size: int = 0  # HND sub-block slots (0: none)
    v_pool: torch.Tensor | None = None  # separate V tensor, if any
    piece_bytes: int = 0    # state element bytes (2 or 4); 0 for KV caches


@dataclass
class Workload:
    """Caches of one KV-cache group plus the requests to checksum."""

    name: str
    block_size: int
    caches: list[CacheSpec]
    pos_offsets: torch.Tensor      # int64 [R+1]
    first_position: torch.Tensor   # int64 [R]
    num_tokens: torch.Tensor       # int64 [R]
    block_ids: torch.Tensor        # int32 [pos_offsets[R]]
    info: dict = field(default_factory=dict)

    @property
    def num_positions(self) -> int:
        return int(self.pos_offsets[-1])

    @property
    def num_requests(self) -> int:
        return int(self.pos_offsets.numel() - 1)


def gather_pages(cache: CacheSpec, block_size: int, ids: torch.Tensor) -> torch.Tensor:
    """The pages of blocks ``ids`` of one cache, packed one after another:
    uint8 ``[halves, len(ids), page]`` on the pool's device (data movement
    only).  Pages are found the way the cache places them: default packing,
    explicit half/block strides, or a separate V tensor."""
    state = cache.layout == LAYOUT_STATE
    halves = 1 if cache.layout in (LAYOUT_LATENT, LAYOUT_STATE) else 2
    page = (1 if state else block_size) * cache.num_heads * cache.head_bytes
    bstride = cache.block_stride or page
    ids = ids.to(cache.pool.device, torch.int64)
    if cache.v_pool is not None:
        return torch.stack([torch.as_strided(t, (cache.num_blocks, page), (bstride, 1))[ids]
                            for t in (cache.pool, cache.v_pool)])
    hstride = cache.half_stride or cache.num_blocks * page
    view = torch.as_strided(cache.pool, (halves, cache.num_blocks, page), (hstride, bstride, 1))
    return view[:, ids]


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device: torch.device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    return g


def fill_bytes(nbytes: int, kind: str, gen: torch.Generator,
               device: torch.device) -> torch.Tensor:
    """``nbytes`` of seeded raw bytes following recipe ``kind``."""
    if kind == BYTES:
        return torch.randint(0, 256, (nbytes,), dtype=torch.uint8,
                             generator=gen, device=device)
    if nbytes % 2:
        raise ValueError("16-bit recipes need an even byte count")
    if kind == BF16_NORMAL:
        v = torch.randn((nbytes // 2,), dtype=torch.bfloat16, generator=gen,
                        device=device)
    elif kind == BITS16:
        v = torch.randint(-32768, 32768, (nbytes // 2,), dtype=torch.int16,
                          generator=gen, device=device)
    else:
        raise ValueError(f"unknown recipe {kind}")
    return v.view(torch.uint8)


def pool_bytes(layout: int, num_blocks: int, block_size: int, num_heads: int,
               head_bytes: int) -> int:
    halves = 1 if layout == LAYOUT_LATENT else 2
    return halves * num_blocks * block_size * num_heads * head_bytes


def blocks_per_request(lengths: Sequence[int], block_size: int,
                       first_positions: Sequence[int] | None = None) -> list[int]:
    """Block positions each request covers: from its first position up to
    the block that holds its last token (at least one when it has tokens)."""
    fp = first_positions or [0] * len(lengths)
    out = []
    for n, f in zip(lengths, fp):
        last = -(-n // block_size)  # positions [0, last) hold the n tokens
        out.append(max(0, last - f))
    return out


def make_requests(lengths: Sequence[int], block_size: int, gen: torch.Generator,
                  num_blocks: int | None = None,
                  first_positions: Sequence[int] | None = None,
                  extra_positions: Sequence[int] | None = None):
    """CSR request tables with block ids drawn as a seeded permutation of the
    pool (so no block is shared), optionally with extra positions past the
    request's tokens (their checksums must come out 0).

    Returns ``(pos_offsets, first_position, num_tokens, block_ids, num_blocks)``
    as CPU tensors; ``num_blocks`` defaults to the number of positions.
    """
    nreq = len(lengths)
    fp = list(first_positions) if first_positions is not None else [0] * nreq
    extra = list(extra_positions) if extra_positions is not None else [0] * nreq
    counts = [c + e for c, e in zip(blocks_per_request(lengths, block_size, fp), extra)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    total = offsets[-1]
    nb = total if num_blocks is None else num_blocks
    if nb < total:
        raise ValueError("pool smaller than the positions to fill")
    perm = torch.randperm(nb, generator=gen)[:total].to(torch.int32)
    return (torch.tensor(offsets, dtype=torch.int64),
            torch.tensor(fp, dtype=torch.int64),
            torch.tensor(list(lengths), dtype=torch.int64),
            perm, nb)


def _build(name: str, seed: int, device, *, layers: int, heads: int,
           head_bytes: int, block_size: int, lengths: Sequence[int],
           layout: int = LAYOUT_NHD, kind: str = BF16_NORMAL,
           first_positions: Sequence[int] | None = None,
           extra_positions: Sequence[int] | None = None,
           spare_blocks: int = 0, layer_numbers: Sequence[int] | None = None,
           head_offset: int = 0) -> Workload:
    device = torch.device(device)
    g = _cpu_gen(seed)
    po, fp, nt, bids, _ = make_requests(lengths, block_size, g,
                                        first_positions=first_positions,
                                        extra_positions=extra_positions)
    nb = int(po[-1]) + spare_blocks
    if spare_blocks:
        bids = torch.randperm(nb, generator=g)[: int(po[-1])].to(torch.int32)
    dg = _dev_gen(seed, device)
    nheads = 1 if layout == LAYOUT_LATENT else heads
    lnum = list(layer_numbers) if layer_numbers is not None else list(range(layers))
    caches = []
    for li in range(layers):
        nbytes = pool_bytes(layout, nb, block_size, nheads, head_bytes)
        pool = fill_bytes(nbytes, kind, dg, device)
        caches.append(CacheSpec(pool, nb, layout, lnum[li], head_offset,
                                nheads, head_bytes))
    return Workload(name, block_size, caches, po.to(device), fp.to(device),
                    nt.to(device), bids.to(device),
                    info=dict(layers=layers, heads=nheads, head_bytes=head_bytes,
                              block_size=block_size, kind=kind, layout=layout,
                              requests=len(lengths), seed=seed))


def tiny(seed: int = 0, device="cpu") -> Workload:
    """2 layers, 2 KV heads, head_size 64 (bf16: 128 B), uniform random
    16-bit patterns, block_size 16, NHD ``[2, 16, 16, 2, 64]`` per layer, one
    request of 100 tokens (7 block positions, the last partial) on a seeded
    shuffle of the 16-page pool; P = 32 pieces per token."""
    return _build("tiny", seed, device, layers=2, heads=2, head_bytes=128,
                  block_size=16, lengths=[100], kind=BITS16, spare_blocks=9)


def llama3_8b(seed: int = 0, device="cpu", num_requests: int = 64,
              min_len: int = 512, max_len: int = 4096, layers: int = 32) -> Workload:
    """Llama-3-8B-shaped paged KV: 32 layers, 8 KV heads, head_size 128,
    bf16 normal(0,1), block_size 16, NHD ``[2, num_blocks, 16, 8, 128]`` per
    layer, ``num_requests`` requests with lengths uniform in
    ``[min_len, max_len]``, block ids a seeded permutation of the pool."""
    g = _cpu_gen(seed + 1000)
    lengths = torch.randint(min_len, max_len + 1, (num_requests,), generator=g).tolist()
    return _build("llama3_8b", seed, device, layers=layers, heads=8,
                  head_bytes=256, block_size=16, lengths=lengths, kind=BF16_NORMAL)


def mla(seed: int = 0, device="cpu", num_requests: int = 32,
        tokens: int = 8192, layers: int = 61) -> Workload:
    """DeepSeek-V3-shaped MLA cache: 61 layers, one latent row per token of
    576 bf16 (512 kv_lora + 64 rope; 1152 B) as uniform random bits,
    block_size 64, ``num_requests`` requests of ``tokens`` tokens; P = 144."""
    return _build("mla", seed, device, layers=layers, heads=1, head_bytes=1152,
                  block_size=64, lengths=[tokens] * num_requests,
                  layout=LAYOUT_LATENT, kind=BITS16)


def llama3_70b(seed: int = 0, device="cpu", num_requests: int = 128,
               tokens: int = 2048, layers: int = 80) -> Workload:
    """Llama-3-70B-shaped: 80 layers, 8 KV heads, head_size 128 in fp8 e4m3
    (random bytes; 128 B per head), block_size 16, ``num_requests`` requests
    of ``tokens`` tokens."""
    return _build("llama3_70b", seed, device, layers=layers, heads=8,
                  head_bytes=128, block_size=16, lengths=[tokens] * num_requests,
                  kind=BYTES)


def llama3_8b_decode(seed: int = 0, device="cpu", num_requests: int = 16384,
                     layout: int = LAYOUT_HND) -> Workload:
    """Decode-shaped checksums of freshly appended blocks: Llama-3-8B
    geometry (32 layers, 8 KV heads, head_size 128 bf16 ``randn``, block_size
    16), ``num_requests`` requests of ``16 k + 1`` tokens with ``k`` uniform
    in [32, 255], each listing only its newest block (position ``k``), which
    holds one token."""
    g = _cpu_gen(seed + 2000)
    ks = torch.randint(32, 256, (num_requests,), generator=g).tolist()
    return _build("llama3_8b_decode", seed, device, layers=32, heads=8, head_bytes=256,
                  block_size=16, lengths=[16 * k + 1 for k in ks], layout=layout,
                  kind=BF16_NORMAL, first_positions=ks)


def random_case(seed: int, device="cpu", *, layout: int = LAYOUT_NHD,
                layers: int = 2, heads: int = 2, head_bytes: int = 32,
                block_size: int = 16, lengths: Sequence[int] = (37,),
                first_positions: Sequence[int] | None = None,
                extra_positions: Sequence[int] | None = None,
                spare_blocks: int = 3, kind: str = BYTES,
                layer_numbers: Sequence[int] | None = None,
                head_offset: int = 0) -> Workload:
    """A small seeded case of any geometry, for parity and edge tests."""
    return _build("random", seed, device, layers=layers, heads=heads,
                  head_bytes=head_bytes, block_size=block_size, lengths=lengths,
                  layout=layout, kind=kind, first_positions=first_positions,
                  extra_positions=extra_positions, spare_blocks=spare_blocks,
                  layer_numbers=layer_numbers, head_offset=head_offset)


# ---------------------------------------------------------------------------
# Logical KV and scatter into several paged layouts (the invariance workload)
# ---------------------------------------------------------------------------

def logical_kv(total_tokens: int, heads: int, head_bytes: int, kind: str,
               gen: torch.Generator, device) -> torch.Tensor:
    """uint8 ``[total_tokens, 2 (K/V), heads, head_bytes]`` for one layer."""
    n = total_tokens * 2 * heads * head_bytes
    return fill_bytes(n, kind, gen, device).view(total_tokens, 2, heads, head_bytes)


def scatter_pool(logical: torch.Tensor, token_offsets: Sequence[int],
                 block_size: int, layout: int, block_ids: torch.Tensor,
                 pos_offsets: Sequence[int], num_blocks: int,
                 heads: slice | None = None) -> torch.Tensor:
    """Write one layer's logical KV (requests concatenated; request r's tokens
    start at ``token_offsets[r]``; ``[T, 2, heads, head_bytes]``, or
    ``[T, row_bytes]`` for a latent pool) into a fresh paged pool, through the
    request's block table: token t of request r goes to slot ``t % bs`` of
    block ``block_ids[pos_offsets[r] + t // bs]``.  Unwritten slots stay 0.
    ``heads`` selects a head range (a simulated TP shard)."""
    if layout == LAYOUT_LATENT:
        lg = logical
        T, hb = lg.shape
        H = 1
    else:
        lg = logical if heads is None else logical[:, :, heads, :]
        T, _, H, hb = lg.shape
    dev = lg.device
    pool = torch.zeros(pool_bytes(layout, num_blocks, block_size, H, hb),
                       dtype=torch.uint8, device=dev)
    nreq = len(token_offsets) - 1
    tok_req = torch.repeat_interleave(
        torch.arange(nreq, device=dev),
        torch.tensor([token_offsets[r + 1] - token_offsets[r] for r in range(nreq)],
                     device=dev))
    starts = torch.tensor(list(token_offsets[:-1]), device=dev, dtype=torch.int64)
    t_in_req = torch.arange(T, device=dev, dtype=torch.int64) - starts[tok_req]
    po = torch.tensor(list(pos_offsets), device=dev, dtype=torch.int64)
    blk = block_ids.to(dev, torch.int64)[po[tok_req] + t_in_req // block_size]
    slot = t_in_req % block_size
    if layout == LAYOUT_NHD:
        view = pool.view(2, num_blocks, block_size, H, hb)
        for kv in range(2):
            view[kv, blk, slot] = lg[:, kv]
    elif layout == LAYOUT_HND:
        view = pool.view(2, num_blocks, H, block_size, hb)
        for kv in range(2):
            view[kv, blk, :, slot] = lg[:, kv]
    else:
        view = pool.view(num_blocks, block_size, hb)
        view[blk, slot] = lg
    return pool


def invariance(seed: int = 0, device="cpu", num_requests: int = 16,
               tokens: int = 3000, layers: int = 32, heads: int = 8,
               head_bytes: int = 256, kind: str = BF16_NORMAL,
               producer_bs: int = 16, consumer_bs: int = 64):
    """The same logical KV written three ways: producer ``producer_bs`` NHD,
    consumer ``consumer_bs`` HND, and two simulated TP shards (heads
    ``[0, heads/2)`` and ``[heads/2, heads)``) in separate NHD pools with
    global head offsets ``0`` and ``heads/2``.

    Returns ``(producer, consumer, shard0, shard1)`` workloads.  Each has its
    own seeded block-id permutation; the shards share theirs, as TP ranks of
    one instance share a block table.
    """
    device = torch.device(device)
    g = _cpu_gen(seed)
    dg = _dev_gen(seed, device)
    lengths = [tokens] * num_requests
    tok_off = [r * tokens for r in range(num_requests + 1)]
    tables = {}
    for key, bs in (("producer", producer_bs), ("consumer", consumer_bs),
                    ("shard", producer_bs)):
        tables[key] = make_requests(lengths, bs, g)
    half = heads // 2
    out = {k: [] for k in ("producer", "consumer", "shard0", "shard1")}
    for layer in range(layers):
        lg = logical_kv(tok_off[-1], heads, head_bytes, kind, dg, device)
        for key, bs, layout in (("producer", producer_bs, LAYOUT_NHD),
                                ("consumer", consumer_bs, LAYOUT_HND)):
            po, _, _, bids, nb = tables[key]
            pool = scatter_pool(lg, tok_off, bs, layout, bids, po.tolist(), nb)
            out[key].append(CacheSpec(pool, nb, layout, layer, 0, heads, head_bytes))
        po, _, _, bids, nb = tables["shard"]
        for s, hs in ((0, slice(0, half)), (1, slice(half, heads))):
            pool = scatter_pool(lg, tok_off, producer_bs, LAYOUT_NHD, bids,
                                po.tolist(), nb, heads=hs)
            out[f"shard{s}"].append(CacheSpec(pool, nb, LAYOUT_NHD, layer,
                                              s * half, half, head_bytes))
        del lg

    def wl(name, key, caches, bs):
        po, fp, nt, bids, _ = tables[key]
        return Workload(name, bs, caches, po.to(device), fp.to(device),
                        nt.to(device), bids.to(device),
                        info=dict(layers=layers, heads=heads, head_bytes=head_bytes,
                                  block_size=bs, kind=kind, requests=num_requests,
                                  seed=seed))

    return (wl("invariance_producer", "producer", out["producer"], producer_bs),
            wl("invariance_consumer", "consumer", out["consumer"], consumer_bs),
            wl("invariance_shard0", "shard", out["shard0"], producer_bs),
            wl("invariance_shard1", "shard", out["shard1"], producer_bs))


# ---------------------------------------------------------------------------
# Mamba running states
# ---------------------------------------------------------------------------

def mamba2(seed: int = 0, device="cpu", num_requests: int = 64, layers: int = 64,
           ssm_heads: int = 80, head_dim: int = 64, d_state: int = 128,
           conv_dim: int = 5376, conv_width: int = 4, spare_blocks: int = 3,
           first_positions=None, positions_per_request: int = 1) -> Workload:
    """Mamba2-shaped running states (d_inner 5120, 80 heads of 64, d_state
    128, conv width 4): per layer an SSM state with one row per head
    (head_dim x d_state fp32 values, 4-byte elements; 32 KiB) and a conv
    state with one row per conv channel (conv_width - 1 bf16 values, 2-byte
    elements), numbered consecutively within the layer (SSM rows, then conv
    rows).  One state block per request at block position 0, block ids a
    seeded permutation of the pool; values are random bits."""
    device = torch.device(device)
    g = _cpu_gen(seed)
    R = num_requests
    per = positions_per_request
    po = torch.arange(0, (R + 1) * per, per, dtype=torch.int64)
    fp = torch.tensor(list(first_positions) if first_positions is not None else [0] * R,
                      dtype=torch.int64)
    nt = torch.full((R,), 1000, dtype=torch.int64)
    nb = R * per + spare_blocks
    bids = torch.randperm(nb, generator=g)[:R * per].to(torch.int32)
    dg = _dev_gen(seed, device)
    ssm_row = head_dim * d_state * 4
    conv_row = (conv_width - 1) * 2
    caches = []
    for li in range(layers):
        ssm = fill_bytes(nb * ssm_heads * ssm_row, BITS16, dg, device)
        conv = fill_bytes(nb * conv_dim * conv_row, BITS16, dg, device)
        caches.append(CacheSpec(ssm, nb, LAYOUT_STATE, li, 0, ssm_heads, ssm_row,
                                piece_bytes=4))
        caches.append(CacheSpec(conv, nb, LAYOUT_STATE, li, ssm_heads, conv_dim, conv_row,
                                piece_bytes=2))
    return Workload("mamba2", 16, caches, po.to(device), fp.to(device), nt.to(device),
                    bids.to(device),
                    info=dict(layers=layers, heads=ssm_heads + conv_dim, head_bytes=ssm_row,
                              block_size=16, kind=BITS16, layout=LAYOUT_STATE,
                              requests=R, seed=seed))


@dataclass
class WriteBatch:
    """New tokens to write into paged caches (the KV-cache page's
    reshape_and_cache inputs), plus the written blocks as checksum
    positions: request r's blocks are positions po[r]..po[r+1] starting at
    block position fp[r], with nt[r] valid tokens."""

    block_size: int
    caches: list[CacheSpec]
    keys: list[torch.Tensor]
    values: list[torch.Tensor]
    slot_mapping: torch.Tensor     # int64 [num_tokens]
    positions: torch.Tensor        # int64 [num_tokens]
    num_blocks: int
    pos_offsets: torch.Tensor      # int64 [R+1]
    first_position: torch.Tensor   # int64 [R]
    num_tokens: torch.Tensor       # int64 [R]
    block_ids: torch.Tensor        # int32 [pos_offsets[R]]
    info: dict = field(default_factory=dict)

    def checksum_workload(self) -> Workload:
        return Workload("written", self.block_size, self.caches, self.pos_offsets,
                        self.first_position, self.num_tokens, self.block_ids, self.info)


def llama3_8b_write(seed: int = 0, device="cpu", kind: str = "prefill",
                    num_requests: int | None = None, layout: int = LAYOUT_NHD,
                    kernel_block_size: int = 0, layers: int = 32) -> WriteBatch:
    """Llama-3-8B-shaped new tokens (8 KV heads, head_size 128, bf16
    ``randn`` K and V, block_size 16) for ``layers`` zeroed pools.
    ``prefill``: ``num_requests`` (default 32) requests of 512 new tokens at
    positions 0..511, written to consecutive slots of seeded-permuted
    blocks.  ``decode``: ``num_requests`` (default 256) requests of one new
    token each at lengths uniform in [512, 4096), each in its own block."""
    device = torch.device(device)
    heads, hb, bs = 8, 256, 16
    g = _cpu_gen(seed)
    if kind == "decode":
        R = num_requests or 256
        lens = torch.randint(512, 4096, (R,), generator=g)
        nb = R + 64
        tables = torch.randperm(nb, generator=g)[:R].view(R, 1)
        slots = tables[:, 0] * bs + lens % bs
        pos = lens
        per = 1
        fp = lens // bs
        nt = lens + 1
    elif kind == "prefill":
        R, L = num_requests or 32, 512
        nb = R * L // bs + 64
        tables = torch.randperm(nb, generator=g)[:R * L // bs].view(R, L // bs)
        t = torch.arange(L)
        slots = (tables[:, t // bs] * bs + t % bs).reshape(-1)
        pos = t.repeat(R)
        per = L // bs
        fp = torch.zeros(R, dtype=torch.int64)
        nt = torch.full((R,), L, dtype=torch.int64)
    else:
        raise ValueError(kind)
    n = slots.numel()
    dg = _dev_gen(seed, device)
    caches = [CacheSpec(torch.zeros(2 * nb * bs * heads * hb, dtype=torch.uint8, device=device),
                        nb, layout, li, 0, heads, hb, kernel_block_size=kernel_block_size)
              for li in range(layers)]
    keys = [torch.randn((n, heads, hb // 2), dtype=torch.bfloat16, device=device, generator=dg)
            for _ in range(layers)]
    vals = [torch.randn((n, heads, hb // 2), dtype=torch.bfloat16, device=device, generator=dg)
            for _ in range(layers)]
    po = torch.arange(0, (R + 1) * per, per, dtype=torch.int64)
    return WriteBatch(bs, caches, keys, vals, slots.to(device), pos.to(device), nb,
                      po.to(device), fp.to(device), nt.to(device),
                      tables.reshape(-1).to(torch.int32).to(device),
                      info=dict(kind=kind, requests=R, layers=layers, heads=heads,
                                head_bytes=hb, block_size=bs, seed=seed))
