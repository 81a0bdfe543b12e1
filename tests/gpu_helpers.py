"""GPU-side test plumbing: run the library on a workload, and build the
oracle's inputs for a sample of positions of a large workload (gathering
only the pages those positions read).  Data movement only."""

from __future__ import annotations

import numpy as np
import torch

from helpers import W, OracleCache, OracleRequests, c_oracle, host_bytes
import paged_kv_cache_kvcs_gb300 as K


def gpu_checksums(wl, stream=None):
    status = torch.zeros(1, dtype=torch.int32, device=wl.pos_offsets.device)
    out = K.workload_checksums(wl, status=status, stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint64), int(status.item())


def sampled_oracle_inputs(wl, positions):
    """Oracle caches/requests covering only ``positions`` (global indices):
    each sampled position becomes a one-block request of its own, reading a
    compact host pool of just the pages it needs."""
    pos = torch.as_tensor(sorted(set(int(p) for p in positions)), dtype=torch.int64)
    po = wl.pos_offsets.cpu()
    req = torch.searchsorted(po, pos, right=True) - 1
    q = wl.first_position.cpu()[req] + (pos - po[req])
    nt = wl.num_tokens.cpu()[req]
    ids = wl.block_ids.cpu()[pos].to(torch.int64)
    k = len(pos)
    caches = []
    for c in wl.caches:
        pages = W.gather_pages(c, wl.block_size, ids)
        caches.append(OracleCache(host_bytes(pages), k, c.layout, c.layer,
                                  c.head_offset, c.num_heads, c.head_bytes,
                                  getattr(c, "piece_bytes", 0) or 8,
                                  getattr(c, "kernel_block_size", 0)))
    reqs = OracleRequests(list(range(k + 1)), q.tolist(), nt.tolist(), list(range(k)))
    return pos.numpy(), caches, reqs


def oracle_sampled(wl, positions, threads=16):
    """The C oracle over ``positions`` of ``wl``: (positions, values, status)."""
    pos, caches, reqs = sampled_oracle_inputs(wl, positions)
    vals, status = c_oracle.block_checksums(caches, wl.block_size, reqs,
                                            num_threads=threads)
    return pos, vals, status


def oracle_every_position(wl, chunk_bytes=4 << 30, threads=None):
    """The oracle's checksum of every position of ``wl`` (uint64 array) and
    its status word.  Consecutive positions are taken in chunks whose pages
    fit in ``chunk_bytes`` of host memory; each chunk's pages are gathered
    (data movement only) and handed to the C form."""
    threads = threads or c_oracle.default_threads()
    per_pos = 0
    for c in wl.caches:
        state = c.layout == W.LAYOUT_STATE
        halves = 1 if c.layout in (W.LAYOUT_LATENT, W.LAYOUT_STATE) else 2
        per_pos += halves * (1 if state else wl.block_size) * c.num_heads * c.head_bytes
    total = wl.num_positions
    step = max(1, chunk_bytes // max(1, per_pos))
    out = np.zeros(total, dtype=np.uint64)
    status = 0
    for lo in range(0, total, step):
        pos, vals, st = oracle_sampled(wl, range(lo, min(total, lo + step)), threads)
        out[pos] = vals
        status |= st
    return out, status


def full_oracle(wl, threads=16):
    from helpers import oracle_inputs
    caches, reqs = oracle_inputs(wl)
    return c_oracle.block_checksums(caches, wl.block_size, reqs, num_threads=threads)
