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
    dev_ids = ids.to(wl.pos_offsets.device)
    for c in wl.caches:
        state = c.layout == W.LAYOUT_STATE
        halves = 1 if c.layout in (W.LAYOUT_LATENT, W.LAYOUT_STATE) else 2
        page = (1 if state else wl.block_size) * c.num_heads * c.head_bytes
        pages = c.pool.view(halves, c.num_blocks, page)[:, dev_ids]
        caches.append(OracleCache(host_bytes(pages), k, c.layout, c.layer,
                                  c.head_offset, c.num_heads, c.head_bytes,
                                  getattr(c, "piece_bytes", 0) or 8))
    reqs = OracleRequests(list(range(k + 1)), q.tolist(), nt.tolist(), list(range(k)))
    return pos.numpy(), caches, reqs


def oracle_sampled(wl, positions, threads=16):
    pos, caches, reqs = sampled_oracle_inputs(wl, positions)
    vals, status = c_oracle.block_checksums(caches, wl.block_size, reqs,
                                            num_threads=threads)
    return pos, vals, status


def full_oracle(wl, threads=16):
    from helpers import oracle_inputs
    caches, reqs = oracle_inputs(wl)
    return c_oracle.block_checksums(caches, wl.block_size, reqs, num_threads=threads)
