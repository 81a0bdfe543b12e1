"""The Python binding without a GPU: it fails loudly, never falls back.
A missing library raises; CPU tensors are refused before the library is
called; arguments the C side would reject are refused with the library's
error codes; write_kv checks its buffers."""

import ctypes
from pathlib import Path

import pytest
import torch

import paged_kv_cache_kvcs_gb300 as K
from paged_kv_cache_kvcs_gb300 import _binding as B
from paged_kv_cache_kvcs_gb300 import workloads as W


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", Path("/nonexistent/libkvcs.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.load_library()


def test_cpu_tensors_are_refused():
    wl = W.tiny(0, "cpu")
    with pytest.raises(ValueError, match="CUDA"):
        K.workload_checksums(wl)
    with pytest.raises(ValueError, match="CUDA"):
        K.Checksummer(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                      wl.num_tokens, wl.block_ids, 7)
    c = wl.caches[0]
    key = torch.zeros((3, c.num_heads, c.head_bytes), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        K.write_kv(c, wl.block_size, key, key.clone(), torch.zeros(3, dtype=torch.int64),
                   torch.zeros(3, dtype=torch.int64))


def test_accumulate_needs_values():
    wl = W.tiny(0, "cpu")
    with pytest.raises(ValueError):
        K.group_checksums([], 16, wl.pos_offsets, wl.first_position, wl.num_tokens,
                          wl.block_ids, 1, accumulate=True, total_positions=0)


def test_write_kv_rejects_before_any_cuda_call():
    """The C entry point validates its host arguments first: these calls
    return error codes with nothing launched (no GPU here)."""
    lib = K.load_library()

    class FakeCache:
        def __init__(self, layout=0, num_blocks=10, num_heads=2, head_bytes=64,
                     layer=0):
            self.pool = 1 << 20
            self.num_blocks = num_blocks
            self.layout = layout
            self.layer = layer
            self.head_offset = 0
            self.num_heads = num_heads
            self.head_bytes = head_bytes

    def call(caches, keys, values, bs=16, n=4):
        arr = K.cache_array(caches)
        kp = (ctypes.c_void_p * len(caches))(*keys)
        vp = (ctypes.c_void_p * len(caches))(*values)
        return lib.kvcs_write_kv(arr, len(caches), bs, n, kp, vp, 4096, 8192, None, None,
                                 None)

    ok_k, ok_v = 1 << 21, 1 << 22
    # a state cache is not per token
    assert call([FakeCache(layout=4)], [ok_k], [ok_v]) == K.KVCS_EINVAL
    # a latent cache takes no value pointer; a KV cache needs one
    assert call([FakeCache(layout=2, num_heads=1)], [ok_k], [ok_v]) == K.KVCS_EINVAL
    assert call([FakeCache()], [ok_k], [None]) == K.KVCS_EINVAL
    # key pointers must be 8-byte aligned
    assert call([FakeCache()], [ok_k + 4], [ok_v]) == K.KVCS_EINVAL
    # rows of 1 GiB or more
    assert call([FakeCache(num_heads=1 << 15, head_bytes=1 << 15)], [ok_k], [ok_v]) == \
        K.KVCS_EUNSUPPORTED
    # two caches weighing the same (layer, head)
    assert call([FakeCache(), FakeCache()], [ok_k, ok_k], [ok_v, ok_v]) == K.KVCS_EINVAL
    # zero tokens: nothing to do
    assert call([FakeCache()], [ok_k], [ok_v], n=0) == K.KVCS_OK
