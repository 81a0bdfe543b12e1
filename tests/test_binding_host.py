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


class FakeTensor:
    """Enough of a CUDA tensor for the binding's argument checks (no GPU
    here): its address is never dereferenced because every case below is
    refused before the library is called."""

    def __init__(self, n, dtype, dev=0):
        self.n, self.dtype = n, dtype
        self.device = torch.device("cuda", dev)
        self.is_cuda = True

    def numel(self):
        return self.n

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 1 << 20

    def element_size(self):
        return torch.empty(0, dtype=self.dtype).element_size()


def _fake_tables(R=3, P=10, ids=None, fp=None, nt=None):
    return (FakeTensor(R + 1, torch.int64), FakeTensor(R if fp is None else fp, torch.int64),
            FakeTensor(R if nt is None else nt, torch.int64),
            FakeTensor(P if ids is None else ids, torch.int32))


class _Cache:
    pool = 1 << 21
    num_blocks, layout, layer, head_offset, num_heads, head_bytes = 16, 0, 0, 0, 2, 64


@pytest.fixture
def on_cuda0(monkeypatch):
    monkeypatch.setattr(B, "_current_device", lambda: torch.device("cuda", 0))


def test_group_checksums_refuses_cpu_tensors():
    wl = W.tiny(0, "cpu")
    with pytest.raises(ValueError, match="CUDA"):
        K.group_checksums(wl.caches, wl.block_size, wl.pos_offsets, wl.first_position,
                          wl.num_tokens, wl.block_ids, 1)


@pytest.mark.parametrize("bad", ["block_ids_short", "first_position_count", "num_tokens_count",
                                 "wrong_dtype", "other_device"])
def test_request_tables_checked(on_cuda0, bad):
    po, fp, nt, ids = _fake_tables()
    if bad == "block_ids_short":
        ids = FakeTensor(9, torch.int32)
    elif bad == "first_position_count":
        fp = FakeTensor(2, torch.int64)
    elif bad == "num_tokens_count":
        nt = FakeTensor(4, torch.int64)
    elif bad == "wrong_dtype":
        ids = FakeTensor(10, torch.int64)
    else:
        nt = FakeTensor(3, torch.int64, dev=1)
    with pytest.raises(ValueError):
        K.block_checksums([_Cache()], 16, po, fp, nt, ids, total_positions=10)
    with pytest.raises(ValueError):
        K.Checksummer([_Cache()], 16, po, fp, nt, ids, 10)
    with pytest.raises(ValueError):
        K.group_checksums([_Cache()], 16, po, fp, nt, ids, 1, total_positions=10)


def test_block_checksums_output_checked(on_cuda0):
    po, fp, nt, ids = _fake_tables()
    for out in (FakeTensor(9, torch.int64), FakeTensor(10, torch.int32),
                FakeTensor(10, torch.int64, dev=1)):
        with pytest.raises(ValueError):
            K.block_checksums([_Cache()], 16, po, fp, nt, ids, out=out, total_positions=10)
    with pytest.raises(ValueError):
        K.block_checksums([_Cache()], 16, po, fp, nt, ids, out=FakeTensor(10, torch.int64),
                          status=FakeTensor(1, torch.int64), total_positions=10)


def test_prepared_call_checks_its_output(on_cuda0):
    po, fp, nt, ids = _fake_tables()
    ck = K.Checksummer([_Cache()], 16, po, fp, nt, ids, 10)
    for out in (FakeTensor(9, torch.int64), FakeTensor(10, torch.float64),
                FakeTensor(10, torch.int64, dev=1)):
        with pytest.raises(ValueError):
            ck(out)


@pytest.mark.parametrize("bad", ["values_short", "row_sums_short", "tags_short",
                                 "expected_short", "mismatch_short", "mismatch_count_dtype",
                                 "columns_zero", "columns_65"])
def test_group_outputs_checked(on_cuda0, bad):
    po, fp, nt, ids = _fake_tables()
    n, cols = 10, 2
    kw = dict(values=FakeTensor(n * cols, torch.int64), row_sums=FakeTensor(n, torch.int64),
              tags=FakeTensor(n, torch.int64), expected=FakeTensor(n, torch.int64),
              mismatch=FakeTensor(n, torch.uint8), mismatch_count=FakeTensor(1, torch.int32))
    short = {"values_short": ("values", FakeTensor(n * cols - 1, torch.int64)),
             "row_sums_short": ("row_sums", FakeTensor(n - 1, torch.int64)),
             "tags_short": ("tags", FakeTensor(n - 1, torch.int64)),
             "expected_short": ("expected", FakeTensor(n - 1, torch.int64)),
             "mismatch_short": ("mismatch", FakeTensor(n - 1, torch.uint8)),
             "mismatch_count_dtype": ("mismatch_count", FakeTensor(1, torch.int64))}
    if bad in short:
        k, v = short[bad]
        kw[k] = v
    else:
        cols = 0 if bad == "columns_zero" else 65
    with pytest.raises(ValueError):
        K.group_checksums([_Cache()], 16, po, fp, nt, ids, cols, total_positions=n, **kw)


def test_workspace_checked(on_cuda0):
    po, fp, nt, ids = _fake_tables()
    for ws in (FakeTensor(K.KVCS_WORKSPACE_WORDS - 1, torch.int64),
               FakeTensor(K.KVCS_WORKSPACE_WORDS, torch.int32),
               FakeTensor(K.KVCS_WORKSPACE_WORDS, torch.int64, dev=1)):
        with pytest.raises(ValueError):
            K.group_checksums([_Cache()], 16, po, fp, nt, ids, 1, total_positions=10,
                              values=FakeTensor(10, torch.int64), workspace=ws)
        with pytest.raises(ValueError):
            K.Checksummer([_Cache()], 16, po, fp, nt, ids, 10, workspace=ws)


def test_output_flags_validated():
    """Unknown flag bits, and a workspace flag without a workspace, are
    refused before any CUDA call (no GPU here)."""
    lib = K.load_library()
    arr = K.cache_array([_Cache()])
    reqs = B.kvcs_requests(1, 16, 32, 48, 64)
    for flags, ws in ((4, None), (K.KVCS_OUT_WORKSPACE, None), (K.KVCS_OUT_WORKSPACE, 4100)):
        outs = B.kvcs_outputs(1, flags, 4096, None, None, None, None, None, ws)
        rc = lib.kvcs_group_checksums(arr, 1, 16, ctypes.byref(reqs), 4, ctypes.byref(outs),
                                      None, None)
        assert rc == K.KVCS_EINVAL, (flags, ws)
