"""Failure handling on the GPU without faulting or hanging it: bounded
waits report through the status word and leave the context usable."""

import time

import numpy as np
import pytest
import torch

from helpers import W
import paged_kv_cache_kvcs_gb300 as K

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_times_out():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    K.selftest_wait_timeout(status, 50_000_000)          # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) & K.KVCS_STATUS_TIMEOUT
    assert 0.04 < dt < 5.0
    # the context is still usable: a checksum call right after is exact
    from gpu_helpers import full_oracle, gpu_checksums
    wl = W.random_case(2, "cuda", layers=2, heads=2, head_bytes=32, block_size=4,
                       lengths=(9,))
    got, st = gpu_checksums(wl)
    exp, _ = full_oracle(wl)
    assert st == 0 and np.array_equal(got, exp)


def test_selftest_rejects_bad_limits():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, -1, 3_000_000_000):
        with pytest.raises(K.KvcsError):
            K.selftest_wait_timeout(status, bad)
