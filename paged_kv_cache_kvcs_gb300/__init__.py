"""GB300 (sm_103a) KV-cache block checksums.

The checksum of page "vllm.distributed.kv_transfer.kv_checksum.checksum"
(vLLM API docs): per block position, over every (layer, KV head) slice,
``s = sum_j x_j (2j+1)`` and ``c = sum m s`` mod 2**64.  The work runs in the
CUDA library ``_build/libkvcs.so`` (C ABI in ``include/kvcs.h``); this
package only marshals arguments to it (``_binding``) and builds seeded
synthetic workloads (``workloads``).
"""

from ._binding import (  # noqa: F401
    KVCS_BLOCK_CHECKSUM_BYTES, KVCS_ECUDA, KVCS_EINVAL, KVCS_EUNSUPPORTED,
    KVCS_LAYOUT_HND, KVCS_LAYOUT_LATENT, KVCS_LAYOUT_NHD, KVCS_LAYOUT_XSPLIT,
    KVCS_LAYOUT_STATE, KVCS_OUT_ACCUMULATE, KVCS_OUT_WORKSPACE, KVCS_WORKSPACE_WORDS,
    KVCS_MAX_KV_HEADS_PER_LAYER, KVCS_OK, KVCS_STATUS_BAD_BLOCK_ID,
    KVCS_STATUS_BAD_REQUESTS, KVCS_STATUS_TIMEOUT, KvcsError, block_checksums,
    cache_array, kvcs_block_checksums, kvcs_cache, kvcs_plan, kvcs_plan_info,
    kvcs_plan_requests,
    kvcs_requests, launch_count, load_library, plan_for, selftest_wait_timeout,
    strerror, version,
    workload_checksums, Checksummer, workload_checksummer, kvcs_outputs,
    group_checksums, block_checksum_tags, write_kv, KVWriter,
    KVCS_ETOOLARGE, KVCS_NOALLOC_MAX_CACHES, block_checksums_noalloc,
    kvcs_block_checksums_noalloc)
