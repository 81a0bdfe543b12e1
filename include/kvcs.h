/*
 * kvcs.h -- C ABI of the GB300 (sm_103a) KV-cache block checksum library.
 *
 * What it computes (page "vllm.distributed.kv_transfer.kv_checksum.checksum",
 * vLLM API docs, module docstring items 1 and 2):
 *
 *   Each (layer, KV head) pair owns one slice of a block.  Its bytes run
 *   through the block's tokens in order, each token contributing the head's
 *   K bytes and then its V bytes; the slice is read as consecutive
 *   little-endian 64-bit words x_j, where j = t*P + p for word p of the token
 *   at request position t and P words per token.  Its checksum is
 *       s = sum_j x_j * (2j + 1)                      mod 2^64
 *   and the block's checksum is
 *       c = sum_{layer, head} m * s                   mod 2^64,
 *       m = 2 * (layer * 65536 + global_head) + 1.
 *   Slots at or past the request's num_tokens are skipped (dataclass
 *   KVChecksumBlocks; function num_valid_tokens): the block at position q
 *   holds request tokens q*block_size .. q*block_size + block_size - 1, and
 *   only those below num_tokens count.
 *
 * Because every slice is weighted by its global layer and head, partial
 * results from several calls (tensor-parallel head shards, pipeline stages,
 * several caches of one layer) combine by wrapping uint64 addition
 * (module docstring, paragraph on TP ranks and PP stages).
 *
 * Memory: the caller owns every buffer.  The library allocates nothing and
 * enqueues all work on the caller's stream; calls are asynchronous.  (Its
 * one piece of device memory of its own is the 128-byte scratch array of
 * kvcs_block_checksums_noalloc, part of the loaded module.)
 * Stream order: a call's kernels touch memory only after the stream's
 * earlier work has finished (kvcs_write_kv's kernel may be scheduled while
 * the previous kernel ends, and waits for it before any access).  The
 * checksum and write kernels let a following kernel that was launched with
 * programmatic stream serialization start before they end;
 * as with any programmatic dependent launch, such a kernel must wait for
 * them (griddepcontrol.wait, cudaGridDependencySynchronize) before it reads
 * what they write.
 * Thread safety: calls may be issued concurrently from several host threads
 * and streams; they share no mutable state apart from a launch counter
 * (and, for kvcs_block_checksums_noalloc, its scratch array: see there).
 */
#ifndef KVCS_H_
#define KVCS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* H in the slice factor: the page's MAX_KV_HEADS_PER_LAYER = 1 << 16.
 * A cache whose global heads reach past it is rejected: the page leaves
 * layers with more KV heads than H out of checksumming. */
#define KVCS_MAX_KV_HEADS_PER_LAYER 65536

/* Bytes per block checksum (the page's BLOCK_CHECKSUM_BYTES: one 64-bit
 * word; values are unsigned). */
#define KVCS_BLOCK_CHECKSUM_BYTES 8

/* Cache layouts (page "【vLLM 源码解析】KV Cache", section "reshape kv_cache":
 * a raw byte pool reshaped to [2, num_blocks, block_size, heads, head_size]).
 *   NHD:    pool [2 (K, V)][num_blocks][block_size][num_heads][head_bytes]
 *   HND:    pool [2 (K, V)][num_blocks][num_heads][block_size][head_bytes]
 *   LATENT: pool [num_blocks][block_size][row_bytes]  (MLA: one latent row
 *           per token, no K/V split; counted as one head whose token slice
 *           is the whole row, P = row_bytes / 8)
 *   XSPLIT: pool [2][num_blocks][num_heads][head_bytes/16][block_size][16]:
 *           the x-split layout of the KV-cache page's reshape_and_cache
 *           section ([num_blocks, heads, head_size/x, block_size, x] with x
 *           elements = 16 bytes), used here for both K and V pages;
 *           head_bytes must be a multiple of 16
 *   STATE:  pool [num_blocks][num_heads rows][head_bytes]: a Mamba layer's
 *           running state, one block per request at block position 0 (the
 *           checksum page, paragraph on Mamba state).  Each row is one
 *           global row along the TP-split dimension (head_offset = global
 *           index of local row 0) and is a slice whose pieces are its
 *           piece_bytes-wide elements (2 or 4) read unsigned, weighted by
 *           element index.  A state whose split is unknown is passed as one
 *           row per TP shard (head_offset = the shard index).  Other block
 *           positions hold no state (0); num_tokens does not apply.  A call
 *           holds either only STATE caches or none. */
typedef enum kvcs_layout {
  KVCS_LAYOUT_NHD = 0,
  KVCS_LAYOUT_HND = 1,
  KVCS_LAYOUT_LATENT = 2,
  KVCS_LAYOUT_XSPLIT = 3,
  KVCS_LAYOUT_STATE = 4
} kvcs_layout;

/* One layer's paged pool (one attention layer, or one of several caches of
 * a layer such as an indexer's, numbered by consecutive head offsets).
 * Read-only to the library.  A page is one block's K, its V, or its latent
 * rows: page_bytes = block_size * num_heads * head_bytes contiguous bytes in
 * the layout's order (STATE: num_heads * head_bytes); the page of
 * (half, block) starts at base + half * half_stride + block * block_stride. */
typedef struct kvcs_cache {
  const void *base;    /* DEVICE pointer to the pool; 8-byte aligned.  Pools
                          and strides that are 16-byte multiples are read
                          with plain bulk copies, those only 8-byte aligned
                          (NHD, latent, HND without sub-blocks, x-split)
                          with bulk copies of the aligned interiors and
                          8-byte copies of the edge words; the rest, and
                          heads of 8 mod 16 bytes, with direct loads.
                          Results are the same either way. */
  int64_t num_blocks;  /* pages in the pool; valid block ids are [0, num_blocks) */
  int32_t layout;      /* a kvcs_layout */
  int32_t layer;       /* layer number taken from the layer's name, >= 0 */
  int32_t head_offset; /* global index of this cache's local head 0 (TP shard
                          offset, or the head count of earlier caches of the
                          same layer); LATENT: the one head's global index */
  int32_t num_heads;   /* local KV heads; 1 for LATENT */
  int32_t head_bytes;  /* NHD/HND/XSPLIT: bytes of one head's K (= its V)
                          for one token; LATENT: bytes of one token row; a
                          positive multiple of 8.  STATE: bytes of one state
                          row, a positive multiple of piece_bytes. */
  int32_t column;      /* replica-key column this cache's layer adds into
                          (kvcs_group_checksums); 0 for kvcs_block_checksums */
  int64_t half_stride; /* NHD/HND: bytes from a block's K page to its V page
                          (may be negative, e.g. separate K and V tensors);
                          0 = num_blocks * page_bytes, the [2][num_blocks]...
                          pool above.  Ignored for LATENT. */
  int64_t block_stride;/* bytes between consecutive blocks' pages;
                          0 = page_bytes.  [num_blocks][2][...] pools
                          (K and V interleaved per block) use half_stride =
                          page_bytes and block_stride = 2 * page_bytes. */
  int32_t kernel_block_size; /* HND only: tokens per kernel sub-block when the
                          attention kernel splits each block into
                          block_size / kernel_block_size sub-blocks (the KV-cache
                          page, section "reshape kv_cache"); a block is then
                          [sub-block][heads][kernel_block_size][head_bytes].
                          0 = block_size.  Must divide block_size.  For NHD and
                          LATENT, consecutive sub-blocks are already the
                          block's rows in order, so the field is ignored. */
  int32_t piece_bytes; /* STATE: element bytes, 2 or 4; other layouts: 0 */
} kvcs_cache;

/* The requests to checksum, in CSR form over requests.  All pointers are
 * DEVICE pointers, read-only to the library.  This is the page's dataclass
 * KVChecksumBlocks (num_tokens; per group the first block position and the
 * block ids at consecutive positions) for one KV-cache group, flattened. */
typedef struct kvcs_requests {
  int64_t num_requests;          /* R >= 0 */
  const int64_t *pos_offsets;    /* [R + 1]: request r owns global position
                                    indices [pos_offsets[r], pos_offsets[r+1]);
                                    pos_offsets[0] = 0, non-decreasing,
                                    pos_offsets[R] = total_positions */
  const int64_t *first_position; /* [R]: block position (>= 0) of the request's
                                    first listed block */
  const int64_t *num_tokens;     /* [R]: tokens whose KV the blocks hold */
  const int32_t *block_ids;      /* [total_positions]: index i holds block
                                    position first_position[r] + i - pos_offsets[r]
                                    of request r */
} kvcs_requests;

/* Return codes (negative: nothing was enqueued unless stated). */
#define KVCS_OK 0
#define KVCS_EINVAL (-1)      /* null pointer, non-positive block_size,
                                 strides not multiples of 8 or smaller than a
                                 page, kernel_block_size not dividing
                                 block_size, bad piece_bytes, STATE caches
                                 mixed with KV caches,
                                 head_bytes not a positive multiple of 8,
                                 unknown layout, latent cache with heads != 1,
                                 negative layer or head offset, a column
                                 outside [0, num_columns) or a column with no
                                 cache, misaligned base, two caches covering
                                 the same (layer, global head) */
#define KVCS_EUNSUPPORTED (-2) /* a geometry the library does not handle:
                                 head_offset + num_heads > 65536 (any call),
                                 or a token row (num_heads * head_bytes) of
                                 1 GiB or more (kvcs_write_kv) */
#define KVCS_ECUDA (-3)       /* a CUDA call failed (launch, attribute query);
                                 work may have been partly enqueued */
#define KVCS_ETOOLARGE (-4)   /* the call is beyond a fixed limit of
                                 kvcs_block_checksums_noalloc (more than
                                 KVCS_NOALLOC_MAX_CACHES caches); nothing is
                                 enqueued */

/* Bits set in the caller's device status word by the kernels (OR-ed in; the
 * caller zeroes the word when it wants a fresh reading).  None of them traps
 * or aborts the context. */
#define KVCS_STATUS_BAD_BLOCK_ID 1u /* some block id was outside [0, num_blocks)
                                       of some cache: that position's output
                                       is 0 */
#define KVCS_STATUS_BAD_REQUESTS 2u /* pos_offsets not starting at 0, decreasing,
                                       or not ending at total_positions, or a
                                       negative first_position: the affected
                                       positions' outputs are 0 */
#define KVCS_STATUS_TIMEOUT 4u      /* an internal pipeline wait ran past its
                                       time limit (about 2 s) and gave up: the
                                       outputs of that call are not valid */

/*
 * kvcs_block_checksums -- one uint64 block checksum per global position index.
 *
 *   caches           HOST array of num_caches descriptors (copied into the
 *                    launch; may be freed when the call returns).
 *   num_caches       >= 1.  Any number; above an internal per-launch limit
 *                    the work is split over several launches.
 *   block_size       tokens per block (> 0), the same for every cache.
 *   reqs             HOST pointer to the request table (whose arrays are on
 *                    the device).
 *   total_positions  pos_offsets[R] as known to the host (>= 0).
 *   out              DEVICE uint64[total_positions], written entirely:
 *                    out[i] = c of global position index i, or 0 where the
 *                    position holds no valid token or is flagged bad.
 *   status           DEVICE uint32 word or NULL; see KVCS_STATUS_*.
 *   stream           a cudaStream_t (NULL = the legacy default stream).
 *
 * Returns KVCS_OK once the work is enqueued.  Validation of the host
 * arguments happens before any CUDA call, so a negative return other than
 * KVCS_ECUDA means nothing was enqueued.  Data-dependent problems in the
 * device arrays are reported through *status, never by a fault.
 */
int kvcs_block_checksums(const kvcs_cache *caches, int32_t num_caches,
                         int32_t block_size, const kvcs_requests *reqs,
                         int64_t total_positions, uint64_t *out,
                         uint32_t *status, void *stream);

/*
 * Per-position outputs of kvcs_group_checksums.  All pointers are DEVICE
 * pointers owned by the caller.
 *
 * When KV is replicated across ranks (an MLA latent cache, or GQA heads
 * copied to several TP ranks), each replica is checked separately: the
 * partial over a set of layers carries the (replicas, replica_index) key of
 * those layers, and one partial is kept per key (the checksum page,
 * paragraph on replicated KV; dataclass KVChecksumGroup, field values).  Here
 * each cache names the column of its key; values[i * num_columns + k] is
 * position i's partial over the caches of column k.
 *
 * A load of offloaded KV is checked against the checksums offloaded with it:
 * each row's partials summed (KVChecksumGroup, field stored), XORed with the
 * block's tag (function block_checksum_tags) so that it matches only the
 * block it was stored for.
 *
 * KVCS_OUT_ACCUMULATE in flags adds this call's partials into values
 * (mod 2^64) instead of overwriting them.  Block checksums are sums over
 * layers (the checksum page, item 2), so a caller that receives KV layer by
 * layer (the connector page: start_load_kv with per-layer events,
 * wait_for_layer_load) can checksum each layer group as it lands, on the
 * stream that waits for that group, and end with the full checksum.  A
 * position with no valid token, or with a bad block id, then adds nothing.
 * Row sums, tags and the comparison, when asked for, are computed from
 * values as they stand after the add.
 */
#define KVCS_OUT_ACCUMULATE 1

/*
 * KVCS_OUT_WORKSPACE in flags: `workspace` (below) points to at least
 * KVCS_WORKSPACE_WORDS uint64 words of DEVICE memory the call may use as
 * scratch while it runs.  With it the bulk-copy kernel balances its work
 * dynamically: each CTA reads a fixed share of the positions and then takes
 * the rest in small chunks from a counter in the workspace, so CTAs on
 * slower or busier SMs take less (without it every CTA's share is fixed and
 * the call ends with its slowest SM).  Only calls of at least 1024 work
 * units (KV pages, kvcs_plan's `units`) per SM use it; smaller calls keep
 * the fixed shares, which suit them better, and leave the workspace alone.
 * The valid-slot kernel (calls of at most two positions per request: their
 * latent and HND caches, and NHD caches of pages of at most 8 KiB) uses it
 * the same way from 64 pages per warp on:
 * each warp reads a fixed quarter share of the pages, then ranges of the
 * rest that shrink as they run out (the positions' valid slots, and so
 * their bytes, differ).  One counter is used per bulk-copy or valid-slot
 * launch, for the first KVCS_WORKSPACE_WORDS launches.  The call zeroes the
 * words it uses itself;
 * their contents afterwards are unspecified.  Calls that may run at the
 * same time on the GPU (other streams) must use different workspaces.
 */
#define KVCS_OUT_WORKSPACE 2
#define KVCS_WORKSPACE_WORDS 16

typedef struct kvcs_outputs {
  int32_t num_columns;       /* >= 1 and <= 64 */
  int32_t flags;             /* KVCS_OUT_ACCUMULATE and/or KVCS_OUT_WORKSPACE;
                                other bits invalid */
  uint64_t *values;          /* required: [total_positions][num_columns] */
  uint64_t *row_sums;        /* or NULL: [total_positions], sum of the row's
                                values XOR tags[i] (when tags is given) */
  const uint64_t *tags;      /* or NULL: [total_positions] */
  const uint64_t *expected;  /* or NULL: [total_positions], the stored values
                                to verify against */
  uint8_t *mismatch;         /* or NULL (needs expected): [total_positions],
                                1 where the tagged row sum != expected, else 0 */
  uint32_t *mismatch_count;  /* or NULL (needs expected): mismatching
                                positions are added to this word */
  uint64_t *workspace;       /* read only with KVCS_OUT_WORKSPACE in flags:
                                DEVICE, KVCS_WORKSPACE_WORDS words, 8-byte
                                aligned, used by this call alone */
} kvcs_outputs;

/*
 * kvcs_group_checksums -- partial checksums per replica-key column, and
 * optionally the tagged row sums and their comparison with stored values.
 *
 * Arguments as kvcs_block_checksums, with the outputs in *outs (a HOST
 * pointer).  Every column in [0, num_columns) must be named by at least one
 * cache.  With one column, values equals kvcs_block_checksums' output.
 * Row sums, tags and the comparison cost one small extra kernel launch that
 * reads values (8 * num_columns bytes per position).
 */
int kvcs_group_checksums(const kvcs_cache *caches, int32_t num_caches,
                         int32_t block_size, const kvcs_requests *reqs,
                         int64_t total_positions, const kvcs_outputs *outs,
                         uint32_t *status, void *stream);

/*
 * kvcs_block_checksums_noalloc -- kvcs_block_checksums for callers that
 * cannot allocate device memory, with the dynamic share-out of a workspace
 * call (KVCS_OUT_WORKSPACE) but no workspace to pass.
 *
 * The paged-KV checksum has no counterpart of this entry point: it exists
 * for the library's users.  Some callers cannot call cudaMalloc or any
 * allocator: code that runs where the process's allocator must not be
 * entered (inside a caching allocator's own hooks, a memory-pool callback,
 * or a real-time serving loop that forbids allocation after start-up), and
 * code that owns no device buffer of its own to lend (a plug-in given only
 * the KV pools and an output array).  This entry point asks for nothing
 * beyond the inputs and the output: its scratch, the bulk kernel's work
 * counters, is a module-scope device array of KVCS_WORKSPACE_WORDS words
 * (128 bytes) that every GPU which loads the library holds until the
 * process exits.  The call itself allocates nothing: no cudaMalloc or
 * cudaFree and no allocating library routine.
 *
 * Arguments, results, status bits and errors as kvcs_block_checksums, plus:
 *   - num_caches above KVCS_NOALLOC_MAX_CACHES returns KVCS_ETOOLARGE before
 *     any CUDA call (within it, every bulk-copy launch of the call has a
 *     counter of the array to itself);
 *   - the first call on a device looks up the array's device address there
 *     (cudaGetSymbolAddress, with that device current) and keeps it, so
 *     make that first call before any stream capture on the device;
 *   - every call on a device shares the one array, which keeps the last
 *     call's counters: each call zeroes the counters it uses (a small kernel
 *     ahead of its checksum launches, in stream order).  Calls that can
 *     overlap on the GPU (other streams, other threads) race on the
 *     counters and may then return wrong checksums: issue them in one
 *     stream order, or use kvcs_group_checksums with a workspace per stream.
 */
#define KVCS_NOALLOC_MAX_CACHES 1024
int kvcs_block_checksums_noalloc(const kvcs_cache *caches, int32_t num_caches,
                                 int32_t block_size, const kvcs_requests *reqs,
                                 int64_t total_positions, uint64_t *out,
                                 uint32_t *status, void *stream);

/*
 * kvcs_block_checksum_tags -- the 64-bit tag of each block (the checksum
 * page, function block_checksum_tags): the first eight bytes of the block's
 * hash read as a little-endian integer, XOR the group's fingerprint.
 *
 *   block_hashes  DEVICE bytes; hash i starts at block_hashes + i*hash_stride
 *   hash_stride   bytes between consecutive hashes, >= 8
 *   n             number of blocks (>= 0)
 *   fingerprint   the group's fingerprint (sum over PP stages of its layers'
 *                 hashes; computed by the caller)
 *   tags          DEVICE uint64[n]
 */
int kvcs_block_checksum_tags(const void *block_hashes, int64_t hash_stride,
                             int64_t n, uint64_t fingerprint, uint64_t *tags,
                             void *stream);

/*
 * kvcs_write_kv -- write new tokens' K and V into layers' paged caches and
 * add each written token's share of its block's checksum to a running word
 * per physical block.
 *
 * The write is the KV-cache page's reshape_and_cache step (section
 * "逻辑到物理地址映射"): token i goes to slot slot_mapping[i] =
 * block * block_size + offset of every cache; a negative slot is a padding
 * token and is skipped.  Because the piece index j = t*P + p runs token by
 * token (the checksum page, item 1), a block's checksum is a sum over its
 * tokens, each token adding sum_h m_h sum_p x_p (2(t*P + p) + 1) with t its
 * position in the request.  So a running word per physical block, zeroed by
 * the caller when the block is allocated and added into for every layer of
 * the group, holds the checksum of the tokens written to the block so far --
 * with no second read of the cache.  One call can write all layers (the
 * receive side of a KV transfer) or one layer (a forward pass).
 *
 *   caches        HOST array of num_caches descriptors (NHD, HND, XSPLIT or
 *                 LATENT) sharing the block table
 *   keys, values  HOST arrays of num_caches DEVICE pointers:
 *                 [num_tokens][num_heads][head_bytes] each (token stride
 *                 num_heads * head_bytes bytes); for a LATENT cache keys[k]
 *                 is [num_tokens][row_bytes] and values[k] must be NULL
 *   slot_mapping  DEVICE int64[num_tokens]
 *   positions     DEVICE int64[num_tokens]: each token's position in its
 *                 request
 *   block_sums    DEVICE uint64[min over caches of num_blocks] or NULL
 *                 (write only)
 *   status        DEVICE word or NULL: KVCS_STATUS_BAD_BLOCK_ID for a slot
 *                 past a pool (token skipped), KVCS_STATUS_BAD_REQUESTS for
 *                 a negative position (token written, not checksummed)
 *   stream        a cudaStream_t
 *
 * Re-writing a slot adds its token again: roll back the running word (or
 * re-zero and re-checksum the block) when tokens are overwritten.
 *
 * Returns KVCS_EINVAL for the argument errors of kvcs_block_checksums, a
 * STATE cache, a missing key pointer, a value pointer given for a LATENT
 * cache (or missing for another), or key/value pointers not 8-byte aligned;
 * KVCS_EUNSUPPORTED when a token's row (num_heads * head_bytes) is 1 GiB or
 * more.
 */
int kvcs_write_kv(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
                  int64_t num_tokens, const void *const *keys,
                  const void *const *values, const int64_t *slot_mapping,
                  const int64_t *positions, uint64_t *block_sums, uint32_t *status,
                  void *stream);

/* Which kernel and launch shape kvcs_block_checksums would use.  Filled by
 * kvcs_plan and kvcs_plan_requests; no CUDA work is enqueued. */
typedef struct kvcs_plan_info {
  int32_t kernel;        /* 0 = bulk-copy pipeline, 1 = generic direct
                            loads, 2 = both (caches the bulk kernel cannot
                            stage go to the generic one), 3 = the valid-slot
                            kernel for every launch (a call with at most two
                            positions per request over latent or HND
                            caches, or NHD caches of pages of at most 8 KiB;
                            the fields below then describe it) */
  int32_t split;         /* 1 if the bulk kernel splits positions across CTAs
                            (output zeroed first, partial sums added with
                            64-bit atomics; the generic kernel always adds) */
  int32_t launches;      /* kernel launches per call (one per cache group) */
  int32_t memsets;       /* output-zeroing launches per call (0 or 1): one
                            small kernel before the checksum launches, which
                            overlap it (programmatic dependent launch) */
  int32_t grid;          /* CTAs per kernel launch (a call with at most two
                            positions per request, mostly partial blocks,
                            launches twice this many CTAs for its NHD
                            caches of pages over 8 KiB) */
  int32_t threads;       /* threads per CTA */
  int32_t smem_bytes;    /* dynamic shared memory per CTA */
  int32_t stage_bytes;   /* bytes per pipeline stage (bulk kernel) */
  int32_t stages;        /* pipeline stages per CTA (bulk kernel) */
  int32_t dynamic;       /* 1 if the same call given a workspace
                            (KVCS_OUT_WORKSPACE) would share the bulk
                            kernel's (or the valid-slot kernel's) last units
                            out dynamically (one more small zeroing launch
                            per call); 0 otherwise */
  int32_t slot_launches; /* launches on the valid-slot kernel (0 from
                            kvcs_plan, which does not know the requests) */
  int64_t units;         /* work units (page pieces; for the valid-slot
                            kernel, pages) per launch */
  int64_t kv_bytes_max;  /* KV bytes if every position held block_size tokens */
} kvcs_plan_info;

/*
 * kvcs_plan -- the plan for a call with these caches and sizes.
 *   num_sms  SM count to plan for; 0 = query the current device (a CUDA call).
 * Returns the same error codes as kvcs_block_checksums for bad arguments.
 */
int kvcs_plan(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
              int64_t total_positions, int32_t num_sms, kvcs_plan_info *info);

/*
 * kvcs_plan_requests -- as kvcs_plan, for a call of num_requests requests
 * (reqs->num_requests of the checksum call): a call of at most two
 * positions per request (total_positions <= 2 num_requests) sends its
 * latent and HND caches (no kernel sub-blocks), and NHD caches of pages of
 * at most 8 KiB (block_size x heads x head_bytes), 16-byte aligned and all
 * of one geometry, to the valid-slot kernel, which kvcs_plan cannot tell.
 * num_requests < 0 plans as kvcs_plan does.
 */
int kvcs_plan_requests(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
                       int64_t total_positions, int64_t num_requests, int32_t num_sms,
                       kvcs_plan_info *info);

/*
 * kvcs_selftest_wait_timeout -- check, on the caller's GPU, that a pipeline
 * wait that can never finish ends with an error status instead of hanging.
 *
 * Launches one thread that waits, with the same bounded wait the checksum
 * kernels use, on a shared-memory mbarrier phase that nothing completes.
 * After about limit_ns the wait gives up and KVCS_STATUS_TIMEOUT is OR-ed
 * into *status (a DEVICE word); the context stays usable.
 *   limit_ns  in (0, 2e9]; else KVCS_EINVAL.
 * Not part of the checksum; it exists so failure handling can be tested
 * without faulting or hanging a GPU.
 */
int kvcs_selftest_wait_timeout(uint32_t *status, int64_t limit_ns, void *stream);

/* Short text for a return code; never NULL. */
const char *kvcs_strerror(int code);

/* Kernels this library has launched in this process (all devices, all
 * threads), the output-zeroing kernel included. */
uint64_t kvcs_launch_count(void);

/* ABI version: (major << 16) | minor.  Minor 2 added kvcs_write_kv and
 * kvcs_outputs.flags (KVCS_OUT_ACCUMULATE; the field was reserved, 0).
 * Minor 3 added kvcs_outputs.workspace, read only when flags has
 * KVCS_OUT_WORKSPACE (callers built against minor 2 never set it).
 * Minor 4 added kvcs_plan_requests and kvcs_plan_info.slot_launches (the
 * struct grew: callers pass the minor-4 layout). */
int32_t kvcs_version(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* KVCS_H_ */
