// kvcs_common.cuh -- constants, device-side descriptors and helpers shared by
// the block-checksum kernels for sm_103a.
//
// What they compute (page "vllm.distributed.kv_transfer.kv_checksum.checksum",
// module docstring items 1 and 2): for every block position, over every
// (layer, KV head) slice of the block,
//     s = sum_j x_j (2j + 1),  j = t P + p,    c = sum m s,   all mod 2^64,
// with m = 2 (layer 65536 + global head) + 1 and slots at or past num_tokens
// skipped.  Everything is exact integer arithmetic mod 2^64, so any
// summation order gives the same bits.
//
// Reformulation used by both kernels' inner loops (plain algebra of the
// definition, not from the page).  Take one 16-byte chunk of a token's slice
// holding pieces p and p+1 (values x0, x1) of the token at t = t0 + slot.
// Its contribution to s is
//     x0 (2(tP + p) + 1) + x1 (2(tP + p) + 3)
//   = (x0 + x1) (2(t0 P + p) + 1) + 2P slot (x0 + x1) + 2 x1.
// So a thread that always handles the same piece pair p of the same head
// only needs three running sums over the slots it visits,
//     S = sum X,  T = sum slot X,  U = sum x1,   X = x0 + x1,
// and adds  m (B S + 2P T + 2U)  with  B = 2(t0 P + p) + 1  once per unit.
// Per 16 bytes that is three 64-bit adds and one 32x64-bit multiply-add
// instead of two full 64x64-bit products.
#pragma once

#include "kvcs_ptx.cuh"

namespace kvcs {

typedef unsigned long long u64;
typedef unsigned int u32;

#ifndef KVCS_MIN_GROUP_WARPS
#define KVCS_MIN_GROUP_WARPS 1
#endif
#ifndef KVCS_UNIT_TARGET_BYTES
#define KVCS_UNIT_TARGET_BYTES 49152
#endif

constexpr int kConsumerWarps = 8;                  // warps reducing staged data
constexpr int kMinGroupWarps = KVCS_MIN_GROUP_WARPS;  // warps sharing one unit, at least
constexpr int kBulkThreads = kConsumerWarps * 32 + 32;  // + one producer warp
constexpr int kMaxStages = 32;                     // pipeline stages, at most
constexpr int kRingSlots = kMaxStages + 2;         // per-position accumulators
constexpr int kUnitTargetBytes = KVCS_UNIT_TARGET_BYTES;
constexpr int kMaxUnitBytes = 65536;               // keeps >= 3 stages
constexpr int kSmemLimit = 232448;                 // dynamic smem per CTA
constexpr int kMaxCachesPerLaunch = 128;
constexpr int kGenericThreads = 256;

constexpr int kLayoutNHD = 0;
constexpr int kLayoutHND = 1;
constexpr int kLayoutLatent = 2;
constexpr int kLayoutXSplit = 3;
constexpr int kLayoutState = 4;

// Layout families: each has its own instance of the bulk kernel holding only
// its own staging and reduction code (a kernel holding every path ran the
// common NHD case 11% slower).
constexpr int kFamRows = 0;    // NHD and latent: rows of a page
constexpr int kFamHnd = 1;     // HND: heads of a page
constexpr int kFamXSplit = 2;  // x-split: heads of 16-byte chunks
constexpr int kFamState = 3;   // Mamba states: rows of a state
constexpr int kFamHndSub = 4;  // HND in kernel sub-blocks: heads of each sub-block
constexpr int kFamRowsMis = 5; // NHD and latent rows of pages 8 bytes past a 16-byte
                               // boundary (some or all)
constexpr int kFamHndMis = 6;  // HND (no kernel sub-blocks) heads of pages 8 bytes past
                               // a 16-byte boundary (some or all)
constexpr int kFamXSplitMis = 7;  // x-split heads of pages 8 bytes past a 16-byte
                                  // boundary (some or all)
constexpr int kNumFamilies = 8;

// Misaligned units (rows or heads): at most this many pages (one flag bit
// each in the unit's metadata).
constexpr int kMisMaxPages = 30;
// Bytes a misaligned page takes in a stage beyond its bytes: its region
// starts 16-byte aligned and its first byte sits 8 bytes in when misaligned.
constexpr int kMisPad = 16;

// Families whose units are runs of whole heads, all block_size slots of them.
__host__ __device__ constexpr bool head_family(int fam) {
  return fam == kFamHnd || fam == kFamHndSub || fam == kFamXSplit || fam == kFamHndMis ||
         fam == kFamXSplitMis;
}

// Families staged with the misaligned pages' split: the 16-byte-aligned
// interior by bulk copy, the edge words by 8-byte cp.async.
__host__ __device__ constexpr bool mis_family(int fam) {
  return fam == kFamRowsMis || fam == kFamHndMis || fam == kFamXSplitMis;
}

constexpr u32 kStatusBadBlockId = 1u;
constexpr u32 kStatusBadRequests = 2u;
constexpr u32 kStatusTimeout = 4u;

constexpr int kFlushStore = 0;   // this CTA owns the whole position: store
constexpr int kFlushAtomic = 1;  // several CTAs or launches add into it

// Per-cache constants, prepared on the host.
struct DevCache {
  const unsigned char *base;
  u64 m0;           // m of the cache's local head 0: 2 (layer H + head_offset) + 1
  u64 page_bytes;   // bytes of one page (one block of K, of V, or of rows)
  long long half_stride;   // bytes from a block's K page to its V page
  long long block_stride;  // bytes between consecutive blocks' pages
  int layout;
  int heads;        // local heads (1 for latent)
  int hb;           // bytes per head per token per half (latent: row bytes)
  int hb_shift;     // log2(hb) when hb is a power of two, else -1
  int rowb;         // bytes of one staged row: NHD heads*hb, HND hb, latent row
  int P;            // pieces per token: NHD/HND 2 hb / 8, latent row / 8
  int halves;       // 2 (K, V) or 1 (latent)
  int upp;          // units per page
  int rpu;          // rows (NHD, latent) or heads (HND) per unit
  int column;       // replica-key column the cache adds into
  int kbs;          // HND: slots per kernel sub-block (block_size if none)
  int chunks;       // HND: 1; x-split: 16-byte chunks per head (hb / 16)
  int pbytes;       // piece bytes: 8, or a state's element bytes (2 or 4)
  int run_end;      // the first cache of the launch after this one with
                    // another column (the caches are sorted by column)
};

struct Params {
  const long long *pos_offsets;
  const long long *first_position;
  const long long *num_tokens;
  const int *block_ids;
  u64 *out;                  // [total_positions][num_columns]
  u32 *status;
  long long num_requests;
  long long total_positions;
  long long units_per_pos;   // sum over this launch's caches of halves * upp
  long long total_units;     // total_positions * units_per_pos
  long long min_num_blocks;  // smallest pool of the whole call
  u64 timeout_ns;
  int block_size;
  int num_caches;
  int all_atomic;            // outputs were zeroed; every result is added
  int split;                 // CTA ranges are in units, not whole positions
  int stages;                // pipeline stages in shared memory
  int stage_bytes;           // bytes per stage (multiple of 128)
  int group_warps;           // consumer warps per group: 1, 2, 4 or 8
  int groups;                // kConsumerWarps / group_warps, <= stages
  unsigned long long *work;  // work counter (zeroed before the launch), or null:
                             // no dynamic share-out
  long long pool_start;      // with `work`: units [pool_start, total_units) are
  long long chunk_units;     // handed out in chunks of chunk_units
  int pack;                  // 1: every cache has the same geometry and each
                             // page is a unit; consecutive pages of a position
                             // are packed into one stage as far as it holds
  int full_pages;            // pack: full pages a stage holds
  int pages_per_pos;         // sum of halves over the caches
  int num_columns;           // replica-key columns of the output
  int state_call;            // the caches hold Mamba states (block position 0)
  int window_groups;         // valid-slot kernel: groups of warps that split
                             // every page's windows of valid chunks (1, or
                             // more for calls of few pages)
  DevCache caches[kMaxCachesPerLaunch];
};

// What the producer tells the consumers about one staged unit.
struct __align__(16) UnitMeta {
  long long dst;   // output word: position * num_columns + column; -1 ends
                   // the group's stream
  long long q;     // block position inside the request
  int cache;
  int half;        // 0: K or latent row, 1: V
  int first;       // NHD/latent: first slot of the unit; HND: first head
  int count;       // NHD/latent: slots in the unit; HND: heads in the unit
  int nv;          // valid slots of the block
  int mode;        // bit 0: kFlushStore or kFlushAtomic; misaligned-rows units:
                   // bit 1 + k set when page k starts 8 bytes past a boundary
  int slot;        // accumulator slot of the position
  int npages;      // consecutive pages in the unit (each packed after the
                   // previous one's valid bytes)
};

// Fixed part of the dynamic shared memory; the stages follow it.
struct SmemHeader {
  UnitMeta meta[kMaxStages];
  u64 full[kMaxStages];
  u64 empty[kMaxStages];
  u64 ring_acc[kRingSlots];
  u32 ring_cnt[kRingSlots];
};
constexpr int kHeaderBytes = (static_cast<int>(sizeof(SmemHeader)) + 127) / 128 * 128;

// The page addressing of a launch's caches, copied into shared memory by the
// wide bulk instance (after the header, before the stages): its producer
// lanes each address a different cache's page, and shared memory serves
// such reads at once where the parameter space would take them one address
// at a time.
struct PageAddr {
  const unsigned char *base;
  long long half_stride;
  long long block_stride;
};
struct WideTable {
  PageAddr page[kMaxCachesPerLaunch];
};
constexpr int kWideTableBytes = (static_cast<int>(sizeof(WideTable)) + 127) / 128 * 128;

__device__ __forceinline__ void set_status(const Params &p, u32 bit) {
  if (p.status) atomicOr(p.status, bit);
}

// ---------------------------------------------------------------------------
// Request bookkeeping (producer side)
// ---------------------------------------------------------------------------

struct PosInfo {
  long long q;
  long long block;
  int nv;
  bool skip;    // nothing to read: no valid slot, or flagged bad
  bool whole;   // every unit of the position is in this CTA's range
};

// Request r with pos_offsets[r] <= pos < pos_offsets[r+1], or -1.  Reads
// only pos_offsets[0 .. R], whatever the array holds.
__device__ long long find_request(const Params &p, long long pos) {
  long long lo = 0, hi = p.num_requests;
  while (lo < hi) {
    long long mid = (lo + hi) >> 1;
    if (p.pos_offsets[mid + 1] <= pos) lo = mid + 1; else hi = mid;
  }
  if (lo >= p.num_requests) return -1;
  if (p.pos_offsets[lo] > pos || p.pos_offsets[lo + 1] <= pos) return -1;
  return lo;
}

// The producer's view of the request holding the current position; its
// fields are reloaded only when the position leaves the request.
struct ReqCursor {
  long long r;        // request index, -1: none holds the position
  long long po0, po1; // pos_offsets[r], pos_offsets[r + 1]
  long long fp, nt;   // first_position[r], num_tokens[r]
};

// The request holding `pos`, found by the 32 lanes of a warp together
// (every lane returns the same cursor): while more than 31 requests remain
// the lanes probe 32 evenly spaced pos_offsets and keep the bucket holding
// pos, then one round of loads reads the remaining offsets with the
// candidates' first_position and num_tokens.  One round of loads when the
// call has at most 31 requests.  Reads only pos_offsets[0 .. R] and
// first_position / num_tokens [0, R), whatever the arrays hold; a position
// no request holds gives r = -1.
__device__ __forceinline__ ReqCursor req_find_warp(const Params &p, long long pos, int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  long long lo = 0, hi = p.num_requests;   // r in [lo, hi)
  while (hi - lo > 31) {
    const long long idx = lo + (hi - lo) * lane / 32;
    const unsigned below = __ballot_sync(kAll, p.pos_offsets[idx] <= pos);
    const int k = below ? 31 - __clz(below) : 0;   // last probe at or below pos
    const long long nlo = __shfl_sync(kAll, idx, k);
    const long long nhi = k < 31 ? __shfl_sync(kAll, idx, k + 1) : hi;
    lo = nlo;
    hi = nhi < hi ? nhi : hi;
    if (!below) hi = lo + 1;                      // pos below every offset: no request
  }
  const long long r = lo + lane;
  const bool in = r < hi;
  const long long a = in ? p.pos_offsets[r] : 0;
  const long long b = in ? p.pos_offsets[r + 1] : 0;
  const long long fp = in ? p.first_position[r] : 0;
  const long long nt = in ? p.num_tokens[r] : 0;
  const unsigned hit = __ballot_sync(kAll, in && a <= pos && pos < b);
  ReqCursor c;
  if (!hit) {
    c.r = -1;
    c.po0 = c.po1 = c.fp = c.nt = 0;
    return c;
  }
  const int k = __ffs(hit) - 1;
  c.r = __shfl_sync(kAll, r, k);
  c.po0 = __shfl_sync(kAll, a, k);
  c.po1 = __shfl_sync(kAll, b, k);
  c.fp = __shfl_sync(kAll, fp, k);
  c.nt = __shfl_sync(kAll, nt, k);
  return c;
}

__device__ __forceinline__ void req_load(const Params &p, ReqCursor &c, long long r) {
  c.r = r;
  if (r < 0) {
    c.po0 = c.po1 = c.fp = c.nt = 0;
    return;
  }
  c.po0 = p.pos_offsets[r];
  c.po1 = p.pos_offsets[r + 1];
  c.fp = p.first_position[r];
  c.nt = p.num_tokens[r];
}

// Move the cursor to the request holding `pos` (positions only grow): the
// next request is tried with one load before a binary search.
__device__ __forceinline__ void req_seek(const Params &p, ReqCursor &c, long long pos) {
  if (c.r >= 0 && pos >= c.po0 && pos < c.po1) return;
  long long r = -1;
  if (c.r >= 0 && c.r + 1 < p.num_requests && pos >= c.po1 &&
      pos < p.pos_offsets[c.r + 2])
    r = c.r + 1;
  if (r < 0) r = find_request(p, pos);
  req_load(p, c, r);
}

// Block position, block and valid slots of global position `pos` (request
// cursor `c` on it, block id `b`); bad tables set status bits when `report`.
__device__ PosInfo position_info_quiet(const Params &p, long long pos, const ReqCursor &c,
                                       long long b, bool report) {
  PosInfo pi;
  pi.whole = false;
  pi.q = 0;
  pi.block = 0;
  pi.nv = 0;
  pi.skip = true;
  if (c.r < 0 || c.fp < 0) {
    if (report) set_status(p, kStatusBadRequests);
    return pi;
  }
  if (b < 0 || b >= p.min_num_blocks) {
    if (report) set_status(p, kStatusBadBlockId);
    return pi;
  }
  const long long q = c.fp + (pos - c.po0);
  // Tokens of this block below num_tokens: slots [0, nv).  A Mamba state
  // block is the running state at position 0, whatever num_tokens is.
  const long long bs = p.block_size;
  long long nv = 0;
  if (p.state_call) {
    nv = q == 0 ? 1 : 0;
  } else if (q <= c.nt / bs) {  // q * bs <= nt without overflow
    nv = c.nt - q * bs;
    if (nv > bs) nv = bs;
  }
  pi.q = q;
  pi.block = b;
  pi.nv = static_cast<int>(nv);
  pi.skip = nv <= 0;
  return pi;
}

// As position_info_quiet, for the bulk kernel's producer lane: also whether
// every unit of the position lies in this CTA's range [u_begin, u_end).
__device__ __forceinline__ PosInfo position_info(const Params &p, long long pos,
                                                 const ReqCursor &c, long long b,
                                                 long long u_begin, long long u_end) {
  PosInfo pi = position_info_quiet(p, pos, c, b, true);
  pi.whole = (pos * p.units_per_pos >= u_begin) && ((pos + 1) * p.units_per_pos <= u_end);
  return pi;
}

// Three 16-byte shared-memory stores of one unit's metadata.
__device__ __forceinline__ void store_meta(UnitMeta *dst, long long out_index, long long q,
                                           int cache, int half, int first, int count,
                                           int nv, int mode, int slot, int npages) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  d[0] = make_uint4(static_cast<u32>(out_index),
                    static_cast<u32>(static_cast<u64>(out_index) >> 32),
                    static_cast<u32>(q), static_cast<u32>(static_cast<u64>(q) >> 32));
  d[1] = make_uint4(static_cast<u32>(cache), static_cast<u32>(half),
                    static_cast<u32>(first), static_cast<u32>(count));
  d[2] = make_uint4(static_cast<u32>(nv), static_cast<u32>(mode),
                    static_cast<u32>(slot), static_cast<u32>(npages));
}

__device__ __forceinline__ u64 warp_sum(u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kvcs
