// kvcs_kernels.cuh -- the block-checksum kernels for sm_103a.
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
constexpr int kNumFamilies = 5;

// Families whose units are runs of whole heads, all block_size slots of them.
__host__ __device__ constexpr bool head_family(int fam) {
  return fam == kFamHnd || fam == kFamHndSub || fam == kFamXSplit;
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
  int pad;
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
  int ppu;                   // pages per unit: > 1 only when every cache has
                             // the same geometry and a page fits a unit
  int pages_per_pos;         // sum of halves over the caches
  int num_columns;           // replica-key columns of the output
  int state_call;            // the caches hold Mamba states (block position 0)
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
  int mode;        // kFlushStore or kFlushAtomic
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

__device__ PosInfo position_info(const Params &p, long long pos, const ReqCursor &c,
                                 long long b, long long u_begin, long long u_end) {
  PosInfo pi;
  pi.whole = (pos * p.units_per_pos >= u_begin) &&
             ((pos + 1) * p.units_per_pos <= u_end);
  pi.q = 0;
  pi.block = 0;
  pi.nv = 0;
  pi.skip = true;
  if (c.r < 0 || c.fp < 0) {
    set_status(p, kStatusBadRequests);
    return pi;
  }
  if (b < 0 || b >= p.min_num_blocks) {
    set_status(p, kStatusBadBlockId);
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

// ---------------------------------------------------------------------------
// Consumer side: reduction of one staged unit
// ---------------------------------------------------------------------------

// How a consumer thread walks staged rows of `rowb` bytes: it always reads
// the same 16-byte column(s), so for NHD and latent units its head and piece
// pair are fixed and for HND units they change only at head boundaries.
struct ThreadMap {
  int rowb;    // geometry this map was made for (-1: none yet)
  int cols;    // 16-byte columns per row
  int col0;    // first column (== cols: this thread is idle)
  int cstep;   // column stride
  int rl;      // first row
  int rstep;   // row stride
  int gtid;    // thread index within the consumer group
  int nt;      // threads per consumer group
};

__device__ __forceinline__ void make_map(ThreadMap &t, int rowb, int gtid,
                                         int group_threads) {
  t.rowb = rowb;
  t.gtid = gtid;
  t.nt = group_threads;
  t.cols = rowb >> 4;
  if (t.cols <= group_threads) {
    t.rstep = group_threads / t.cols;
    t.rl = gtid / t.cols;
    t.col0 = gtid - t.rl * t.cols;
    t.cstep = t.cols;
    if (t.rl >= t.rstep) t.col0 = t.cols;
  } else {
    t.rstep = 1;
    t.rl = 0;
    t.col0 = gtid;
    t.cstep = group_threads;
  }
}

// Running sums S, T, U over slots [s_lo, s_hi) of one (head, 16-byte column)
// group whose slot s is staged at p0 + (s - s_off) * stride (s >= s_off);
// eight independent shared loads per iteration.
__device__ __forceinline__ void accum_slots(const unsigned char *p0, size_t stride,
                                            int s_lo, int s_hi, int s_off, u64 &S,
                                            u64 &T, u64 &U) {
  int s = s_lo;
  for (; s + 7 < s_hi; s += 8) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = *reinterpret_cast<const uint4 *>(p0 + static_cast<size_t>(s + k - s_off) * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const u64 x0 = (static_cast<u64>(v[k].y) << 32) | v[k].x;
      const u64 x1 = (static_cast<u64>(v[k].w) << 32) | v[k].z;
      const u64 X = x0 + x1;
      S += X;
      U += x1;
      T += static_cast<u64>(static_cast<u32>(s + k)) * X;
    }
  }
  for (; s < s_hi; ++s) {
    const uint4 v =
        *reinterpret_cast<const uint4 *>(p0 + static_cast<size_t>(s - s_off) * stride);
    const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
    const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
    const u64 X = x0 + x1;
    S += X;
    U += x1;
    T += static_cast<u64>(static_cast<u32>(s)) * X;
  }
}

// As accum_slots over all nv slots of an x-split group (a contiguous run of
// 16-byte rows at gp), starting at slot s0 and wrapping: groups start at
// different slots so a warp's reads spread over the shared-memory banks;
// four independent loads per iteration.
__device__ __forceinline__ void accum_slots_rotated(const unsigned char *gp, int s0,
                                                    int nv, u64 &S, u64 &T, u64 &U) {
  int k = 0;
  for (; k + 3 < nv; k += 4) {
    int sl[4];
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sl[i] = s0 + k + i;
      if (sl[i] >= nv) sl[i] -= nv;
      v[i] = *reinterpret_cast<const uint4 *>(gp + static_cast<size_t>(sl[i]) * 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const u64 x0 = (static_cast<u64>(v[i].y) << 32) | v[i].x;
      const u64 x1 = (static_cast<u64>(v[i].w) << 32) | v[i].z;
      const u64 X = x0 + x1;
      S += X;
      U += x1;
      T += static_cast<u64>(static_cast<u32>(sl[i])) * X;
    }
  }
  for (; k < nv; ++k) {
    int sl = s0 + k;
    if (sl >= nv) sl -= nv;
    const uint4 v = *reinterpret_cast<const uint4 *>(gp + static_cast<size_t>(sl) * 16);
    const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
    const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
    const u64 X = x0 + x1;
    S += X;
    U += x1;
    T += static_cast<u64>(static_cast<u32>(sl)) * X;
  }
}

// As accum_slots for an HND group in a sub-blocked stage: slot s of the
// group is at p0 + (s / kbs) * sub_bytes + (s % kbs) * hb; eight independent
// loads per iteration, whatever sub-blocks they fall in.
__device__ __forceinline__ void accum_slots_sub(const unsigned char *p0, int hb, int kbs,
                                                size_t sub_bytes, int nv, u64 &S, u64 &T,
                                                u64 &U) {
  int s = 0;
  // When kbs is a multiple of 4 a run of four slots never straddles a
  // sub-block: track (sub-block, offset) incrementally, one address per run,
  // two runs (eight independent loads) per iteration.
  const bool whole = (kbs & 3) == 0;
  int sb4 = 0, so4 = 0;
  for (; s + 7 < nv; s += 8) {
    uint4 v[8];
    if (whole) {
#pragma unroll
      for (int run = 0; run < 2; ++run) {
        const unsigned char *b = p0 + sb4 * sub_bytes + static_cast<size_t>(so4) * hb;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[run * 4 + i] = *reinterpret_cast<const uint4 *>(b + static_cast<size_t>(i) * hb);
        so4 += 4;
        if (so4 == kbs) {
          so4 = 0;
          ++sb4;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sb = (s + i) / kbs;
        v[i] = *reinterpret_cast<const uint4 *>(
            p0 + sb * sub_bytes + static_cast<size_t>(s + i - sb * kbs) * hb);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const u64 x0 = (static_cast<u64>(v[i].y) << 32) | v[i].x;
      const u64 x1 = (static_cast<u64>(v[i].w) << 32) | v[i].z;
      const u64 X = x0 + x1;
      S += X;
      U += x1;
      T += static_cast<u64>(static_cast<u32>(s + i)) * X;
    }
  }
  for (; s < nv; ++s) {
    const int sb = s / kbs;
    const uint4 v = *reinterpret_cast<const uint4 *>(
        p0 + sb * sub_bytes + static_cast<size_t>(s - sb * kbs) * hb);
    const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
    const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
    const u64 X = x0 + x1;
    S += X;
    U += x1;
    T += static_cast<u64>(static_cast<u32>(s)) * X;
  }
}

// This thread's share of one staged unit's contribution to the block
// checksum (see the reformulation at the top of this file).
template <int kFam>
__device__ __forceinline__ u64 unit_sum(const DevCache &C, const UnitMeta &m,
                                        int half, const unsigned char *stage,
                                        const ThreadMap &t, u64 bsz) {
  const u64 P = static_cast<u64>(C.P);
  const u64 t0P = static_cast<u64>(m.q) * bsz * P;
  const int half_pieces = half * (C.hb >> 3);
  const int rowb = t.rowb;
  u64 acc = 0;
  if constexpr (kFam == kFamState) {
    // Mamba state unit: rows [first, first + count) of the state, each a
    // slice of global row head_offset + row whose pieces are 2- or 4-byte
    // elements weighted 2e+1 by element index e.  The 16-byte column `col`
    // of a row holds elements e0 = col*k .. e0+k-1; with A = sum x_i and
    // B = sum i x_i over them it adds (2 e0 + 1) A + 2 B.  Summed over a
    // thread's columns of one row that is SA + 2k SCA + 2 SB with
    // SA = sum A, SCA = sum col A, SB = sum B (adds and small multiplies
    // only); the row factor m0 + 2 row multiplies it once per row.
    const int nrows = m.count;
    const u32 r0 = static_cast<u32>(m.first);
    const u64 per = static_cast<u64>(16 / C.pbytes);
    const bool two = C.pbytes == 2;
    auto column = [two](const uint4 v, u64 &A, u64 &Bk) {
      if (two) {
        A = (v.x & 0xffffu) + (v.x >> 16) + (v.y & 0xffffu) + (v.y >> 16) +
            (v.z & 0xffffu) + (v.z >> 16) + (v.w & 0xffffu) + (v.w >> 16);
        Bk = (v.x >> 16) + 2u * (v.y & 0xffffu) + 3u * (v.y >> 16) + 4u * (v.z & 0xffffu) +
             5u * (v.z >> 16) + 6u * (v.w & 0xffffu) + 7u * (v.w >> 16);
      } else {
        A = static_cast<u64>(v.x) + v.y + v.z + v.w;
        Bk = static_cast<u64>(v.y) + 2ull * v.z + 3ull * v.w;
      }
    };
    for (int r = t.rl; r < nrows; r += t.rstep) {
      u64 SA = 0, SCA = 0, SB = 0;
      const unsigned char *rowp = stage + static_cast<size_t>(r) * rowb;
      int col = t.col0;
      // four columns per iteration: four independent shared loads in flight
      for (; col + 3 * t.cstep < t.cols; col += 4 * t.cstep) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = *reinterpret_cast<const uint4 *>(rowp + ((col + k * t.cstep) << 4));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          u64 A, Bk;
          column(v[k], A, Bk);
          SA += A;
          SCA += static_cast<u64>(static_cast<u32>(col + k * t.cstep)) * A;
          SB += Bk;
        }
      }
      for (; col < t.cols; col += t.cstep) {
        u64 A, Bk;
        column(*reinterpret_cast<const uint4 *>(rowp + (col << 4)), A, Bk);
        SA += A;
        SCA += static_cast<u64>(static_cast<u32>(col)) * A;
        SB += Bk;
      }
      const u64 mrow = C.m0 + 2ull * static_cast<u64>(r0 + static_cast<u32>(r));
      acc += mrow * (SA + 2ull * per * SCA + 2ull * SB);
    }
  } else if constexpr (kFam == kFamRows) {
    const int nrows = m.count;
    const u32 r0 = static_cast<u32>(m.first);
    for (int col = t.col0; col < t.cols; col += t.cstep) {
      int h_col, p_col;
      if (C.layout == kLayoutNHD) {
        const int cb = col << 4;
        h_col = C.hb_shift >= 0 ? (cb >> C.hb_shift) : cb / C.hb;
        p_col = ((cb - h_col * C.hb) >> 3) + half_pieces;
      } else {
        h_col = 0;
        p_col = col << 1;
      }
      u64 S = 0, T = 0, U = 0;
      const unsigned char *sp = stage + static_cast<size_t>(t.rl) * rowb + (col << 4);
      const size_t step = static_cast<size_t>(t.rstep) * rowb;
      int r = t.rl;
      // eight rows per iteration: eight independent shared loads in flight
      for (; r + 7 * t.rstep < nrows; r += 8 * t.rstep, sp += 8 * step) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = *reinterpret_cast<const uint4 *>(sp + k * step);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const u64 x0 = (static_cast<u64>(v[k].y) << 32) | v[k].x;
          const u64 x1 = (static_cast<u64>(v[k].w) << 32) | v[k].z;
          const u64 X = x0 + x1;
          S += X;
          U += x1;
          T += static_cast<u64>(r0 + static_cast<u32>(r + k * t.rstep)) * X;
        }
      }
      for (; r < nrows; r += t.rstep, sp += step) {
        const uint4 v = *reinterpret_cast<const uint4 *>(sp);
        const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
        const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
        const u64 X = x0 + x1;
        S += X;
        U += x1;
        T += static_cast<u64>(r0 + static_cast<u32>(r)) * X;
      }
      const u64 mh = C.m0 + 2ull * static_cast<u64>(h_col);
      const u64 B = 2ull * (t0P + static_cast<u64>(p_col)) + 1ull;
      acc += mh * (B * S + 2ull * P * T + 2ull * U);
    }
  } else {
    // HND and x-split units: heads [first, first + count) staged as they lie
    // in the page, all block_size slots of them (the valid ones are the
    // first nv):
    //   HND       [sub-block][head][kbs][hb]   (one sub-block unless the
    //             attention kernel splits blocks)
    //   x-split   [head][chunk][block_size][16]
    // A thread owns whole groups (head, 16-byte column of the head's bytes):
    // head and piece pair are fixed for a group, so the thread walks its nv
    // slots with the running sums and weights the group once.
    const int nv = m.nv;
    const int bsi = static_cast<int>(bsz);
    const int cpr = C.hb >> 4;                 // 16-byte columns per head
    const int groups = m.count * cpr;
    for (int g = t.gtid; g < groups; g += t.nt) {
      const int hl = g / cpr;
      const int col = g - hl * cpr;
      u64 S = 0, T = 0, U = 0;
      if constexpr (kFam == kFamXSplit) {
        // the group's slots are one contiguous run of 16-byte rows; start
        // at a group-dependent slot so a warp's reads spread over the banks
        const unsigned char *gp = stage + static_cast<size_t>(g) * bsi * 16;
        accum_slots_rotated(gp, g % nv, nv, S, T, U);
      } else if constexpr (kFam == kFamHnd) {
        accum_slots(stage + static_cast<size_t>(hl) * bsi * C.hb + (col << 4),
                    static_cast<size_t>(C.hb), 0, nv, 0, S, T, U);
      } else {
        // sub-block sb holds slots [sb*kbs, (sb+1)*kbs) of every head
        accum_slots_sub(stage + static_cast<size_t>(hl) * C.kbs * C.hb + (col << 4), C.hb,
                        C.kbs, static_cast<size_t>(m.count) * C.kbs * C.hb, nv, S, T, U);
      }
      const u64 mh = C.m0 + 2ull * static_cast<u64>(m.first + hl);
      const u64 B = 2ull * (t0P + static_cast<u64>((col << 1) + half_pieces)) + 1ull;
      acc += mh * (B * S + 2ull * P * T + 2ull * U);
    }
  }
  return acc;
}

__device__ __forceinline__ u64 warp_sum(u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Write a finished (position, column) checksum: a plain store when this CTA
// holds every unit of the position, else a 64-bit atomic add into the
// pre-zeroed output.
__device__ __forceinline__ void finalize_slot(const Params &p, SmemHeader *hdr,
                                              int slot, long long dst, int mode) {
  __threadfence_block();
  const u64 total = atomicAdd(&hdr->ring_acc[slot], 0ull);
  if (mode == kFlushStore) p.out[dst] = total;
  else atomicAdd(p.out + dst, total);
}

// ---------------------------------------------------------------------------
// The bulk-copy pipeline kernel
// ---------------------------------------------------------------------------
//
// Persistent: CTA g owns a contiguous range of work units.  A unit is a run
// of whole rows of one page (one block's K, its V, or its latent rows), or
// of whole heads for HND, of about 16 KiB; the stage size is the launch's
// largest unit, and as many stages as fit in shared memory form a ring.
// When the positions outnumber the CTAs the ranges are whole positions and
// every result is stored once, without atomics; otherwise the ranges are cut
// at unit granularity and positions shared by two CTAs are combined with
// 64-bit atomics into the pre-zeroed output.
//
// Warp 0, lane 0 is the producer: it walks the range, turns (position,
// cache, half) into page addresses through the block table and issues one
// bulk copy per unit (one per head for a partial HND block) into the next
// stage, signalling the stage's "full" mbarrier by transaction bytes.  The
// consumer warps form `groups` groups of `group_warps` warps; emitted unit i
// goes to group i % groups, which reduces it, adds its share into the
// position's accumulator slot and releases the stage on its "empty" mbarrier.
//
// Parity waits only tell a phase from the one before it, so a waiter must
// never be two phases ahead.  Stage s holds units s, s + NS, s + 2 NS, ...
// consumed by different groups; before waiting for fill f of stage s a group
// therefore first waits for the release of fill f - 1.  That wait is itself
// safe because groups <= stages: the group has consumed its own previous
// unit, so every unit up to f - 1's was emitted, and the producer emitted
// fill f - 1 only after fill f - 2 was released.
//
// A (position, column) slot counts the contributions: each consumer warp
// adds 1 per unit, and the producer subtracts (warps per group) x (units it
// emitted) once the column of the position is done.  Whoever brings the count back to zero writes
// the result, so no CTA-wide barrier is needed and a warp that gave up on a
// timed-out wait can never block another.  Slots are reused kRingSlots
// positions later; since a stage is refilled only after it was released, and
// a contribution is made before its stage is released, a slot's last user
// has finished long before the producer re-initialises it.
//
// Every wait is bounded; a wait that runs out sets KVCS_STATUS_TIMEOUT and
// the kernel returns without hanging.
//
// kFam is the layout family of every cache in the launch.
template <int kFam>
__global__ void __launch_bounds__(kBulkThreads, 1)
    kvcs_bulk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  SmemHeader *hdr = reinterpret_cast<SmemHeader *>(smem);
  unsigned char *stages = smem + kHeaderBytes;
  const int NS = p.stages;
  const int SB = p.stage_bytes;

  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(ptx::smem_addr(&hdr->full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&hdr->empty[s]), p.group_warps);
    }
    ptx::fence_barrier_init();
  }
  __syncthreads();

  // This CTA's unit range.
  long long u_begin, u_end;
  const long long G = gridDim.x, g = blockIdx.x;
  if (p.split) {
    u_begin = p.total_units * g / G;
    u_end = p.total_units * (g + 1) / G;
  } else {
    u_begin = p.total_positions * g / G * p.units_per_pos;
    u_end = p.total_positions * (g + 1) / G * p.units_per_pos;
  }

  if (tid < 32) {
    if (tid != 0) return;
    // ------------------------------ producer ------------------------------
    if (g == 0 && p.num_requests >= 0) {
      if (p.pos_offsets[0] != 0 || p.pos_offsets[p.num_requests] != p.total_positions)
        set_status(p, kStatusBadRequests);
    }
    const u64 policy = ptx::policy_evict_first();
    const long long U = p.units_per_pos;
    const long long bs = p.block_size;
    int s = 0;          // stage of the next unit
    u32 f = 0;          // fill number of that stage
    u32 it = 0;         // units emitted
    u32 seq = 0;        // positions that got an accumulator slot
    bool aborted = false;
    if (u_begin < u_end) {
      long long pos = u_begin / U;
      const int k = static_cast<int>(u_begin - pos * U);
      int ci = 0, half = 0, sub = 0;
      if (p.ppu > 1) {
        const int page = k * p.ppu;
        ci = page / p.caches[0].halves;
        half = page - ci * p.caches[0].halves;
      } else {
        int kk = k;
        while (kk >= p.caches[ci].halves * p.caches[ci].upp) {
          kk -= p.caches[ci].halves * p.caches[ci].upp;
          ++ci;
        }
        half = kk / p.caches[ci].upp;
        sub = kk - half * p.caches[ci].upp;
      }
      ReqCursor rc;
      rc.r = -1;
      req_seek(p, rc, pos);
      long long b_cur = p.block_ids[pos];
      long long b_next = pos + 1 < p.total_positions ? p.block_ids[pos + 1] : 0;
      PosInfo cur = position_info(p, pos, rc, b_cur, u_begin, u_end);
      int mode = (cur.whole && !p.all_atomic) ? kFlushStore : kFlushAtomic;
      int slot = 0;
      u32 n_emit = 0;
      int col = p.caches[ci].column;
      for (long long u = u_begin; u < u_end; ++u) {
        const DevCache &C = p.caches[ci];
        // One accumulator slot per (position, column); the caches arrive
        // sorted by column, so a column's units are consecutive.
        const long long dst = pos * p.num_columns + col;
        int npg = 1;
        if (p.ppu > 1) npg = min(p.ppu, p.pages_per_pos - (ci * C.halves + half));
        if (!cur.skip) {
          const int first = sub * C.rpu;
          int count;
          u32 pbytes;   // bytes copied per page of the unit
          u32 pstride;  // bytes a page of the unit occupies in the stage
          if constexpr (head_family(kFam)) {
            // whole-slot runs of the unit's heads, staged as in memory
            count = max(0, min(C.rpu, C.heads - first));
            pstride = static_cast<u32>(count) * static_cast<u32>(bs) * static_cast<u32>(C.hb);
            pbytes = pstride;
            if constexpr (kFam == kFamHndSub) {
              const int nsb = (cur.nv + C.kbs - 1) / C.kbs;  // sub-blocks with valid slots
              pbytes = static_cast<u32>(count) * static_cast<u32>(nsb * C.kbs) *
                       static_cast<u32>(C.hb);
            }
          } else if constexpr (kFam == kFamState) {
            count = max(0, min(C.rpu, C.heads - first));
            pbytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
            pstride = pbytes;
          } else {
            count = max(0, min(C.rpu, cur.nv - first));
            pbytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
            pstride = pbytes;
          }
          if (pbytes > 0) {
            if (!ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->empty[s]), (f & 1u) ^ 1u,
                                        p.timeout_ns)) {
              set_status(p, kStatusTimeout);
              aborted = true;
              break;
            }
            if (n_emit == 0) {
              slot = static_cast<int>(seq % kRingSlots);
              ++seq;
              hdr->ring_acc[slot] = 0ull;
              hdr->ring_cnt[slot] = 0u;
            }
            store_meta(&hdr->meta[s], dst, cur.q, ci, half, first, count, cur.nv,
                       mode, slot, npg);
            const u32 fb = ptx::smem_addr(&hdr->full[s]);
            ptx::mbar_arrive_expect_tx(fb, pbytes * static_cast<u32>(npg));
            u32 dst = ptx::smem_addr(stages + static_cast<size_t>(s) * SB);
            int pci = ci, phalf = half;
            for (int k2 = 0; k2 < npg; ++k2) {
              const DevCache &D = p.caches[pci];
              const unsigned char *page = D.base +
                  static_cast<long long>(phalf) * D.half_stride +
                  cur.block * D.block_stride;
              if constexpr (kFam == kFamHndSub) {
                // [sub-block][heads][kbs][hb]: in each sub-block that holds
                // valid slots the unit's heads are one contiguous run; when
                // the unit has every head those runs are one range
                const u64 sub_page = static_cast<u64>(D.heads) * D.kbs * D.hb;
                const u32 run = static_cast<u32>(count) * static_cast<u32>(D.kbs * D.hb);
                if (count == D.heads) {
                  ptx::bulk_g2s(dst, page, pbytes, fb, policy);
                } else {
                  for (int sb = 0; sb * D.kbs < cur.nv; ++sb)
                    ptx::bulk_g2s(dst + static_cast<u32>(sb) * run,
                                  page + static_cast<u64>(sb) * sub_page +
                                      static_cast<u64>(first) * D.kbs * D.hb,
                                  run, fb, policy);
                }
              } else if constexpr (head_family(kFam)) {
                // [heads][block_size][hb] or [heads][chunks][block_size][16]:
                // the unit's heads are one contiguous run of whole slots
                ptx::bulk_g2s(dst, page + static_cast<u64>(first) * bs * D.hb, pstride,
                              fb, policy);
              } else {
                ptx::bulk_g2s(dst, page + static_cast<u64>(first) * D.rowb, pbytes,
                              fb, policy);
              }
              dst += pstride;
              if (++phalf == D.halves) {
                phalf = 0;
                ++pci;
              }
            }
            ++it;
            ++n_emit;
            if (++s == NS) {
              s = 0;
              ++f;
            }
          }
        }
        // advance the cursor past this unit
        bool pos_done = false;
        if (p.ppu > 1) {
          // every cache has C.halves halves when pages are packed
          const int flat = ci * C.halves + half + npg;
          ci = flat / C.halves;
          half = flat - ci * C.halves;
          pos_done = ci >= p.num_caches;
        } else if (++sub == C.upp) {
          sub = 0;
          if (++half == C.halves) {
            half = 0;
            pos_done = ++ci == p.num_caches;
          }
        }
        if (pos_done) ci = 0;
        if (pos_done || u + 1 == u_end || p.caches[ci].column != col) {
          // close the (position, column): this thread's share of the count
          if (n_emit > 0) {
            const u32 delta = 0u - static_cast<u32>(p.group_warps) * n_emit;
            const u32 prev = atomicAdd(&hdr->ring_cnt[slot], delta);
            if (prev + delta == 0u) finalize_slot(p, hdr, slot, dst, mode);
          } else if (cur.whole && !p.all_atomic) {
            p.out[dst] = 0ull;
          }
          n_emit = 0;
        }
        col = p.caches[ci].column;
        if (pos_done && u + 1 < u_end) {
          ++pos;
          b_cur = b_next;
          b_next = pos + 1 < p.total_positions ? p.block_ids[pos + 1] : 0;
          req_seek(p, rc, pos);
          cur = position_info(p, pos, rc, b_cur, u_begin, u_end);
          mode = (cur.whole && !p.all_atomic) ? kFlushStore : kFlushAtomic;
        }
      }
    }
    if (!aborted) {
      // one end-of-stream marker per consumer group
      for (int k = 0; k < p.groups; ++k) {
        if (!ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->empty[s]), (f & 1u) ^ 1u,
                                    p.timeout_ns)) {
          set_status(p, kStatusTimeout);
          break;
        }
        hdr->meta[s].dst = -1;
        ptx::mbar_arrive(ptx::smem_addr(&hdr->full[s]));
        ++it;
        if (++s == NS) {
          s = 0;
          ++f;
        }
      }
    }
    // Wait (bounded) until every copy this thread issued has landed, so no
    // bulk copy is still writing into shared memory when the CTA exits.
    for (int st = 0; st < NS; ++st) {
      if (it > static_cast<u32>(st)) {
        const u32 last = (it - 1 - st) / static_cast<u32>(NS);
        ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->full[st]), last & 1u, p.timeout_ns);
      }
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  const int cw = (tid >> 5) - 1;              // consumer warp 0..7
  const int gw = p.group_warps;
  const int group = cw / gw;
  const int gtid = (cw - group * gw) * 32 + (tid & 31);
  const int lane = tid & 31;
  const u64 bsz = static_cast<u64>(p.block_size);
  ThreadMap map;
  map.rowb = -1;
  int s = group;       // stage of this group's next unit (groups <= stages)
  u32 f = 0;           // its fill number
  while (true) {
    // fill f - 1 of this stage (another group's unit) must be released
    // before fill f can be told apart from fill f - 2
    if (f > 0 && !ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->empty[s]),
                                         (f - 1u) & 1u, p.timeout_ns)) {
      set_status(p, kStatusTimeout);
      return;
    }
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->full[s]), f & 1u, p.timeout_ns)) {
      set_status(p, kStatusTimeout);
      return;
    }
    const UnitMeta m = hdr->meta[s];
    if (m.dst < 0) break;
    const unsigned char *sp = stages + static_cast<size_t>(s) * SB;
    int ci = m.cache, half = m.half;
    u64 v = 0;
    for (int k = 0; k < m.npages; ++k) {
      const DevCache &C = p.caches[ci];
      if (C.rowb != map.rowb) make_map(map, C.rowb, gtid, gw * 32);
      v += unit_sum<kFam>(C, m, half, sp, map, bsz);
      sp += head_family(kFam)
                ? static_cast<size_t>(m.count) * static_cast<size_t>(bsz) * C.hb
                : static_cast<size_t>(m.count) * C.rowb;
      if (++half == C.halves) {
        half = 0;
        ++ci;
      }
    }
    v = warp_sum(v);
    if (lane == 0) {
      atomicAdd(&hdr->ring_acc[m.slot], v);
      __threadfence_block();
      const u32 prev = atomicAdd(&hdr->ring_cnt[m.slot], 1u);
      if (prev + 1u == 0u) finalize_slot(p, hdr, m.slot, m.dst, m.mode);
      ptx::mbar_arrive(ptx::smem_addr(&hdr->empty[s]));
    }
    s += p.groups;
    if (s >= NS) {
      s -= NS;
      ++f;
    }
  }
}

// Dynamic shared memory of a launch with `stages` stages of `stage_bytes`.
constexpr int bulk_smem_bytes(int stages, int stage_bytes) {
  return kHeaderBytes + stages * stage_bytes;
}

// ---------------------------------------------------------------------------
// Generic kernel: direct loads, any geometry the ABI accepts
// ---------------------------------------------------------------------------
//
// Used for caches the bulk kernel cannot stage: pools or strides not 16-byte
// aligned, per-head bytes not a multiple of 16, rows larger than a stage,
// state rows of any size.  Work items are (position, cache) pairs, taken
// grid-stride by CTAs of 256 threads; a CTA's threads stride over the item's
// valid pieces in logical order and weight each piece directly.  Each item's
// sum is added with a 64-bit atomic into the pre-zeroed output word of its
// (position, column), so a few positions with large states still spread
// over the whole GPU.
__device__ __forceinline__ u64 load_piece(const unsigned char *p, int bytes) {
  if (bytes == 8) return __ldg(reinterpret_cast<const u64 *>(p));
  if (bytes == 4) return __ldg(reinterpret_cast<const unsigned int *>(p));
  return __ldg(reinterpret_cast<const unsigned short *>(p));
}

// A state block whose rows are short, read as a flat run of 16-byte chunks
// (the block starts 16-byte aligned and its size is a multiple of 16): the
// chunk's elements are walked in order, each weighted 2e+1 by its index e
// within its row, and a row's part is multiplied by the row factor when the
// row ends or the chunk does.  Element sizes 2 and 4 divide 16, so no
// element straddles two chunks.
template <int kPb>
__device__ __forceinline__ u64 state_chunk_sum(const uint4 v, long long c, u32 epr, u64 m0) {
  constexpr u32 kEpc = 16 / kPb;  // elements per chunk
  const u32 w[4] = {v.x, v.y, v.z, v.w};
  const u32 e0 = static_cast<u32>(c) * kEpc;
  const u32 row = e0 / epr;
  u32 e = e0 - row * epr;
  u64 mrow = m0 + 2ull * row;
  u64 part = 0, acc = 0;
#pragma unroll
  for (u32 k = 0; k < kEpc; ++k) {
    const u32 x = kPb == 2 ? (w[k >> 1] >> ((k & 1) * 16)) & 0xffffu : w[k];
    part += static_cast<u64>(x) * (2u * e + 1u);
    if (++e == epr) {
      acc += mrow * part;
      part = 0;
      e = 0;
      mrow += 2ull;
    }
  }
  return acc + mrow * part;
}

template <int kPb>
__device__ __forceinline__ u64 state_flat_sum(const unsigned char *blk, long long nchunks,
                                              u32 epr, u64 m0, int tid) {
  const uint4 *src = reinterpret_cast<const uint4 *>(blk);
  u64 acc = 0;
  long long c = tid;
  // four chunks per thread in flight
  for (; c + 3 * kGenericThreads < nchunks; c += 4 * kGenericThreads) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(src + c + k * kGenericThreads);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc += state_chunk_sum<kPb>(v[k], c + k * kGenericThreads, epr, m0);
  }
  for (; c < nchunks; c += kGenericThreads) acc += state_chunk_sum<kPb>(__ldg(src + c), c, epr, m0);
  return acc;
}

__global__ void __launch_bounds__(kGenericThreads)
    kvcs_generic_kernel(const __grid_constant__ Params p) {
  __shared__ u64 red[kGenericThreads / 32];
  const int tid = threadIdx.x;
  const long long bs = p.block_size;
  if (blockIdx.x == 0 && tid == 0 && p.num_requests >= 0) {
    if (p.pos_offsets[0] != 0 || p.pos_offsets[p.num_requests] != p.total_positions)
      set_status(p, kStatusBadRequests);
  }
  const long long items = p.total_positions * p.num_caches;
  for (long long item = blockIdx.x; item < items; item += gridDim.x) {
    const long long pos = item / p.num_caches;
    const int ci = static_cast<int>(item - pos * p.num_caches);
    const DevCache &C = p.caches[ci];
    // every thread derives the same position info (uniform loads)
    const long long r = find_request(p, pos);
    long long q = 0, b = 0, nv = 0;
    bool ok = r >= 0;
    if (ok) {
      q = p.first_position[r] + (pos - p.pos_offsets[r]);
      b = p.block_ids[pos];
      const long long nt = p.num_tokens[r];
      if (p.first_position[r] < 0) ok = false;
      if (q <= nt / bs) nv = min(nt - q * bs, bs);
    }
    if (tid == 0 && ci == 0) {
      if (!ok) set_status(p, kStatusBadRequests);
      else if (b < 0 || b >= p.min_num_blocks) set_status(p, kStatusBadBlockId);
    }
    if (ok && (b < 0 || b >= p.min_num_blocks)) ok = false;
    u64 acc = 0;
    if (ok && C.layout == kLayoutState) {
      // a state block lives at position 0 only; rows are its slices and
      // its elements are the pieces
      if (q == 0) {
        const long long P = C.P;
        const unsigned char *blk = C.base + b * C.block_stride;
        const long long bytes = static_cast<long long>(C.heads) * C.hb;
        if (P <= 64 && (reinterpret_cast<uintptr_t>(blk) & 15) == 0 && (bytes & 15) == 0 &&
            bytes / C.pbytes < (1LL << 31)) {
          // short rows (e.g. conv states), aligned: flat 16-byte chunks
          acc = C.pbytes == 2 ? state_flat_sum<2>(blk, bytes >> 4, static_cast<u32>(P), C.m0, tid)
                              : state_flat_sum<4>(blk, bytes >> 4, static_cast<u32>(P), C.m0, tid);
        } else if (P <= 64) {
          // short rows, unaligned: one row per thread
          for (long long row = tid; row < C.heads; row += kGenericThreads) {
            const unsigned char *rp = blk + row * C.hb;
            u64 s = 0;
            for (long long pc = 0; pc < P; ++pc)
              s += load_piece(rp + pc * C.pbytes, C.pbytes) * (2ull * static_cast<u64>(pc) + 1ull);
            acc += s * (C.m0 + 2ull * static_cast<u64>(row));
          }
        } else {
          // long rows: the CTA strides over each row's elements
          for (long long row = 0; row < C.heads; ++row) {
            const unsigned char *rp = blk + row * C.hb;
            u64 s = 0;
            for (long long pc = tid; pc < P; pc += kGenericThreads)
              s += load_piece(rp + pc * C.pbytes, C.pbytes) * (2ull * static_cast<u64>(pc) + 1ull);
            acc += s * (C.m0 + 2ull * static_cast<u64>(row));
          }
        }
      }
    } else if (ok && nv > 0) {
      const u64 t0 = static_cast<u64>(q) * static_cast<u64>(bs);
      const long long P = C.P;
      const long long per_slot = static_cast<long long>(C.heads) * P;
      const long long n = nv * per_slot;
      const int hp = C.hb >> 3;  // pieces per half
      for (long long idx = tid; idx < n; idx += kGenericThreads) {
        const long long slot = idx / per_slot;
        const long long rem = idx - slot * per_slot;
        const long long h = rem / P;
        const long long pc = rem - h * P;
        long long off;
        if (C.layout == kLayoutLatent) {
          off = b * C.block_stride + slot * C.hb + 8 * pc;
        } else {
          const long long half = pc >= hp ? 1 : 0;
          const long long e = (pc - half * hp) * 8;
          const long long page = half * C.half_stride + b * C.block_stride;
          if (C.layout == kLayoutNHD) {
            off = page + (slot * C.heads + h) * C.hb + e;
          } else if (C.layout == kLayoutXSplit) {
            off = page + ((h * (C.hb >> 4) + (e >> 4)) * bs + slot) * 16 + (e & 15);
          } else {
            const long long sb = slot / C.kbs;
            off = page + ((sb * C.heads + h) * C.kbs + (slot - sb * C.kbs)) * C.hb + e;
          }
        }
        const u64 x = __ldg(reinterpret_cast<const u64 *>(C.base + off));
        const u64 j = (t0 + static_cast<u64>(slot)) * static_cast<u64>(P) +
                      static_cast<u64>(pc);
        const u64 mh = C.m0 + 2ull * static_cast<u64>(h);
        acc += x * ((2ull * j + 1ull) * mh);
      }
    }
    acc = warp_sum(acc);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      u64 total = 0;
      for (int w = 0; w < kGenericThreads / 32; ++w) total += red[w];
      if (total) atomicAdd(p.out + pos * p.num_columns + C.column, total);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// KV write fused with the checksum (reshape_and_cache + running block sums)
// ---------------------------------------------------------------------------

constexpr int kMaxWriteCaches = 64;

struct WriteParams {
  const long long *slots;      // slot_mapping
  const long long *positions;  // token positions in their requests
  u64 *block_sums;             // running word per physical block, or null
  u32 *status;
  long long num_tokens;
  long long num_blocks;        // smallest pool of the call
  int block_size;
  int num_caches;
  int chunk;                   // 16 or 8: bytes moved per thread per step
  int caches_per_item;         // caches one warp moves for its token
  int heads_per_item;          // x-split: heads one warp moves for its tokens
  int head_chunks;             // x-split: ceil(largest head count / heads_per_item)
  DevCache c[kMaxWriteCaches];
  const unsigned char *key[kMaxWriteCaches];    // [num_tokens][heads][hb]
  const unsigned char *value[kMaxWriteCaches];  // same, or null (latent)
};

constexpr int kWriteThreads = 256;
constexpr int kWriteBatch = 8;  // chunks per lane in flight

// One cache's K and V rows of one token: moved into the page slot `o` of
// block `b` by the calling warp, up to eight chunks per lane in flight (the
// K and V chunks of one batch together); returns the lane's share of the
// token's checksum term for this cache.  Byte `off` of a row (head
// h = off / hb, byte e = off mod hb) goes to, per layout:
//   NHD, latent  o*row + off
//   HND          ((o/kbs*heads + h)*kbs + o mod kbs)*hb + e
// (x-split pages have their own kernel below.)
template <int kLayout>
__device__ __forceinline__ u64 write_token_rows(const DevCache &C, const unsigned char *srck,
                                                const unsigned char *srcv, long long bs,
                                                long long b, long long o, u64 t, int ch,
                                                int lane) {
  const int row = C.heads * C.hb;
  const int nh = row / ch;          // chunks per half
  const int n = nh * C.halves;      // chunks of the token
  unsigned char *page = const_cast<unsigned char *>(C.base) + b * C.block_stride;
  long long slot_base;              // address of byte 0 of head 0 of slot o
  long long head_step = 0;          // HND: bytes between heads
  if (kLayout == kLayoutHND) {
    const long long sb = o / C.kbs;
    slot_base = (sb * C.heads * C.kbs + (o - sb * C.kbs)) * C.hb;
    head_step = static_cast<long long>(C.kbs - 1) * C.hb;
  } else {
    slot_base = o * row;
  }
  const u64 tP = t * static_cast<u64>(C.P);
  u64 acc = 0;
  for (int base = lane; base < n; base += kWriteBatch * 32) {
    uint4 v[kWriteBatch];
#pragma unroll
    for (int k = 0; k < kWriteBatch; ++k) {
      const int idx = base + 32 * k;
      if (idx < n) {
        const bool hv = idx >= nh;
        const unsigned char *src = (hv ? srcv : srck) + (idx - (hv ? nh : 0)) * ch;
        if (ch == 16) {
          v[k] = *reinterpret_cast<const uint4 *>(src);
        } else {
          const u64 x = *reinterpret_cast<const u64 *>(src);
          v[k] = make_uint4(static_cast<u32>(x), static_cast<u32>(x >> 32), 0u, 0u);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kWriteBatch; ++k) {
      const int idx = base + 32 * k;
      if (idx >= n) break;
      const int half = idx >= nh ? 1 : 0;
      const int off = (idx - half * nh) * ch;
      const int h = C.hb_shift >= 0 ? (off >> C.hb_shift) : off / C.hb;
      const int e = off - h * C.hb;
      const long long d = kLayout == kLayoutHND ? slot_base + off + h * head_step
                                                : slot_base + off;
      unsigned char *dst = page + half * C.half_stride + d;
      const u64 x0 = (static_cast<u64>(v[k].y) << 32) | v[k].x;
      const u64 mh = C.m0 + 2ull * static_cast<u64>(h);
      const u64 w0 = 2ull * (tP + static_cast<u64>((e >> 3) + half * (C.hb >> 3))) + 1ull;
      if (ch == 16) {
        *reinterpret_cast<uint4 *>(dst) = v[k];
        const u64 x1 = (static_cast<u64>(v[k].w) << 32) | v[k].z;
        acc += mh * (x0 * w0 + x1 * (w0 + 2ull));
      } else {
        *reinterpret_cast<u64 *>(dst) = x0;
        acc += mh * (x0 * w0);
      }
    }
  }
  return acc;
}

// A warp per (token, run of caches) item, grid-stride: for each cache of its
// run it moves the token's K and V rows into the page slot and weights the
// pieces it moved; the item's total goes into its block's running word with
// one atomic add.  A run is every cache of the launch when the tokens alone
// give enough warps (prefill), down to one cache when they are few (decode).  One instance per layout family (NHD
// and latent, HND, x-split); a call with several families makes one launch
// per family.
template <int kLayout>
__global__ void __launch_bounds__(kWriteThreads, 2)
    kvcs_write_kernel(const __grid_constant__ WriteParams w) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kWriteThreads / 32);
  const long long bs = w.block_size;
  const int ch = w.chunk;
  const int cpi = w.caches_per_item;
  const long long items = w.num_tokens * ((w.num_caches + cpi - 1) / cpi);
  for (long long it = blockIdx.x * (kWriteThreads / 32) + (threadIdx.x >> 5); it < items;
       it += warps) {
    // items chunk-major: neighbouring warps take neighbouring tokens
    const int chunk = static_cast<int>(it / w.num_tokens);
    const long long i = it - static_cast<long long>(chunk) * w.num_tokens;
    const int c_lo = chunk * cpi;
    const int c_hi = min(w.num_caches, c_lo + cpi);
    const long long slot = w.slots[i];
    if (slot < 0) continue;  // padding token
    const long long b = slot / bs;
    const long long o = slot - b * bs;
    if (b >= w.num_blocks) {
      if (lane == 0 && chunk == 0 && w.status) atomicOr(w.status, kStatusBadBlockId);
      continue;
    }
    const long long t = w.positions[i];
    if (t < 0 && lane == 0 && chunk == 0 && w.status) atomicOr(w.status, kStatusBadRequests);
    u64 acc = 0;
    for (int ci = c_lo; ci < c_hi; ++ci) {
      const DevCache &C = w.c[ci];
      const long long row = static_cast<long long>(C.heads) * C.hb;
      acc += write_token_rows<kLayout>(C, w.key[ci] + i * row, w.value[ci] + i * row, bs, b, o,
                                       static_cast<u64>(t), ch, lane);
    }
    if (w.block_sums != nullptr && t >= 0) {
      acc = warp_sum(acc);
      if (lane == 0) atomicAdd(w.block_sums + b, acc);
    }
  }
}

// x-split pages keep slot o's 16-byte piece c of head h at
// ((h*hb/16 + c)*block_size + o)*16, so neighbouring slots' pieces are
// neighbours in memory.  A warp takes a run of heads of one cache for 32
// consecutive tokens (items cache-major, grid-stride; the run is every head
// unless the tokens are too few to give enough warps) and moves them
// through a shared-memory tile, one head's run of at most 16 pieces at a
// time: loads read the tokens' rows coalesced (a token's run is
// contiguous), stores give each lane one token, so lanes holding
// consecutive slots of a block store one contiguous run.  The lane weights
// its token's pieces as it stores them and adds its term to its block's
// word with one atomic.
constexpr int kXTile = 16;  // pieces per tile row

__global__ void __launch_bounds__(kWriteThreads, 2)
    kvcs_write_xsplit_kernel(const __grid_constant__ WriteParams w) {
  // per warp: 32 tokens x (kXTile + 1) pieces; the pad spreads a column's
  // reads over the banks
  __shared__ uint4 tile[kWriteThreads / 32][32 * (kXTile + 1)];
  const int lane = threadIdx.x & 31;
  uint4 *my = tile[threadIdx.x >> 5];
  const long long warps = static_cast<long long>(gridDim.x) * (kWriteThreads / 32);
  const long long bs = w.block_size;
  const long long groups = (w.num_tokens + 31) / 32;
  const int nhc = w.head_chunks;
  const long long items = groups * w.num_caches * nhc;
  for (long long it = blockIdx.x * (kWriteThreads / 32) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const long long rest = it / nhc;
    const int hk = static_cast<int>(it - rest * nhc);
    const int ci = static_cast<int>(rest / groups);
    const long long gi = rest - static_cast<long long>(ci) * groups;
    const long long i0 = gi * 32;
    const long long i = i0 + lane;
    bool live = i < w.num_tokens;
    long long b = 0, o = 0, t = -1;
    if (live) {
      const long long slot = w.slots[i];
      live = slot >= 0;  // padding token
      if (live) {
        b = slot / bs;
        o = slot - b * bs;
        if (b >= w.num_blocks) {
          if (ci == 0 && hk == 0 && w.status) atomicOr(w.status, kStatusBadBlockId);
          live = false;
        } else {
          t = w.positions[i];
          if (ci == 0 && hk == 0 && t < 0 && w.status)
            atomicOr(w.status, kStatusBadRequests);
        }
      }
    }
    const u32 live_mask = __ballot_sync(0xffffffffu, live);
    u64 acc = 0;
    {
      const DevCache &C = w.c[ci];
      const int row = C.heads * C.hb;
      const int cph = C.hb >> 4;  // pieces per head
      const u64 tP = static_cast<u64>(t) * static_cast<u64>(C.P);
      unsigned char *page = const_cast<unsigned char *>(C.base) + b * C.block_stride + o * 16;
      const long long pstep = bs * 16;  // bytes between a slot's consecutive pieces
      for (int half = 0; half < C.halves; ++half) {
        const unsigned char *src = (half ? w.value[ci] : w.key[ci]) + i0 * row;
        unsigned char *dst = page + half * C.half_stride;
        const u64 hp = static_cast<u64>(half) * (C.hb >> 3);
        const int h_hi = min(C.heads, (hk + 1) * w.heads_per_item);
        for (int h = hk * w.heads_per_item; h < h_hi; ++h) {
          const u64 mh = C.m0 + 2ull * static_cast<u64>(h);
          for (int c0 = 0; c0 < cph; c0 += kXTile) {
            const int cs = min(kXTile, cph - c0);
            // load: piece q of the tile is token q / cs, piece c0 + q % cs;
            // eight loads per lane in flight
            __syncwarp();
            const int nq = 32 * cs;
            for (int q0 = 0; q0 < nq; q0 += 32 * 8) {
              uint4 v[8];
              int at[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int q = q0 + lane + 32 * k;
                const int tk = q / cs;
                const int c = q - tk * cs;
                at[k] = -1;
                if (q < nq && ((live_mask >> tk) & 1u)) {
                  const unsigned char *sp =
                      src + static_cast<long long>(tk) * row + h * C.hb + (c0 + c) * 16;
                  if (w.chunk == 16) {
                    v[k] = *reinterpret_cast<const uint4 *>(sp);
                  } else {
                    const u64 a = *reinterpret_cast<const u64 *>(sp);
                    const u64 d = *reinterpret_cast<const u64 *>(sp + 8);
                    v[k] = make_uint4(static_cast<u32>(a), static_cast<u32>(a >> 32),
                                      static_cast<u32>(d), static_cast<u32>(d >> 32));
                  }
                  at[k] = tk * (kXTile + 1) + c;
                }
              }
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if (at[k] >= 0) my[at[k]] = v[k];
            }
            __syncwarp();
            // store: lane = token
            if (live) {
              for (int c = 0; c < cs; ++c) {
                const uint4 v = my[lane * (kXTile + 1) + c];
                unsigned char *dp = dst + static_cast<long long>(h * cph + c0 + c) * pstep;
                if (w.chunk == 16) {
                  *reinterpret_cast<uint4 *>(dp) = v;
                } else {
                  *reinterpret_cast<u64 *>(dp) = (static_cast<u64>(v.y) << 32) | v.x;
                  *reinterpret_cast<u64 *>(dp + 8) = (static_cast<u64>(v.w) << 32) | v.z;
                }
                const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
                const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
                const u64 w0 = 2ull * (tP + static_cast<u64>(2 * (c0 + c)) + hp) + 1ull;
                acc += mh * (x0 * w0 + x1 * (w0 + 2ull));
              }
            }
          }
        }
      }
    }
    if (live && w.block_sums != nullptr && t >= 0 && acc != 0) atomicAdd(w.block_sums + b, acc);
  }
}

// ---------------------------------------------------------------------------
// Row sums, tags and verification (offloaded-KV checks)
// ---------------------------------------------------------------------------

struct RowParams {
  const u64 *values;        // [n][num_columns]
  long long n;
  int num_columns;
  u64 *row_sums;            // or null
  const u64 *tags;          // or null
  const u64 *expected;      // or null
  unsigned char *mismatch;  // or null
  u32 *mismatch_count;      // or null
};

// Per position: the row's partials summed mod 2^64, XOR its tag; compared
// with the stored value when one is given.
__global__ void __launch_bounds__(256) kvcs_rows_kernel(const RowParams rp) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       i - threadIdx.x < rp.n; i += stride) {
    bool bad = false;
    if (i < rp.n) {
      u64 r = 0;
      for (int k = 0; k < rp.num_columns; ++k) r += rp.values[i * rp.num_columns + k];
      if (rp.tags) r ^= rp.tags[i];
      if (rp.row_sums) rp.row_sums[i] = r;
      if (rp.expected) {
        bad = r != rp.expected[i];
        if (rp.mismatch) rp.mismatch[i] = bad ? 1 : 0;
      }
    }
    if (rp.mismatch_count) {
      const unsigned votes = __ballot_sync(0xffffffffu, bad);
      if ((threadIdx.x & 31) == 0 && votes) atomicAdd(rp.mismatch_count, __popc(votes));
    }
  }
}

// tags[i] = (first eight bytes of hash i, little-endian) XOR fingerprint.
__global__ void __launch_bounds__(256)
    kvcs_tags_kernel(const unsigned char *hashes, long long stride, long long n,
                     u64 fingerprint, u64 *tags) {
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       i < n; i += step) {
    const unsigned char *h = hashes + i * stride;
    u64 w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) w |= static_cast<u64>(h[k]) << (8 * k);
    tags[i] = w ^ fingerprint;
  }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait
// ---------------------------------------------------------------------------

// One thread waits on a phase of a fresh mbarrier that nothing will ever
// complete (count 1, no arrival); the bounded wait must give up and report.
__global__ void kvcs_wait_selftest_kernel(u32 *status, u64 limit_ns) {
  __shared__ __align__(8) u64 bar;
  if (threadIdx.x != 0) return;
  const u32 b = ptx::smem_addr(&bar);
  ptx::mbar_init(b, 1);
  ptx::fence_barrier_init();
  if (!ptx::mbar_wait_bounded(b, 0u, limit_ns)) atomicOr(status, kStatusTimeout);
}

}  // namespace kvcs
