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

constexpr int kStageBytes = 32768;    // one pipeline stage (max unit size)
constexpr int kStages = 6;            // stages in the shared-memory ring
constexpr int kConsumerWarps = 8;     // warps reducing staged data
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kBulkThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kRing = kStages + 2;    // flush slots (see consumer_flush)
constexpr int kMaxCachesPerLaunch = 128;
constexpr int kGenericThreads = 256;

constexpr int kLayoutNHD = 0;
constexpr int kLayoutHND = 1;
constexpr int kLayoutLatent = 2;

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
  u64 half_stride;  // num_blocks * page_bytes: offset of the V half
  int layout;
  int heads;        // local heads (1 for latent)
  int hb;           // bytes per head per token per half (latent: row bytes)
  int rowb;         // bytes of one staged row: NHD heads*hb, HND hb, latent row
  int P;            // pieces per token: NHD/HND 2 hb / 8, latent row / 8
  int halves;       // 2 (K, V) or 1 (latent)
  int upp;          // units per page
  int rpu;          // rows (NHD, latent) or heads (HND) per unit
};

struct Params {
  const long long *pos_offsets;
  const long long *first_position;
  const long long *num_tokens;
  const int *block_ids;
  u64 *out;
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
  DevCache caches[kMaxCachesPerLaunch];
};

// What the producer tells the consumers about one staged unit.
struct UnitMeta {
  long long pos;   // global position index; -1 ends the stream
  long long q;     // block position inside the request
  int cache;
  int half;        // 0: K or latent row, 1: V
  int first;       // NHD/latent: first slot of the unit; HND: first head
  int count;       // NHD/latent: slots in the unit; HND: heads in the unit
  int nv;          // valid slots of the block
  int mode;        // kFlushStore or kFlushAtomic
};

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

// Step the request cursor to the one holding `pos` (positions only grow).
__device__ __forceinline__ long long advance_request(const Params &p,
                                                     long long r, long long pos) {
  if (r < 0) return find_request(p, pos);
  while (r < p.num_requests && p.pos_offsets[r + 1] <= pos) ++r;
  if (r >= p.num_requests || p.pos_offsets[r] > pos) return find_request(p, pos);
  return r;
}

__device__ PosInfo position_info(const Params &p, long long pos, long long r,
                                 long long u_begin, long long u_end) {
  PosInfo pi;
  pi.whole = (pos * p.units_per_pos >= u_begin) &&
             ((pos + 1) * p.units_per_pos <= u_end);
  pi.q = 0;
  pi.block = 0;
  pi.nv = 0;
  pi.skip = true;
  if (r < 0) {
    set_status(p, kStatusBadRequests);
    return pi;
  }
  const long long q = p.first_position[r] + (pos - p.pos_offsets[r]);
  const long long nt = p.num_tokens[r];
  const long long b = p.block_ids[pos];
  if (p.first_position[r] < 0) {
    set_status(p, kStatusBadRequests);
    return pi;
  }
  if (b < 0 || b >= p.min_num_blocks) {
    set_status(p, kStatusBadBlockId);
    return pi;
  }
  // Tokens of this block below num_tokens: slots [0, nv).
  const long long bs = p.block_size;
  long long nv = 0;
  if (q <= nt / bs) {  // q * bs <= nt without overflow
    nv = nt - q * bs;
    if (nv > bs) nv = bs;
  }
  pi.q = q;
  pi.block = b;
  pi.nv = static_cast<int>(nv);
  pi.skip = nv <= 0;
  return pi;
}

// ---------------------------------------------------------------------------
// Consumer side: reduction of one staged unit
// ---------------------------------------------------------------------------

// Sum over one staged unit of this thread's share of the block checksum.
// Staged rows are `rowb` bytes; the thread always reads the same 16-byte
// column of every row it visits, so the head and piece pair are fixed for it
// (NHD, latent) or change only at head boundaries (HND).
__device__ __forceinline__ u64 unit_sum(const DevCache &C, const UnitMeta &m,
                                        const unsigned char *stage, int ctid,
                                        u64 bsz) {
  const int rowb = C.rowb;
  const int cols = rowb >> 4;
  int col0, cstep, rl, rstep;
  if (cols <= kConsumerThreads) {
    rstep = kConsumerThreads / cols;
    rl = ctid / cols;
    if (rl >= rstep) return 0;
    col0 = ctid - rl * cols;
    cstep = cols;
  } else {
    rstep = 1;
    rl = 0;
    col0 = ctid;
    cstep = kConsumerThreads;
  }
  const u64 P = static_cast<u64>(C.P);
  const u64 t0P = static_cast<u64>(m.q) * bsz * P;
  const int half_pieces = m.half * (C.hb >> 3);
  u64 acc = 0;
  if (C.layout != kLayoutHND) {
    const int nrows = m.count;
    const u32 r0 = static_cast<u32>(m.first);
    for (int col = col0; col < cols; col += cstep) {
      int h_col, p_col;
      if (C.layout == kLayoutNHD) {
        const int cb = col << 4;
        h_col = cb / C.hb;
        p_col = ((cb - h_col * C.hb) >> 3) + half_pieces;
      } else {
        h_col = 0;
        p_col = col << 1;
      }
      u64 S = 0, T = 0, U = 0;
      const unsigned char *sp = stage + static_cast<size_t>(rl) * rowb + (col << 4);
      const size_t step = static_cast<size_t>(rstep) * rowb;
#pragma unroll 4
      for (int r = rl; r < nrows; r += rstep, sp += step) {
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
    // HND unit: heads [first, first + count), each with nv staged rows
    // (slots 0 .. nv-1) of hb bytes, packed head after head.
    const int nv = m.nv;
    const int nrows = m.count * nv;
    for (int col = col0; col < cols; col += cstep) {
      int r = rl;
      if (r >= nrows) continue;
      const u64 B = 2ull * (t0P + static_cast<u64>((col << 1) + half_pieces)) + 1ull;
      int hh = r / nv;
      int slot = r - hh * nv;
      u64 S = 0, T = 0, U = 0;
      const unsigned char *sp = stage + static_cast<size_t>(r) * rowb + (col << 4);
      const size_t step = static_cast<size_t>(rstep) * rowb;
      while (true) {
        const uint4 v = *reinterpret_cast<const uint4 *>(sp);
        const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
        const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
        const u64 X = x0 + x1;
        S += X;
        U += x1;
        T += static_cast<u64>(static_cast<u32>(slot)) * X;
        r += rstep;
        sp += step;
        slot += rstep;
        if (slot >= nv || r >= nrows) {
          const u64 mh = C.m0 + 2ull * static_cast<u64>(m.first + hh);
          acc += mh * (B * S + 2ull * P * T + 2ull * U);
          S = T = U = 0;
          if (r >= nrows) break;
          const int adv = slot / nv;
          hh += adv;
          slot -= adv * nv;
        }
      }
    }
  }
  return acc;
}

__device__ __forceinline__ u64 warp_sum(u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Combine the consumer warps' sums for one position without a CTA barrier:
// each warp adds its sum into ring slot `seq % kRing` and bumps the slot's
// count; the warp that completes the count writes the result and clears the
// slot.  A warp can run at most kStages units ahead of the slowest one (the
// producer refills a stage only after every warp released it), hence at most
// kStages flushes ahead, so kRing = kStages + 2 slots are never reused early.
// Without a barrier a warp that gave up on a timed-out wait cannot leave the
// others blocked.
__device__ __forceinline__ void consumer_flush(const Params &p, u64 *ring_acc,
                                               u32 *ring_cnt, u32 seq,
                                               long long pos, int mode, u64 acc,
                                               int lane) {
  const u64 v = warp_sum(acc);
  if (lane == 0) {
    const u32 slot = seq % kRing;
    atomicAdd(&ring_acc[slot], v);
    __threadfence_block();
    const u32 prev = atomicAdd(&ring_cnt[slot], 1u);
    if (prev == kConsumerWarps - 1) {
      __threadfence_block();
      const u64 total = atomicAdd(&ring_acc[slot], 0ull);
      ring_acc[slot] = 0;
      ring_cnt[slot] = 0;
      if (mode == kFlushStore) p.out[pos] = total;
      else atomicAdd(p.out + pos, total);
    }
  }
}

// ---------------------------------------------------------------------------
// The bulk-copy pipeline kernel
// ---------------------------------------------------------------------------
//
// Persistent: CTA g owns a contiguous range of work units.  A unit is a run
// of whole rows of one page (one block's K, its V, or its latent rows) that
// fits a 32 KiB stage; for HND a unit is a run of whole heads.  When the
// positions outnumber the CTAs the ranges are whole positions and every
// result is stored once (no atomics); otherwise they are cut at unit
// granularity and positions shared by two CTAs are combined with 64-bit
// atomics into the pre-zeroed output.
//
// Warp 0, lane 0 is the producer: it walks the range, turns (position,
// cache, half) into page addresses through the block table and issues one
// bulk copy per unit (one per head for a partial HND block) into the next
// free stage, signalling the stage's "full" mbarrier by transaction bytes.
// Warps 1..8 consume stages in order and release them on the "empty"
// mbarrier.  Every wait is bounded; a wait that runs out sets
// KVCS_STATUS_TIMEOUT and the kernel returns without hanging.
__global__ void __launch_bounds__(kBulkThreads, 1)
    kvcs_bulk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stages = smem;
  UnitMeta *meta = reinterpret_cast<UnitMeta *>(smem + kStages * kStageBytes);
  u64 *full = reinterpret_cast<u64 *>(meta + kStages);
  u64 *empty = full + kStages;
  u64 *ring_acc = empty + kStages;
  u32 *ring_cnt = reinterpret_cast<u32 *>(ring_acc + kRing);

  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(full + s), 1);
      ptx::mbar_init(ptx::smem_addr(empty + s), kConsumerWarps);
    }
    ptx::fence_barrier_init();
  }
  if (tid < kRing) {
    ring_acc[tid] = 0;
    ring_cnt[tid] = 0;
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
    u32 it = 0;
    bool aborted = false;
    if (u_begin < u_end) {
      long long pos = u_begin / U;
      int k = static_cast<int>(u_begin - pos * U);
      int ci = 0;
      while (k >= p.caches[ci].halves * p.caches[ci].upp) {
        k -= p.caches[ci].halves * p.caches[ci].upp;
        ++ci;
      }
      int half = k / p.caches[ci].upp;
      int sub = k - half * p.caches[ci].upp;
      long long r = find_request(p, pos);
      PosInfo cur = position_info(p, pos, r, u_begin, u_end);
      bool emitted = false;
      for (long long u = u_begin; u < u_end && !aborted; ++u) {
        const DevCache &C = p.caches[ci];
        if (!cur.skip) {
          int first = sub * C.rpu, count;
          u32 bytes;
          if (C.layout == kLayoutHND) {
            count = max(0, min(C.rpu, C.heads - first));
            bytes = static_cast<u32>(count) * static_cast<u32>(cur.nv) *
                    static_cast<u32>(C.hb);
          } else {
            count = max(0, min(C.rpu, cur.nv - first));
            bytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
          }
          if (bytes > 0) {
            const int s = static_cast<int>(it % kStages);
            const u32 f = it / kStages;
            if (!ptx::mbar_wait_bounded(ptx::smem_addr(empty + s), (f & 1u) ^ 1u,
                                        p.timeout_ns)) {
              set_status(p, kStatusTimeout);
              aborted = true;
              break;
            }
            UnitMeta &mm = meta[s];
            mm.pos = pos;
            mm.q = cur.q;
            mm.cache = ci;
            mm.half = half;
            mm.first = first;
            mm.count = count;
            mm.nv = cur.nv;
            mm.mode = (cur.whole && !p.all_atomic) ? kFlushStore : kFlushAtomic;
            const u32 fb = ptx::smem_addr(full + s);
            ptx::mbar_arrive_expect_tx(fb, bytes);
            const unsigned char *page = C.base +
                static_cast<u64>(half) * C.half_stride +
                static_cast<u64>(cur.block) * C.page_bytes;
            const u32 dst = ptx::smem_addr(stages + static_cast<size_t>(s) * kStageBytes);
            if (C.layout == kLayoutHND) {
              const u64 head_stride = static_cast<u64>(bs) * C.hb;
              if (cur.nv == bs) {
                ptx::bulk_g2s(dst, page + static_cast<u64>(first) * head_stride,
                              bytes, fb, policy);
              } else {
                const u32 run = static_cast<u32>(cur.nv) * static_cast<u32>(C.hb);
                for (int h = 0; h < count; ++h)
                  ptx::bulk_g2s(dst + static_cast<u32>(h) * run,
                                page + static_cast<u64>(first + h) * head_stride,
                                run, fb, policy);
              }
            } else {
              ptx::bulk_g2s(dst, page + static_cast<u64>(first) * C.rowb, bytes,
                            fb, policy);
            }
            ++it;
            emitted = true;
          }
        }
        // advance to the next unit
        if (++sub == C.upp) {
          sub = 0;
          if (++half == C.halves) {
            half = 0;
            if (++ci == p.num_caches) {
              ci = 0;
              // position finished in this CTA
              if (cur.whole && !emitted && !p.all_atomic) p.out[pos] = 0ull;
              ++pos;
              emitted = false;
              if (u + 1 < u_end) {
                r = advance_request(p, r, pos);
                cur = position_info(p, pos, r, u_begin, u_end);
              }
            }
          }
        }
      }
    }
    if (!aborted) {
      // end-of-stream marker
      const int s = static_cast<int>(it % kStages);
      const u32 f = it / kStages;
      if (ptx::mbar_wait_bounded(ptx::smem_addr(empty + s), (f & 1u) ^ 1u,
                                 p.timeout_ns)) {
        meta[s].pos = -1;
        ptx::mbar_arrive(ptx::smem_addr(full + s));
        ++it;
      } else {
        set_status(p, kStatusTimeout);
      }
    }
    // Wait (bounded) until every copy this thread issued has landed, so no
    // bulk copy is still writing into shared memory when the CTA exits.
    for (int s = 0; s < kStages; ++s) {
      if (it > static_cast<u32>(s)) {
        const u32 last = (it - 1 - s) / kStages;
        ptx::mbar_wait_bounded(ptx::smem_addr(full + s), last & 1u, p.timeout_ns);
      }
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  const int ctid = tid - 32;
  const int lane = tid & 31;
  const u64 bsz = static_cast<u64>(p.block_size);
  u64 acc = 0;
  long long cur_pos = -1;
  int cur_mode = kFlushStore;
  u32 seq = 0;
  for (u32 it = 0;; ++it) {
    const int s = static_cast<int>(it % kStages);
    const u32 f = it / kStages;
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(full + s), f & 1u, p.timeout_ns)) {
      set_status(p, kStatusTimeout);
      return;
    }
    const UnitMeta m = meta[s];
    if (m.pos < 0) break;
    if (m.pos != cur_pos) {
      if (cur_pos >= 0) {
        consumer_flush(p, ring_acc, ring_cnt, seq, cur_pos, cur_mode, acc, lane);
        ++seq;
      }
      cur_pos = m.pos;
      cur_mode = m.mode;
      acc = 0;
    }
    acc += unit_sum(p.caches[m.cache], m,
                    stages + static_cast<size_t>(s) * kStageBytes, ctid, bsz);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(empty + s));
  }
  if (cur_pos >= 0) consumer_flush(p, ring_acc, ring_cnt, seq, cur_pos, cur_mode, acc, lane);
}

constexpr int kBulkSmemBytes =
    kStages * kStageBytes + kStages * static_cast<int>(sizeof(UnitMeta)) +
    2 * kStages * 8 + kRing * 8 + kRing * 4;

// ---------------------------------------------------------------------------
// Generic kernel: direct 8-byte loads, any geometry the ABI accepts
// ---------------------------------------------------------------------------
//
// Used when a cache is not 16-byte aligned, has per-head bytes that are not
// a multiple of 16, or rows larger than a stage.  One CTA per position
// (grid-stride), each thread striding over the block's valid pieces in
// logical order (slot, head, piece) and weighting each piece directly.
__global__ void __launch_bounds__(kGenericThreads)
    kvcs_generic_kernel(const __grid_constant__ Params p) {
  __shared__ u64 red[kGenericThreads / 32];
  const int tid = threadIdx.x;
  const long long bs = p.block_size;
  if (blockIdx.x == 0 && tid == 0 && p.num_requests >= 0) {
    if (p.pos_offsets[0] != 0 || p.pos_offsets[p.num_requests] != p.total_positions)
      set_status(p, kStatusBadRequests);
  }
  for (long long pos = blockIdx.x; pos < p.total_positions; pos += gridDim.x) {
    // every thread derives the same position info (uniform loads)
    long long r = find_request(p, pos);
    long long q = 0, b = 0, nv = 0;
    bool ok = r >= 0;
    if (ok) {
      q = p.first_position[r] + (pos - p.pos_offsets[r]);
      b = p.block_ids[pos];
      const long long nt = p.num_tokens[r];
      if (p.first_position[r] < 0) ok = false;
      if (q <= nt / bs) nv = min(nt - q * bs, bs);
    }
    if (tid == 0) {
      if (r < 0 || (ok == false)) set_status(p, kStatusBadRequests);
      else if (b < 0 || b >= p.min_num_blocks) set_status(p, kStatusBadBlockId);
    }
    if (ok && (b < 0 || b >= p.min_num_blocks)) ok = false;
    u64 acc = 0;
    if (ok && nv > 0) {
      const u64 t0 = static_cast<u64>(q) * static_cast<u64>(bs);
      for (int ci = 0; ci < p.num_caches; ++ci) {
        const DevCache &C = p.caches[ci];
        const long long P = C.P;
        const long long per_slot = static_cast<long long>(C.heads) * P;
        const long long n = nv * per_slot;
        const int hp = C.hb >> 3;  // pieces per half
        for (long long idx = tid; idx < n; idx += kGenericThreads) {
          const long long slot = idx / per_slot;
          const long long rem = idx - slot * per_slot;
          const long long h = rem / P;
          const long long pc = rem - h * P;
          u64 off;
          if (C.layout == kLayoutLatent) {
            off = (static_cast<u64>(b) * bs + slot) * C.hb + 8 * pc;
          } else {
            const long long half = pc >= hp ? 1 : 0;
            const long long e = (pc - half * hp) * 8;
            const u64 page = static_cast<u64>(half) * C.half_stride +
                             static_cast<u64>(b) * C.page_bytes;
            if (C.layout == kLayoutNHD)
              off = page + (static_cast<u64>(slot) * C.heads + h) * C.hb + e;
            else
              off = page + (static_cast<u64>(h) * bs + slot) * C.hb + e;
          }
          const u64 x = __ldg(reinterpret_cast<const u64 *>(C.base + off));
          const u64 j = (t0 + static_cast<u64>(slot)) * static_cast<u64>(P) +
                        static_cast<u64>(pc);
          const u64 mh = C.m0 + 2ull * static_cast<u64>(h);
          acc += x * ((2ull * j + 1ull) * mh);
        }
      }
    }
    acc = warp_sum(acc);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      u64 total = 0;
      for (int w = 0; w < kGenericThreads / 32; ++w) total += red[w];
      if (p.all_atomic) atomicAdd(p.out + pos, total);
      else p.out[pos] = total;
    }
    __syncthreads();
  }
}

}  // namespace kvcs
