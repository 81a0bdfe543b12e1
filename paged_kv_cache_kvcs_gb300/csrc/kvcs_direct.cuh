// kvcs_direct.cuh -- the direct-load kernel: KV pages the bulk-copy kernel
// cannot stage (pools, strides or rows not 16-byte aligned, per-head bytes
// not a multiple of 16, rows or head runs larger than a stage), read
// straight from global memory with 16-byte loads.
#pragma once

#include "kvcs_common.cuh"

namespace kvcs {

constexpr int kDirectThreads = 256;
constexpr int kDirectBatch = 8;  // independent 16-byte loads per lane in flight

__device__ __forceinline__ uint4 ld_stream16(const unsigned char *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ u64 ld_stream8(const unsigned char *p) {
  u64 v;
  asm volatile("ld.global.nc.L1::no_allocate.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// What a run's rows are: a run is nrows consecutive rows of rowb bytes
// (rowb a multiple of 8) starting at an 8-byte-aligned address; in-row word
// w (8 bytes) of row r is piece piece0 + (w mod hw) of head w / hw (or
// piece piece0 + w of head `head`, when the run has one head), of the token
// in slot slot0 + r.
struct RunShape {
  int rowb;
  int hw;      // words per head (hb / 8), for runs holding several heads
  int head;    // the run's one head, or -1: head = w / hw
  int piece0;
  int slot0;
};

// This lane's share of one run's contribution to the block checksum,
// 2 * ((t0 + slot) * P + p) + 1 weighting each piece, m0 + 2 head each head.
//
// The lane walks 16-byte chunks at addresses that are multiples of 16.  When
// the run starts 8 bytes past such an address, a chunk holds the last word
// of one 16-byte column and the first of the next; the chunk's two words
// are then handled as two separate columns.  Rows of rowb = 8 mod 16 bytes
// repeat their chunk pattern every two rows, so rows are taken in groups
// ("super-rows") of pr = 1 or 2 rows, of cps chunks each.  The lane owns
// fixed chunk positions c within a super-row, so each of its two words has
// a fixed (row within the super-row, head, piece), and only the super-row
// index s changes from one chunk to the next: running sums S = sum x and
// T = sum s x give the weighted sum with one multiply per column,
//   sum x (B + 2 P pr s) = B S + 2 P pr T,   B = 2 ((t0 + slot0 + rin) P + p) + 1.
// Words outside [0, nrows * rowb) are never read.  Of a lane's chunks, those
// holding two words of the run are read in batches of eight 16-byte loads
// (the last batch predicated); a column's at most one chunk before them
// (the run's first word, when misaligned) and at most one after them (the
// run's last word) are read as single 8-byte words.
__device__ __forceinline__ u64 run_sum(const unsigned char *base, int nrows, const RunShape &R,
                                       u64 m0, u64 t0, u64 P, int lane) {
  if (nrows <= 0) return 0;
  const int d = static_cast<int>(reinterpret_cast<uintptr_t>(base) & 15u);  // 0 or 8
  const unsigned char *A = base - d;     // 16-byte aligned; never read below base
  const int pr = (R.rowb & 15) ? 2 : 1;
  const int srb = pr * R.rowb;           // bytes per super-row, a multiple of 16
  const int cps = srb >> 4;              // chunks per super-row
  const long long len = static_cast<long long>(nrows) * R.rowb;
  // super-rows whose chunks touch the run: one more when misaligned (the
  // last word sits in the first chunk of the next super-row)
  const int nsr = (nrows + pr - 1) / pr + (d ? 1 : 0);
  int c0, cstep, sr0, rstep;
  if (cps <= 32) {
    rstep = 32 / cps;
    sr0 = lane / cps;
    c0 = lane - sr0 * cps;
    cstep = cps;
    if (sr0 >= rstep) c0 = cps;          // idle lane
  } else {
    rstep = 1;
    sr0 = 0;
    c0 = lane;
    cstep = 32;
  }
  const long long lstep = static_cast<long long>(rstep) * srb;  // bytes between a lane's chunks
  u64 acc = 0;
  for (int c = c0; c < cps; c += cstep) {
    // chunks s < s_full hold two words of the run: 16 (s cps + c) - d + 8 < len
    const long long room = len + d - 8 - 16LL * c;
    long long s_full_l = room > 0 ? (room + srb - 1) / srb : 0;
    if (s_full_l > nsr) s_full_l = nsr;
    const int s_full = static_cast<int>(s_full_l);
    // The edge words are loaded first and added after the batches, so their
    // latency overlaps the batches': the run's first word (the upper half of
    // the chunk before the run, when misaligned), and the one chunk past
    // s_full whose first word still lies in the run.
    int s = sr0;
    u64 xh = 0, xt = 0;
    if (d && c == 0 && s == 0) {
      xh = ld_stream8(base);
      s += rstep;
    }
    const long long ot = static_cast<long long>(s_full) * srb + 16LL * c - d;
    const bool tail = s_full < nsr && ot >= 0 && ot < len && s_full >= sr0 &&
                      (s_full - sr0) % rstep == 0;
    if (tail) xt = ld_stream8(A + static_cast<long long>(s_full) * srb + 16LL * c);
    u64 S0 = 0, T0 = 0, S1 = 0, T1 = 0;   // T: sum of (chunk's super-row) x
    const unsigned char *cp = A + (static_cast<long long>(s) * cps + c) * 16;
    for (; s < s_full; s += kDirectBatch * rstep) {
      uint4 v[kDirectBatch];
#pragma unroll
      for (int k = 0; k < kDirectBatch; ++k) {
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (s + k * rstep < s_full) v[k] = ld_stream16(cp + k * lstep);
      }
      cp += kDirectBatch * lstep;
#pragma unroll
      for (int k = 0; k < kDirectBatch; ++k) {
        // a chunk not loaded is 0 and adds nothing
        const u64 sk = static_cast<u64>(static_cast<u32>(s + k * rstep));
        const u64 x0 = (static_cast<u64>(v[k].y) << 32) | v[k].x;
        const u64 x1 = (static_cast<u64>(v[k].w) << 32) | v[k].z;
        S0 += x0;
        T0 += sk * x0;
        S1 += x1;
        T1 += sk * x1;
      }
    }
    // the chunk's two words: offsets u within a super-row; word 0 belongs
    // to the previous super-row (srd = 1) when the chunk starts before it
    int rin[2], hd[2], pc[2], srd[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      int u = 16 * c - d + 8 * j;
      srd[j] = 0;
      if (u < 0) {
        u += srb;
        srd[j] = 1;
      }
      rin[j] = u / R.rowb;
      const int w = (u - rin[j] * R.rowb) >> 3;
      if (R.head >= 0) {
        hd[j] = R.head;
        pc[j] = R.piece0 + w;
      } else {
        hd[j] = w / R.hw;
        pc[j] = R.piece0 + (w - hd[j] * R.hw);
      }
    }
    S1 += xh;                       // super-row 0
    S0 += xt;
    T0 += static_cast<u64>(static_cast<u32>(s_full)) * xt;
    // word j's super-row is the chunk's minus srd[j]
    T0 -= static_cast<u64>(srd[0]) * S0;
    T1 -= static_cast<u64>(srd[1]) * S1;
    const u64 twoPpr = 2ull * P * static_cast<u64>(pr);
    const u64 B0 = 2ull * ((t0 + static_cast<u64>(R.slot0 + rin[0])) * P +
                           static_cast<u64>(pc[0])) + 1ull;
    const u64 B1 = 2ull * ((t0 + static_cast<u64>(R.slot0 + rin[1])) * P +
                           static_cast<u64>(pc[1])) + 1ull;
    acc += (m0 + 2ull * static_cast<u64>(hd[0])) * (B0 * S0 + twoPpr * T0);
    acc += (m0 + 2ull * static_cast<u64>(hd[1])) * (B1 * S1 + twoPpr * T1);
  }
  return acc;
}

// A lane's part in every run of one shape (rows of rowb <= 512 bytes, nrows
// rows, starting d = 0 or 8 bytes past a 16-byte boundary), worked out once
// for the runs of a page that share it: HND heads (or sub-blocks of heads)
// and x-split chunks.  It is run_sum's mapping with everything that depends
// only on the shape taken out of the run: the lane's chunk column, its
// super-rows, the edge words, and for its two words the row within a
// super-row, the word within the row and the super-row shift.
struct RunPlan {
  int rowb, nrows, d;   // the shape (rowb = -1: none yet)
  int active;           // the lane holds a column
  int pr;               // rows per super-row
  int s0, s_full;       // the lane's batched super-rows: s0, s0 + rstep, ... < s_full
  int rstep;
  int lstep;            // bytes between the lane's chunks
  int first_off;        // its first batched chunk, from the aligned base
  int head_word;        // 1: its chunk's second word is the run's first word (read alone)
  int tail;             // 1: one more chunk past s_full whose first word is in the run
  int tail_off, tail_s; // that chunk's offset from the aligned base, and its super-row
  int rin0, rin1;       // row within the super-row of word 0 and word 1
  int w0, w1;           // word within the row
  int srd0, srd1;       // word j belongs to the previous super-row
};

__device__ __forceinline__ void plan_runs(RunPlan &pl, int rowb, int nrows, int d, int lane) {
  pl.rowb = rowb;
  pl.nrows = nrows;
  pl.d = d;
  pl.pr = (rowb & 15) ? 2 : 1;
  const int srb = pl.pr * rowb;
  const int cps = srb >> 4;                       // <= 32 here
  const int len = nrows * rowb;
  const int nsr = (nrows + pl.pr - 1) / pl.pr + (d ? 1 : 0);
  pl.rstep = 32 / cps;
  const int sr0 = lane / cps;
  const int c = lane - sr0 * cps;
  pl.active = sr0 < pl.rstep && nrows > 0;
  pl.lstep = pl.rstep * srb;
  const int room = len + d - 8 - 16 * c;
  int s_full = room > 0 ? (room + srb - 1) / srb : 0;
  if (s_full > nsr) s_full = nsr;
  pl.s_full = s_full;
  int s = sr0;
  pl.head_word = d && c == 0 && s == 0;
  if (pl.head_word) s += pl.rstep;
  pl.s0 = s;
  pl.first_off = (s * cps + c) * 16;
  const int ot = s_full * srb + 16 * c - d;
  pl.tail = s_full < nsr && ot >= 0 && ot < len && s_full >= sr0 && (s_full - sr0) % pl.rstep == 0;
  pl.tail_off = s_full * srb + 16 * c;
  pl.tail_s = s_full;
  int rin[2], w[2], srd[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    int u = 16 * c - d + 8 * j;
    srd[j] = 0;
    if (u < 0) {
      u += srb;
      srd[j] = 1;
    }
    rin[j] = u / rowb;
    w[j] = (u - rin[j] * rowb) >> 3;
  }
  pl.rin0 = rin[0];
  pl.rin1 = rin[1];
  pl.w0 = w[0];
  pl.w1 = w[1];
  pl.srd0 = srd[0];
  pl.srd1 = srd[1];
}

// This lane's share of one run of the planned shape whose words are pieces
// piece0 + (word in the row) of one head, weighted m = m0 + 2 head, the
// run's row r holding the token in slot slot0 + r: run_sum's result.
template <int kB = kDirectBatch>
__device__ __forceinline__ u64 run_sum_planned(const unsigned char *base, const RunPlan &pl,
                                               u64 m, u64 t0, u64 P, int slot0, int piece0) {
  if (!pl.active) return 0;
  const unsigned char *A = base - pl.d;
  u64 xh = 0, xt = 0;
  if (pl.head_word) xh = ld_stream8(base);
  if (pl.tail) xt = ld_stream8(A + pl.tail_off);
  u64 S0 = 0, T0 = 0, S1 = 0, T1 = 0;
  const unsigned char *cp = A + pl.first_off;
  for (int s = pl.s0; s < pl.s_full; s += kB * pl.rstep) {
    uint4 v[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (s + k * pl.rstep < pl.s_full) v[k] = ld_stream16(cp + k * pl.lstep);
    }
    cp += kB * pl.lstep;
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const u64 sk = static_cast<u64>(static_cast<u32>(s + k * pl.rstep));
      const u64 x0 = (static_cast<u64>(v[k].y) << 32) | v[k].x;
      const u64 x1 = (static_cast<u64>(v[k].w) << 32) | v[k].z;
      S0 += x0;
      T0 += sk * x0;
      S1 += x1;
      T1 += sk * x1;
    }
  }
  S1 += xh;
  S0 += xt;
  T0 += static_cast<u64>(static_cast<u32>(pl.tail_s)) * xt;
  T0 -= static_cast<u64>(pl.srd0) * S0;
  T1 -= static_cast<u64>(pl.srd1) * S1;
  // B_j = 2 ((t0 + slot0 + rin_j) P + piece0 + w_j) + 1 = K + 2 (rin_j P + w_j)
  const u64 K = 2ull * ((t0 + static_cast<u64>(slot0)) * P + static_cast<u64>(piece0)) + 1ull;
  const u64 B0 = K + 2ull * (static_cast<u64>(pl.rin0) * P + static_cast<u64>(pl.w0));
  const u64 B1 = K + 2ull * (static_cast<u64>(pl.rin1) * P + static_cast<u64>(pl.w1));
  return m * (B0 * S0 + B1 * S1 + 2ull * P * static_cast<u64>(pl.pr) * (T0 + T1));
}

// This lane's share of one page (one half of one cache at one position) in
// the page's layout, cut into runs of whole rows:
//   NHD, latent   one run of nv rows of heads * hb (latent: one row) bytes
//   HND           per head one run of nv slots of hb bytes; in kernel
//                 sub-blocks, per (sub-block, head) one run of its valid slots
//   x-split       per (head, 16-byte chunk) one run of nv 16-byte slots
__device__ __forceinline__ u64 page_sum(const DevCache &C, const unsigned char *page, int half,
                                        int nv, u64 t0, long long bs, int lane, RunPlan &pl) {
  const u64 P = static_cast<u64>(C.P);
  const int hw = C.hb >> 3;
  RunShape R;
  R.hw = hw;
  R.slot0 = 0;
  R.piece0 = half * hw;
  u64 acc = 0;
  if (C.layout == kLayoutNHD || C.layout == kLayoutLatent) {
    R.rowb = C.layout == kLayoutNHD ? C.heads * C.hb : C.hb;
    R.head = C.layout == kLayoutNHD ? -1 : 0;
    acc = run_sum(page, nv, R, C.m0, t0, P, lane);
  } else if (C.layout == kLayoutHND) {
    R.rowb = C.hb;
    const int kbs = C.kbs;
    // runs of one shape (rows of at most 512 bytes) share a plan
    const bool planned = (C.hb & 15) == 0 ? C.hb <= 512 : 2 * C.hb <= 512;
    for (int sb = 0; sb * kbs < nv; ++sb) {
      R.slot0 = sb * kbs;
      const int rows = min(kbs, nv - sb * kbs);
      const long long hstride = static_cast<long long>(kbs) * C.hb;
      const unsigned char *sbp = page + static_cast<long long>(sb) * C.heads * hstride;
      if (planned && (hstride & 15) == 0) {
        // every head run of the sub-block has one shape: four runs at a time,
        // two loads each, in flight together
        const int d = static_cast<int>(reinterpret_cast<uintptr_t>(sbp) & 15u);
        if (pl.nrows != rows || pl.d != d || pl.rowb != C.hb) plan_runs(pl, C.hb, rows, d, lane);
        int h = 0;
        for (; h + 3 < C.heads; h += 4) {
          u64 a[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            a[i] = run_sum_planned<2>(sbp + (h + i) * hstride, pl,
                                      C.m0 + 2ull * static_cast<u64>(h + i), t0, P, R.slot0,
                                      R.piece0);
          acc += (a[0] + a[1]) + (a[2] + a[3]);
        }
        for (; h < C.heads; ++h)
          acc += run_sum_planned<4>(sbp + h * hstride, pl, C.m0 + 2ull * static_cast<u64>(h),
                                    t0, P, R.slot0, R.piece0);
        continue;
      }
      for (int h = 0; h < C.heads; ++h) {
        R.head = h;
        const unsigned char *run =
            page + (static_cast<long long>(sb) * C.heads + h) * kbs * C.hb;
        if (planned) {
          const int d = static_cast<int>(reinterpret_cast<uintptr_t>(run) & 15u);
          if (pl.nrows != rows || pl.d != d || pl.rowb != C.hb) plan_runs(pl, C.hb, rows, d, lane);
          acc += run_sum_planned(run, pl, C.m0 + 2ull * static_cast<u64>(h), t0, P, R.slot0,
                                 R.piece0);
        } else {
          acc += run_sum(run, rows, R, C.m0, t0, P, lane);
        }
      }
    }
  } else {  // x-split
    R.rowb = 16;
    const int chunks = C.hb >> 4;
    for (int h = 0; h < C.heads; ++h) {
      R.head = h;
      for (int c = 0; c < chunks; ++c) {
        R.piece0 = half * hw + 2 * c;
        const unsigned char *run = page + (static_cast<long long>(h) * chunks + c) * bs * 16;
        const int d = static_cast<int>(reinterpret_cast<uintptr_t>(run) & 15u);
        if (pl.rowb != 16 || pl.d != d || pl.nrows != nv) plan_runs(pl, 16, nv, d, lane);
        acc += run_sum_planned(run, pl, C.m0 + 2ull * static_cast<u64>(h), t0, P, 0,
                               R.piece0);
      }
    }
  }
  return acc;
}

// A warp's walk over its pages, kept in shared memory rather than registers
// (the registers go to the loads in flight); lane 0 writes it, every lane
// reads it.
struct DirectWalk {
  ReqCursor rc;
  long long pos;   // current position
  long long q;     // its block position
  long long block; // its physical block
  int nv;          // its valid slots
  int skip;        // nothing to read there
  int ci, half;    // the next page: cache and half
};

__device__ __forceinline__ void walk_seek(const Params &p, DirectWalk &w, long long pos,
                                          int lane, bool first) {
  ReqCursor rc = w.rc;
  if (first) rc = req_find_warp(p, pos, lane);
  else req_seek(p, rc, pos);
  const PosInfo pi = position_info_quiet(p, pos, rc, p.block_ids[pos], lane == 0);
  __syncwarp();
  if (lane == 0) {
    w.rc = rc;
    w.pos = pos;
    w.q = pi.q;
    w.block = pi.block;
    w.nv = pi.nv;
    w.skip = pi.skip ? 1 : 0;
  }
  __syncwarp();
}

// Persistent warps: warp w of the grid owns a contiguous range of pages in
// (position, cache, half) order, walks it with its own request cursor and
// adds each (position, column) total into the pre-zeroed output (or the
// caller's words, for accumulating calls) with one 64-bit atomic per warp.
// No CTA-wide barrier: warps never wait for each other.
__global__ void __launch_bounds__(kDirectThreads, 4)
    kvcs_direct_kernel(const __grid_constant__ Params p) {
  __shared__ DirectWalk walks[kDirectThreads / 32];
  // each lane's run plan, kept in shared memory (the registers go to the
  // loads in flight) and reused while the run shape stays the same
  __shared__ RunPlan plans[kDirectThreads];
  RunPlan &pl = plans[threadIdx.x];
  pl.rowb = -1;
  const int lane = threadIdx.x & 31;
  const long long wpc = kDirectThreads / 32;
  const long long warp = static_cast<long long>(blockIdx.x) * wpc + (threadIdx.x >> 5);
  const long long W = static_cast<long long>(gridDim.x) * wpc;
  DirectWalk &wk = walks[threadIdx.x >> 5];
  if (warp == 0 && lane == 0 && p.num_requests >= 0) {
    if (p.pos_offsets[0] != 0 || p.pos_offsets[p.num_requests] != p.total_positions)
      set_status(p, kStatusBadRequests);
  }
  const long long ipp = p.pages_per_pos;            // pages (halves) per position
  const long long items = p.total_positions * ipp;
  const long long i0 = items * warp / W, i1 = items * (warp + 1) / W;
  if (i0 >= i1) return;
  const long long bs = p.block_size;
  {
    const long long pos = i0 / ipp;
    int ci = 0, k = static_cast<int>(i0 - pos * ipp);
    while (k >= p.caches[ci].halves) {
      k -= p.caches[ci].halves;
      ++ci;
    }
    if (lane == 0) {
      wk.rc.r = -1;
      wk.ci = ci;
      wk.half = k;
    }
    __syncwarp();
    walk_seek(p, wk, pos, lane, true);
  }
  u64 acc = 0;
  for (long long it = i0; it < i1; ++it) {
    const int ci = wk.ci, half = wk.half;
    const DevCache &C = p.caches[ci];
    if (!wk.skip) {
      const unsigned char *page = C.base + static_cast<long long>(half) * C.half_stride +
                                  wk.block * C.block_stride;
      acc += page_sum(C, page, half, wk.nv, static_cast<u64>(wk.q) * static_cast<u64>(bs), bs,
                      lane, pl);
    }
    int nci = ci, nhalf = half + 1;
    bool pos_done = false;
    if (nhalf == C.halves) {
      nhalf = 0;
      pos_done = ++nci == p.num_caches;
    }
    if (pos_done) nci = 0;
    const int col = C.column;
    if (pos_done || it + 1 == i1 || p.caches[nci].column != col) {
      const u64 v = warp_sum(acc);
      if (lane == 0 && v != 0) {
        ptx::grid_dep_wait();   // the output is zeroed by the kernel before this one
        atomicAdd(p.out + wk.pos * p.num_columns + col, v);
      }
      acc = 0;
    }
    __syncwarp();
    if (lane == 0) {
      wk.ci = nci;
      wk.half = nhalf;
    }
    __syncwarp();
    if (pos_done && it + 1 < i1) walk_seek(p, wk, wk.pos + 1, lane, false);
  }
}

}  // namespace kvcs
