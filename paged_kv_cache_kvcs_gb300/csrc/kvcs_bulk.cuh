// kvcs_bulk.cuh -- the bulk-copy pipeline kernel (staging through shared
// memory with bulk copies) and its consumer-side reductions.
#pragma once

#include "kvcs_common.cuh"

namespace kvcs {

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
// (kHalves: each 16-byte column read as two 8-byte loads, for stages whose
// columns sit 8 bytes past a 16-byte boundary)
template <bool kHalves = false>
__device__ __forceinline__ uint4 col16(const unsigned char *p) {
  if constexpr (kHalves) {
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    const uint2 b = *reinterpret_cast<const uint2 *>(p + 8);
    return make_uint4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const uint4 *>(p);
  }
}

template <bool kHalves = false>
__device__ __forceinline__ void accum_slots(const unsigned char *p0, size_t stride,
                                            int s_lo, int s_hi, int s_off, u64 &S,
                                            u64 &T, u64 &U) {
  int s = s_lo;
  for (; s + 7 < s_hi; s += 8) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = col16<kHalves>(p0 + static_cast<size_t>(s + k - s_off) * stride);
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
    const uint4 v = col16<kHalves>(p0 + static_cast<size_t>(s - s_off) * stride);
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
template <bool kHalves = false>
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
      v[i] = col16<kHalves>(gp + static_cast<size_t>(sl[i]) * 16);
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
    const uint4 v = col16<kHalves>(gp + static_cast<size_t>(sl) * 16);
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

// One 16-byte column of a staged row: a 16-byte shared load, or, for
// misaligned-rows pages (whose rows may start 8 bytes past a 16-byte
// boundary in the stage), two 8-byte loads.
template <int kFam>
__device__ __forceinline__ uint4 stage_col(const unsigned char *p) {
  if constexpr (kFam == kFamRowsMis) {
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    const uint2 b = *reinterpret_cast<const uint2 *>(p + 8);
    return make_uint4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const uint4 *>(p);
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
  } else if constexpr (kFam == kFamRows || kFam == kFamRowsMis) {
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
        for (int k = 0; k < 8; ++k) v[k] = stage_col<kFam>(sp + k * step);
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
        const uint4 v = stage_col<kFam>(sp);
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
      if constexpr (kFam == kFamXSplit || kFam == kFamXSplitMis) {
        // the group's slots are one contiguous run of 16-byte rows; start
        // at a group-dependent slot so a warp's reads spread over the banks
        // (misaligned pages: the stage's copy may sit 8 bytes past a
        // 16-byte boundary, read as 8-byte halves)
        const unsigned char *gp = stage + static_cast<size_t>(g) * bsi * 16;
        accum_slots_rotated<kFam == kFamXSplitMis>(gp, g % nv, nv, S, T, U);
      } else if constexpr (kFam == kFamHnd) {
        // heads staged one after another, nv slots each
        accum_slots(stage + static_cast<size_t>(hl) * nv * C.hb + (col << 4),
                    static_cast<size_t>(C.hb), 0, nv, 0, S, T, U);
      } else if constexpr (kFam == kFamHndMis) {
        // heads staged as they lie in the page (all block_size slots), the
        // stage's copy possibly 8 bytes past a 16-byte boundary
        accum_slots<true>(stage + static_cast<size_t>(hl) * bsi * C.hb + (col << 4),
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

// This thread's share of a packed unit of several pages (launches whose
// pages all look alike: same layout, heads and head bytes, one page per
// (cache, half) from the unit's first on), for the rows family.  What the
// pages share is worked out once: the thread's 16-byte columns, their head
// and piece, and the piece weight B of each half.  Per page only the cache's m0 and the
// half change, so a page costs the running sums of its few valid rows and
// one fold, m (B S + 2P T + 2U).  The sum is the one unit_sum gives page by
// page, in another order.
template <int kFam>
__device__ __forceinline__ u64 packed_sum(const Params &p, const UnitMeta &m, int first,
                                          const unsigned char *stage, int gtid, int nt,
                                          u64 bsz) {
  const DevCache &C0 = p.caches[m.cache];
  const u64 P = static_cast<u64>(C0.P);
  const u64 twoP = 2ull * P;
  const u64 t0P = static_cast<u64>(m.q) * bsz * P;
  const u64 hstep = 2ull * static_cast<u64>(C0.hb >> 3);  // B of the V half - B of the K half
  const int H = C0.halves;
  const int npg = m.npages;
  u64 acc = 0;
  static_assert(kFam == kFamRows, "packed units of several pages: rows");
  {
    const int rowb = C0.rowb;
    const int cols = rowb >> 4;
    const int nrows = m.count;
    const u32 r0 = static_cast<u32>(first);
    const size_t pstride = static_cast<size_t>(nrows) * rowb;
    int col0, cstep, rl, rstep;
    if (cols <= nt) {
      rstep = nt / cols;
      rl = gtid / cols;
      col0 = gtid - rl * cols;
      cstep = cols;
      if (rl >= rstep) col0 = cols;
    } else {
      rstep = 1;
      rl = 0;
      col0 = gtid;
      cstep = nt;
    }
    const size_t step = static_cast<size_t>(rstep) * rowb;
    for (int col = col0; col < cols; col += cstep) {
      int h_col, p_col;
      if (C0.layout == kLayoutNHD) {
        const int cb = col << 4;
        h_col = C0.hb_shift >= 0 ? (cb >> C0.hb_shift) : cb / C0.hb;
        p_col = (cb - h_col * C0.hb) >> 3;
      } else {
        h_col = 0;
        p_col = col << 1;
      }
      const u64 mh_off = 2ull * static_cast<u64>(h_col);
      const u64 B0 = 2ull * (t0P + static_cast<u64>(p_col)) + 1ull;
      const unsigned char *sp0 = stage + static_cast<size_t>(rl) * rowb + (col << 4);
      int ci = m.cache, half = m.half;
      // pages are independent: let the compiler overlap several
#pragma unroll 4
      for (int k = 0; k < npg; ++k) {
        u64 S = 0, T = 0, U = 0;
        const unsigned char *sp = sp0 + static_cast<size_t>(k) * pstride;
        for (int r = rl; r < nrows; r += rstep, sp += step) {
          const uint4 v = *reinterpret_cast<const uint4 *>(sp);
          const u64 x0 = (static_cast<u64>(v.y) << 32) | v.x;
          const u64 x1 = (static_cast<u64>(v.w) << 32) | v.z;
          const u64 X = x0 + x1;
          S += X;
          U += x1;
          T += static_cast<u64>(r0 + static_cast<u32>(r)) * X;
        }
        const u64 B = half ? B0 + hstep : B0;
        acc += (p.caches[ci].m0 + mh_off) * (B * S + twoP * T + 2ull * U);
        if (++half == H) {
          half = 0;
          ++ci;
        }
      }
    }
  }
  return acc;
}

// Pages of one position a stage holds in packed launches (every page alike,
// each a unit): the host's count for full pages; for a partial block of the
// row and HND families, as many pages as their valid bytes allow; a skipped
// position is passed over at once.
template <int kFam>
__device__ __forceinline__ int stage_fit(const Params &p, const PosInfo &cur, int stage_bytes) {
  if (!p.pack) return 1;
  if (cur.skip) return 1 << 30;
  if (cur.nv == p.block_size || (kFam != kFamRows && kFam != kFamHnd && kFam != kFamRowsMis))
    return p.full_pages;
  const DevCache &C = p.caches[0];
  const u32 bytes = kFam == kFamRows ? static_cast<u32>(cur.nv) * static_cast<u32>(C.rowb)
                    : kFam == kFamRowsMis
                        ? static_cast<u32>(cur.nv) * static_cast<u32>(C.rowb) + kMisPad
                        : static_cast<u32>(C.heads) * static_cast<u32>(cur.nv) *
                              static_cast<u32>(C.hb);
  return max(1, static_cast<int>(static_cast<u32>(stage_bytes) / bytes));
}

// Write a finished (position, column) checksum: a plain store when this CTA
// holds every unit of the position, else a 64-bit atomic add into the
// pre-zeroed output.
__device__ __forceinline__ void finalize_slot(const Params &p, SmemHeader *hdr,
                                              int slot, long long dst, int mode) {
  __threadfence_block();
  const u64 total = atomicAdd(&hdr->ring_acc[slot], 0ull);
  ptx::grid_dep_wait();   // the output is zeroed by the kernel before this one
  if (mode == kFlushStore) p.out[dst] = total;
  else atomicAdd(p.out + dst, total);
}

// ---------------------------------------------------------------------------
// The bulk-copy pipeline kernel
// ---------------------------------------------------------------------------
//
// Persistent: CTA g owns a contiguous range of work units.  A unit is a run
// of whole rows of one page (one block's K, its V, its latent rows or its
// state rows), or of whole heads for HND and x-split, of at most about
// 48 KiB; when every page of the launch fits a unit and all look alike,
// consecutive pages of a position are packed into one unit.  The stage size
// is the launch's largest unit, and as many stages as fit in shared memory
// form a ring.  When the positions balance over the CTAs the ranges are
// whole positions and every result is stored once, without atomics;
// otherwise the ranges are cut at unit granularity and positions shared by
// two CTAs are combined with 64-bit atomics into the pre-zeroed output.
//
// Warp 0, lane 0 is the producer: it walks the range, turns (position,
// cache, half) into page addresses through the block table and issues one
// bulk copy per page of the unit (one per sub-block for a partial-head run
// of an HND page in kernel sub-blocks) into the next stage, signalling the
// stage's "full" mbarrier by transaction bytes.  The
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
// kFam is the layout family of every cache in the launch.  kWide (rows
// family, for calls whose blocks are mostly partial, such as the newest
// block of each request) keeps the whole producer warp in the loop:
// every lane computes the same cursor, lane 0 alone waits, writes metadata
// and counters, and the lanes share out the copies of a unit's pages; the
// consumers then reduce packed units of several pages with packed_sum.
// The wide instance runs two CTAs a SM (each with half the shared memory).
template <int kFam, bool kWide>
__global__ void __launch_bounds__(kBulkThreads, kWide ? 2 : 1)
    kvcs_bulk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  SmemHeader *hdr = reinterpret_cast<SmemHeader *>(smem);
  unsigned char *stages = smem + kHeaderBytes + (kWide ? kWideTableBytes : 0);
  WideTable *wt = reinterpret_cast<WideTable *>(smem + kHeaderBytes);
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
  if constexpr (kWide) {
    for (int i = tid; i < p.num_caches; i += kBulkThreads)
      wt->page[i] = PageAddr{p.caches[i].base, p.caches[i].half_stride,
                             p.caches[i].block_stride};
  }
  __syncthreads();

  // This CTA's unit range: its fixed share.  With a work counter the units
  // past pool_start are not shared out here: CTAs take them in chunks from
  // the counter once their share is done.
  long long u_begin, u_end;
  const long long G = gridDim.x, g = blockIdx.x;
  if (p.work) {
    u_begin = p.pool_start * g / G;
    u_end = p.pool_start * (g + 1) / G;
  } else if (p.split) {
    u_begin = p.total_units * g / G;
    u_end = p.total_units * (g + 1) / G;
  } else {
    u_begin = p.total_positions * g / G * p.units_per_pos;
    u_end = p.total_positions * (g + 1) / G * p.units_per_pos;
  }

  if (tid < 32) {
    // ------------------------------ producer ------------------------------
    // The whole warp looks up the request of the range's first position (one
    // round of loads for up to 31 requests), with that position's block ids
    // loaded alongside; lane 0 then runs the producer alone (kWide: the
    // warp runs it, lane 0 leading).
    ReqCursor rc;
    rc.r = -1;
    long long b_cur = 0, b_next = 0;
    if (u_begin < u_end) {
      const long long pos0 = u_begin / p.units_per_pos;
      if (kWide || tid == 0) {
        b_cur = p.block_ids[pos0];
        b_next = pos0 + 1 < p.total_positions ? p.block_ids[pos0 + 1] : 0;
      }
      rc = req_find_warp(p, pos0, tid);
    }
    if (!kWide && tid != 0) return;
    const bool lead = !kWide || tid == 0;
    if (lead && g == 0 && p.num_requests >= 0) {
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
    // Ranges of units: this CTA's fixed share, then, with a work counter,
    // chunks taken from it until the pool is used up.  After the first
    // chunk the next one is claimed a range ahead, so the atomic's latency
    // overlaps the work.
    long long ra = u_begin, rb = u_end;
    unsigned long long next_chunk = 0ull;
    bool first_range = true, claimed = false;
    while (true) {
      if (ra < rb) {
        if (!first_range) {
          // a chunk starts anywhere in the pool: find its request and
          // block ids afresh (positions still only grow)
          const long long pos0 = ra / p.units_per_pos;
          req_seek(p, rc, pos0);
          b_cur = p.block_ids[pos0];
          b_next = pos0 + 1 < p.total_positions ? p.block_ids[pos0 + 1] : 0;
        }
        long long pos = ra / U;
        int ci = 0, half = 0, sub = 0;
        {
          int kk = static_cast<int>(ra - pos * U);
          if (p.pack) {
            // every cache has the same halves, one unit per page
            ci = kk / p.caches[0].halves;
            half = kk - ci * p.caches[0].halves;
          } else {
            while (kk >= p.caches[ci].halves * p.caches[ci].upp) {
              kk -= p.caches[ci].halves * p.caches[ci].upp;
              ++ci;
            }
            half = kk / p.caches[ci].upp;
            sub = kk - half * p.caches[ci].upp;
          }
        }
        PosInfo cur = position_info(p, pos, rc, b_cur, ra, rb);
        int mode = (cur.whole && !p.all_atomic) ? kFlushStore : kFlushAtomic;
        int fit = stage_fit<kFam>(p, cur, SB);
        int slot = 0;
        u32 n_emit = 0;
        int col = p.caches[ci].column;
        for (long long u = ra; u < rb;) {
          const DevCache &C = p.caches[ci];
          // One accumulator slot per (position, column); the caches arrive
          // sorted by column, so a column's units are consecutive.
          const long long dst_word = pos * p.num_columns + col;
          const int first = sub * C.rpu;
          int count = 0;
          u32 pbytes = 0;   // bytes copied per page of the unit
          u32 pstride = 0;  // bytes a page of the unit occupies in the stage
          if (!cur.skip) {
            if constexpr (head_family(kFam)) {
              count = max(0, min(C.rpu, C.heads - first));
              if constexpr (kFam == kFamHnd) {
                // each head's first nv slots (its valid ones), heads packed
                // one after another in the stage
                pstride = static_cast<u32>(count) * static_cast<u32>(cur.nv) *
                          static_cast<u32>(C.hb);
                pbytes = pstride;
              } else {
                // the unit's heads with all their slots, staged as in memory
                pstride = static_cast<u32>(count) * static_cast<u32>(bs) * static_cast<u32>(C.hb);
                pbytes = pstride;
                // (misaligned: in a 16-byte-aligned region with room for the shift)
                if constexpr (mis_family(kFam)) pstride = pbytes + kMisPad;
                if constexpr (kFam == kFamHndSub) {
                  const int nsb = (cur.nv + C.kbs - 1) / C.kbs;  // sub-blocks with valid slots
                  pbytes = static_cast<u32>(count) * static_cast<u32>(nsb * C.kbs) *
                           static_cast<u32>(C.hb);
                }
              }
            } else if constexpr (kFam == kFamState) {
              count = max(0, min(C.rpu, C.heads - first));
              pbytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
              pstride = pbytes;
            } else if constexpr (kFam == kFamRowsMis) {
              // the rows, in a 16-byte-aligned region with room for the shift;
              // pbytes counts the bytes the bulk copies bring (the two edge
              // words of a misaligned page come by cp.async)
              count = max(0, min(C.rpu, cur.nv - first));
              pbytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
              pstride = pbytes + kMisPad;
            } else {
              count = max(0, min(C.rpu, cur.nv - first));
              pbytes = static_cast<u32>(count) * static_cast<u32>(C.rowb);
              pstride = pbytes;
            }
          }
          // Pages per unit: one, or, when the launch's pages all look alike and
          // each is a unit, as many consecutive pages of the position (in this
          // CTA's range) as the stage holds -- many more when blocks are
          // partial.  A skipped position is passed over in one step.
          int npg = 1;
          // (the two forms of the test and of the cursor step below measured
          // fastest for their families: rows a packed step per unit, heads the
          // one-page step whenever a unit holds one page)
          if (kFam == kFamRows ? p.pack != 0 : fit > 1) {
            int left = p.pages_per_pos - (ci * C.halves + half);
            if (rb - u < left) left = static_cast<int>(rb - u);
            npg = max(1, min(left, fit));
            if constexpr (mis_family(kFam)) npg = min(npg, kMisMaxPages);
          }
          if (pbytes > 0) {
            bool free_stage = true;
            if (lead)
              free_stage = ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->empty[s]),
                                                  (f & 1u) ^ 1u, p.timeout_ns);
            if constexpr (kWide) free_stage = __shfl_sync(0xffffffffu, free_stage, 0);
            if (!free_stage) {
              if (lead) set_status(p, kStatusTimeout);
              aborted = true;
              break;
            }
            if (n_emit == 0) {
              slot = static_cast<int>(seq % kRingSlots);
              ++seq;
              if (lead) {
                hdr->ring_acc[slot] = 0ull;
                hdr->ring_cnt[slot] = 0u;
              }
            }
            const u32 fb = ptx::smem_addr(&hdr->full[s]);
            if constexpr (mis_family(kFam)) {
              static_assert(!kWide, "the misaligned instances have one producer lane");
              // Per page: the 16-byte-aligned interior of its unit's bytes (rows,
              // or heads with all their slots) by bulk copy, and when they start
              // 8 bytes past a boundary their first and last words by 8-byte
              // cp.async, tracked on the same barrier.
              u32 dst = ptx::smem_addr(stages + static_cast<size_t>(s) * SB);
              u32 tx = 0, dmask = 0;
              int pci = ci, phalf = half;
              for (int k2 = 0; k2 < npg; ++k2) {
                const DevCache &D = p.caches[pci];
                const unsigned char *src =
                    D.base + static_cast<long long>(phalf) * D.half_stride +
                    cur.block * D.block_stride +
                    (head_family(kFam) ? static_cast<u64>(first) * bs * D.hb
                                       : static_cast<u64>(first) * D.rowb);
                if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
                  ptx::bulk_g2s(dst, src, pbytes, fb, policy);
                  tx += pbytes;
                } else {
                  dmask |= 1u << k2;
                  if (pbytes > 16) {
                    ptx::bulk_g2s(dst + 16, src + 8, pbytes - 16, fb, policy);
                    tx += pbytes - 16;
                  }
                  ptx::cp_async8(dst + 8, src);
                  ptx::cp_async8(dst + pbytes, src + pbytes - 8);
                }
                dst += pstride;
                if (++phalf == D.halves) {
                  phalf = 0;
                  ++pci;
                }
              }
              store_meta(&hdr->meta[s], dst_word, cur.q, ci, half, first, count, cur.nv,
                         mode | static_cast<int>(dmask << 1), slot, npg);
              if (dmask) ptx::cp_async_mbar_arrive(fb);
              ptx::mbar_arrive_expect_tx(fb, tx);
            } else {
            if (lead) {
              store_meta(&hdr->meta[s], dst_word, cur.q, ci, half, first, count, cur.nv,
                         mode, slot, npg);
              ptx::mbar_arrive_expect_tx(fb, pbytes * static_cast<u32>(npg));
            }
            if constexpr (kWide) {
              static_assert(kFam == kFamRows, "the wide producer stages rows");
              // the lanes share the unit's copies: page k2 by lane k2 mod 32,
              // once lane 0 has set the stage's byte count
              __syncwarp();
              const u32 dst0 = ptx::smem_addr(stages + static_cast<size_t>(s) * SB);
              const int H0 = C.halves;
              for (int k2 = tid; k2 < npg; k2 += 32) {
                int pci = ci, phalf = half;
                if (k2 > 0) {  // packed pages: every cache has H0 halves
                  const int flat = ci * H0 + half + k2;
                  pci = H0 == 1 ? flat : flat >> 1;
                  phalf = flat - pci * H0;
                }
                // (packed pages share their geometry: C's rowb holds for every
                // page; only the addressing differs)
                const PageAddr D = wt->page[pci];
                const unsigned char *page = D.base +
                    static_cast<long long>(phalf) * D.half_stride + cur.block * D.block_stride;
                ptx::bulk_g2s(dst0 + static_cast<u32>(k2) * pstride,
                              page + static_cast<u64>(first) * C.rowb, pbytes, fb, policy);
              }
            } else {
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
              } else if constexpr (kFam == kFamHnd) {
                // [heads][block_size][hb]: a full block's heads are one
                // contiguous run; a partial block's valid slots are one run of
                // nv slots per head, copied one after another
                const unsigned char *src = page + static_cast<u64>(first) * bs * D.hb;
                if (cur.nv == bs) {
                  ptx::bulk_g2s(dst, src, pstride, fb, policy);
                } else {
                  const u32 run = static_cast<u32>(cur.nv) * static_cast<u32>(D.hb);
                  const u64 hstep = static_cast<u64>(bs) * static_cast<u64>(D.hb);
                  for (int h = 0; h < count; ++h)
                    ptx::bulk_g2s(dst + static_cast<u32>(h) * run, src + h * hstep, run, fb,
                                  policy);
                }
              } else if constexpr (head_family(kFam)) {
                // [heads][chunks][block_size][16]: the unit's heads are one
                // contiguous run of whole slots
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
            }
            }
            ++it;
            ++n_emit;
            if (++s == NS) {
              s = 0;
              ++f;
            }
          }
          // advance the cursor past this unit's npg host units
          u += npg;
          bool pos_done = false;
          if (kFam == kFamRows && p.pack) {
            // packed pages: every cache has C.halves halves
            const int flat = ci * C.halves + half + npg;
            ci = flat / C.halves;
            half = flat - ci * C.halves;
            pos_done = ci >= p.num_caches;
          } else if (npg > 1) {
            half += npg;
            while (half >= C.halves) {
              half -= C.halves;
              ++ci;
            }
            pos_done = ci >= p.num_caches;
          } else if (++sub == C.upp) {
            sub = 0;
            if (++half == C.halves) {
              half = 0;
              pos_done = ++ci == p.num_caches;
            }
          }
          if (pos_done) ci = 0;
          if (pos_done || u == rb || p.caches[ci].column != col) {
            // close the (position, column): this thread's share of the count
            if (n_emit > 0) {
              if (lead) {
                const u32 delta = 0u - static_cast<u32>(p.group_warps) * n_emit;
                const u32 prev = atomicAdd(&hdr->ring_cnt[slot], delta);
                if (prev + delta == 0u) finalize_slot(p, hdr, slot, dst_word, mode);
              }
            } else if (cur.whole && !p.all_atomic) {
              if (lead) {
                ptx::grid_dep_wait();
                p.out[dst_word] = 0ull;
              }
            }
            n_emit = 0;
          }
          col = p.caches[ci].column;
          if (pos_done && u < rb) {
            ++pos;
            b_cur = b_next;
            b_next = pos + 1 < p.total_positions ? p.block_ids[pos + 1] : 0;
            req_seek(p, rc, pos);
            cur = position_info(p, pos, rc, b_cur, ra, rb);
            mode = (cur.whole && !p.all_atomic) ? kFlushStore : kFlushAtomic;
            fit = stage_fit<kFam>(p, cur, SB);
          }
        }
        if (aborted) break;
      }
      if (!p.work) break;
      if (!claimed) {
        // the counter is zeroed by the kernel launched before this one
        ptx::grid_dep_wait();
        if (lead) next_chunk = atomicAdd(p.work, 1ull);
        if constexpr (kWide) next_chunk = __shfl_sync(0xffffffffu, next_chunk, 0);
        claimed = true;
      }
      const long long ca = p.pool_start + static_cast<long long>(next_chunk) * p.chunk_units;
      if (ca >= p.total_units) break;
      ra = ca;
      rb = min(p.total_units, ca + p.chunk_units);
      if (lead) next_chunk = atomicAdd(p.work, 1ull);
      if constexpr (kWide) next_chunk = __shfl_sync(0xffffffffu, next_chunk, 0);
      first_range = false;
    }
    // Every copy of this CTA is issued: a following kernel launched with
    // programmatic stream serialization may start (it waits for this grid
    // before it touches anything this grid writes).
    ptx::grid_dep_launch();
    if (!lead) return;
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
    bool ok = f == 0 || ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->empty[s]),
                                               (f - 1u) & 1u, p.timeout_ns);
    ok = ok && ptx::mbar_wait_bounded(ptx::smem_addr(&hdr->full[s]), f & 1u, p.timeout_ns);
    // Each lane waits on its own, so near the time limit lanes can disagree;
    // the warp leaves as a whole if any lane gave up, so no lane reaches the
    // full-mask shuffles below with others of its warp gone.
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) set_status(p, kStatusTimeout);
      return;
    }
    const UnitMeta m = hdr->meta[s];
    if (m.dst < 0) break;
    const unsigned char *sp = stages + static_cast<size_t>(s) * SB;
    int ci = m.cache, half = m.half;
    u64 v = 0;
    bool packed = false;
    if constexpr (kWide) {
      if (m.npages > 1) {
        v = packed_sum<kFam>(p, m, m.first, sp, gtid, gw * 32, bsz);
        packed = true;
      }
    }
    for (int k = 0; !packed && k < m.npages; ++k) {
      const DevCache &C = p.caches[ci];
      if (C.rowb != map.rowb) make_map(map, C.rowb, gtid, gw * 32);
      if constexpr (mis_family(kFam)) {
        // the page's first byte sits 8 bytes into its region when the page
        // starts 8 bytes past a boundary
        v += unit_sum<kFam>(C, m, half, sp + ((m.mode >> (1 + k)) & 1) * 8, map, bsz);
        sp += (head_family(kFam) ? static_cast<size_t>(m.count) * bsz * C.hb
                                 : static_cast<size_t>(m.count) * C.rowb) + kMisPad;
      } else {
        v += unit_sum<kFam>(C, m, half, sp, map, bsz);
        sp += kFam == kFamHnd ? static_cast<size_t>(m.count) * static_cast<size_t>(m.nv) * C.hb
              : head_family(kFam)
                  ? static_cast<size_t>(m.count) * static_cast<size_t>(bsz) * C.hb
                  : static_cast<size_t>(m.count) * C.rowb;
      }
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
      if (prev + 1u == 0u) finalize_slot(p, hdr, m.slot, m.dst, m.mode & 1);
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

}  // namespace kvcs
