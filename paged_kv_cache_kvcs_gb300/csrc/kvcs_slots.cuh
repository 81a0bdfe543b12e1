// kvcs_slots.cuh -- the valid-slot kernel: calls whose blocks are mostly
// partial (at most about two positions a request, such as the newest block
// of each request) over latent or HND pages, or NHD pages of at most 8 KiB,
// that are 16-byte aligned and alike (the planner keeps larger NHD pages of
// such calls on the bulk kernel).  A page then holds a few valid slots
// (nv of block_size), a few hundred bytes to a few KiB in one or a few runs,
// and staging it through shared memory costs more instructions than reading
// it: each warp reads its pages' valid bytes straight into registers with
// 16-byte loads, several pages' worth in flight.
#pragma once

#include "kvcs_common.cuh"
#include "kvcs_direct.cuh"

namespace kvcs {

constexpr int kSlotsThreads = 256;
constexpr int kSlotsWarps = kSlotsThreads / 32;
constexpr int kSlotsCtasPerSm = 2;
constexpr int kSlotsCols = 4;      // 16-byte chunks of a page a lane holds per window
constexpr int kSlotsWindow = 32 * kSlotsCols;   // chunks of a page per window
constexpr int kSlotsPages = 2;     // pages a lane loads together
constexpr u32 kSlotsNone = 0xffffffffu;
// Dynamic share-out (calls with a work counter and at least
// kSlotsDynamicPages pages a warp): each warp's fixed share is the first
// 1 / kSlotsFixedShare of the pages; the rest go out in ranges of about the
// remaining pages / (2 warps), at least kSlotsMinRange pages.
constexpr long long kSlotsDynamicPages = 64;
constexpr long long kSlotsFixedShare = 4;
constexpr long long kSlotsMinRange = 16;

// A lane's share of the valid bytes of a page: chunks c = c0 + lane + 32 i
// (i < kSlotsCols) of the page's nv valid slots, 16 bytes each, numbered in
// address order.  For each: its byte offset from the page's start
// (kSlotsNone past the valid bytes), 2 h for its head h, and the part
// 2 (r P + p) + 1 of the weight base B = 2 ((t0 + r) P + p) + 1 of its first
// piece p of slot r in the K half that does not depend on the block's first
// token t0 (the V half's pieces follow the K half's: B + 2 hb / 8).  The
// pieces of a 16-byte chunk, x0 and x1, then add
//   x0 B + x1 (B + 2) = B (x0 + x1) + 2 x1
// to the slice of head h (checksum page, module docstring item 1).  The map
// depends on nv and the window only, so a warp keeps it while they repeat.
struct SlotMap {
  u32 off[kSlotsCols];
  u32 mh[kSlotsCols];
  u64 B[kSlotsCols];
  u32 nv, c0;      // what it was made for (nv 0: nothing yet)
};

// The map of chunks c0 + lane + 32 i.  NHD and latent pages hold their valid
// slots as nv whole rows, one run of nv rowb bytes; HND pages as one run of
// nv hb bytes per head, heads block_size hb bytes apart.
template <bool kHnd>
__device__ __forceinline__ void slot_map(SlotMap &sm, const DevCache &C, u32 nv, u32 bs,
                                         u32 c0, int lane) {
  sm.nv = nv;
  sm.c0 = c0;
  const u32 hb = static_cast<u32>(C.hb);
  const u32 row16 = static_cast<u32>(C.heads) * hb >> 4;   // chunks of one slot, all heads
  const u32 nch = nv * row16;
  const u64 P = static_cast<u64>(C.P);
#pragma unroll
  for (int i = 0; i < kSlotsCols; ++i) {
    const u32 c = c0 + static_cast<u32>(lane) + 32u * static_cast<u32>(i);
    u32 r, h, pp, off;
    if constexpr (kHnd) {
      const u32 cph = hb >> 4;           // chunks of one head's slot
      const u32 per_head = nv * cph;     // chunks of one head's valid run
      h = c / per_head;
      const u32 rem = c - h * per_head;
      r = rem / cph;
      pp = 2u * (rem - r * cph);
      off = h * bs * hb + (rem << 4);
    } else {
      r = c / row16;
      const u32 byte = (c - r * row16) << 4;
      h = C.hb_shift >= 0 ? byte >> C.hb_shift : byte / hb;
      pp = (byte - h * hb) >> 3;
      off = c << 4;
    }
    sm.off[i] = c < nch ? off : kSlotsNone;
    sm.mh[i] = 2u * h;
    sm.B[i] = 2ull * (static_cast<u64>(r) * P + static_cast<u64>(pp)) + 1ull;
  }
}

// Pages [i0, i1) of the (position, cache, half) order, walked by one warp:
// for each position with valid slots and each run of its pages of one
// column (the caches are sorted by column), windows wg, wg + G, ... of the
// valid chunks over the run's pages, two pages' loads at a time, then one
// 64-bit atomic of the warp's total into the output.
template <bool kHnd>
__device__ __forceinline__ void slots_range(const Params &p, long long i0, long long i1,
                                            u32 wg, u32 G, SlotMap &sm, int lane) {
  const long long ipp = p.pages_per_pos;
  const DevCache &C0 = p.caches[0];
  const int H = C0.halves;
  const u32 bs = static_cast<u32>(p.block_size);
  const u64 hstep = 2ull * static_cast<u64>(C0.hb >> 3);
  const u64 P = static_cast<u64>(C0.P);
  const u32 row16 = static_cast<u32>(C0.heads) * static_cast<u32>(C0.hb) >> 4;
  long long pos = i0 / ipp;
  int k = static_cast<int>(i0 - pos * ipp);
  ReqCursor rc = req_find_warp(p, pos, lane);
  while (true) {
    const int kend = static_cast<int>(min(ipp, i1 - pos * ipp));
    const long long b = p.block_ids[pos];
    const PosInfo pi = position_info_quiet(p, pos, rc, b, lane == 0 && k == 0);
    if (!pi.skip) {
      const u64 tw = 2ull * static_cast<u64>(pi.q) * static_cast<u64>(bs) * P;
      const u32 nv = static_cast<u32>(pi.nv);
      const u32 nch = nv * row16;
      for (int ka = k; ka < kend;) {
        const DevCache &Ca = p.caches[ka / H];
        const int col = Ca.column;
        const int kb = min(kend, Ca.run_end * H);
        u64 acc = 0;
        for (u32 cb = wg * kSlotsWindow; cb < nch; cb += G * kSlotsWindow) {
          if (sm.nv != nv || sm.c0 != cb) slot_map<kHnd>(sm, C0, nv, bs, cb, lane);
          for (int kk = ka; kk < kb; kk += kSlotsPages) {
            uint4 v[kSlotsPages][kSlotsCols];
            u64 m[kSlotsPages], bh[kSlotsPages];
#pragma unroll
            for (int j = 0; j < kSlotsPages; ++j) {
              const int pg = kk + j;
              const bool live = pg < kb;
              const int ci = (live ? pg : ka) / H;
              const int half = (live ? pg : ka) - ci * H;
              const DevCache &C = p.caches[ci];
              const unsigned char *src = C.base + static_cast<long long>(half) * C.half_stride +
                                         pi.block * C.block_stride;
              m[j] = C.m0;
              bh[j] = tw + (half ? hstep : 0ull);
#pragma unroll
              for (int i = 0; i < kSlotsCols; ++i)
                v[j][i] = live && sm.off[i] != kSlotsNone ? ld_stream16(src + sm.off[i])
                                                          : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < kSlotsPages; ++j) {
#pragma unroll
              for (int i = 0; i < kSlotsCols; ++i) {
                const u64 x0 = (static_cast<u64>(v[j][i].y) << 32) | v[j][i].x;
                const u64 x1 = (static_cast<u64>(v[j][i].w) << 32) | v[j][i].z;
                acc += (m[j] + sm.mh[i]) * ((sm.B[i] + bh[j]) * (x0 + x1) + 2ull * x1);
              }
            }
          }
        }
        const u64 tot = warp_sum(acc);
        if (lane == 0 && tot != 0) {
          ptx::grid_dep_wait();   // the output is zeroed by the kernel before this one
          atomicAdd(p.out + pos * p.num_columns + col, tot);
        }
        ka = kb;
      }
    }
    if ((pos + 1) * ipp >= i1) break;
    ++pos;
    k = 0;
    req_seek(p, rc, pos);
  }
}

// Persistent warps, as in the direct-load kernel: warp w of the grid owns a
// contiguous range of the first pool_start pages in (position, cache, half)
// order; with a work counter it then takes ranges of the remaining pages
// from the counter, of a size that shrinks as they run out (guided
// self-scheduling: the pages of a position hold the same valid slots, but
// positions differ, so fixed ranges alone can end far apart).  Each
// (position, column) total is added into the pre-zeroed output (or the
// caller's words, for accumulating calls) with one 64-bit atomic per warp.
// A call of few pages (never shared out dynamically) runs window_groups
// groups of warps, group g over all the pages but only windows g,
// g + window_groups, ... of each, so a page with many valid slots is read
// by several warps at once.  Every page of the launch has the same
// geometry; kHnd selects the HND walk (else NHD or latent).  No shared
// memory, no barrier: warps never wait for each other.
template <bool kHnd>
__global__ void __launch_bounds__(kSlotsThreads, kSlotsCtasPerSm)
    kvcs_slots_kernel(const __grid_constant__ Params p) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const long long warp = static_cast<long long>(blockIdx.x) * kSlotsWarps + (tid >> 5);
  const long long W = static_cast<long long>(gridDim.x) * kSlotsWarps;
  if (warp == 0 && lane == 0 && p.num_requests >= 0) {
    if (p.pos_offsets[0] != 0 || p.pos_offsets[p.num_requests] != p.total_positions)
      set_status(p, kStatusBadRequests);
  }
  const long long items = p.total_positions * p.pages_per_pos;
  SlotMap sm;
  sm.nv = 0;
  sm.c0 = 0;
  const long long G = p.window_groups > 1 ? p.window_groups : 1;
  if (G > 1) {
    // the grid is G groups of W / G warps (the host launches a multiple)
    const long long W0 = W / G, g = warp / W0, w0 = warp - g * W0;
    const long long i0 = items * w0 / W0, i1 = items * (w0 + 1) / W0;
    if (g < G && i0 < i1)
      slots_range<kHnd>(p, i0, i1, static_cast<u32>(g), static_cast<u32>(G), sm, lane);
    return;
  }
  const long long fixed = p.work ? p.pool_start : items;
  const long long i0 = fixed * warp / W, i1 = fixed * (warp + 1) / W;
  if (i0 < i1) slots_range<kHnd>(p, i0, i1, 0u, 1u, sm, lane);
  if (!p.work) return;
  // a range is taken only once the warp is free for it: taking one ahead
  // would hand out the pool before the warps' speeds are known
  long long left = items - fixed;   // pages left when this warp last took some
  while (true) {
    const long long n = max(kSlotsMinRange, left / (2 * W));
    u64 v = 0;
    if (lane == 0) v = atomicAdd(p.work, static_cast<u64>(n));
    const long long lo = fixed + static_cast<long long>(__shfl_sync(0xffffffffu, v, 0));
    if (lo >= items) break;
    const long long hi = min(lo + n, items);
    left = items - hi;
    slots_range<kHnd>(p, lo, hi, 0u, 1u, sm, lane);
  }
}

}  // namespace kvcs
