// kvcs_write.cuh -- the KV write fused with the running block checksums.
#pragma once

#include "kvcs_common.cuh"

namespace kvcs {

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

// Loads of one batch of a token's row chunks for one cache: chunk idx = base
// + 32 k (K chunks first, then V chunks), up to eight per lane; chunks past
// the row are left untouched.
__device__ __forceinline__ void load_row_batch(const DevCache &C, const unsigned char *srck,
                                               const unsigned char *srcv, int base, int ch,
                                               uint4 (&v)[kWriteBatch]) {
  const int nh = (C.heads * C.hb) / ch;  // chunks per half
  const int n = nh * C.halves;
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
}

// One cache's K and V rows of one token: moved into the page slot `o` of
// block `b` by the calling warp, up to eight chunks per lane in flight (the
// K and V chunks of one batch together); returns the lane's share of the
// token's checksum term for this cache.  When `first` is set, the batch at
// base = lane was already loaded into v (its source does not depend on the
// slot, so it was issued together with the slot's load).  Byte `off` of a
// row (head h = off / hb, byte e = off mod hb) goes to, per layout:
//   NHD, latent  o*row + off
//   HND          ((o/kbs*heads + h)*kbs + o mod kbs)*hb + e
// (x-split pages have their own kernel below.)
template <int kLayout>
__device__ __forceinline__ u64 write_token_rows(const DevCache &C, const unsigned char *srck,
                                                const unsigned char *srcv, long long bs,
                                                long long b, long long o, u64 t, int ch,
                                                int lane, uint4 (&v)[kWriteBatch], bool first) {
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
    if (!(first && base == lane)) load_row_batch(C, srck, srcv, base, ch, v);
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
  // launched with programmatic stream serialization: wait for the stream's
  // earlier work before any access, then let the next kernel be scheduled
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
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
    // the table loads and the first cache's first batch of chunks in flight
    // together
    const long long slot = w.slots[i];
    const long long t = w.positions[i];
    uint4 v[kWriteBatch];
    {
      const DevCache &C0 = w.c[c_lo];
      const long long row0 = static_cast<long long>(C0.heads) * C0.hb;
      load_row_batch(C0, w.key[c_lo] + i * row0, w.value[c_lo] + i * row0, lane, ch, v);
    }
    if (slot < 0) continue;  // padding token
    const long long b = slot / bs;
    const long long o = slot - b * bs;
    if (b >= w.num_blocks) {
      if (lane == 0 && chunk == 0 && w.status) atomicOr(w.status, kStatusBadBlockId);
      continue;
    }
    if (t < 0 && lane == 0 && chunk == 0 && w.status) atomicOr(w.status, kStatusBadRequests);
    u64 acc = 0;
    for (int ci = c_lo; ci < c_hi; ++ci) {
      const DevCache &C = w.c[ci];
      const long long row = static_cast<long long>(C.heads) * C.hb;
      acc += write_token_rows<kLayout>(C, w.key[ci] + i * row, w.value[ci] + i * row, bs, b, o,
                                       static_cast<u64>(t), ch, lane, v, ci == c_lo);
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
  ptx::grid_dep_wait();   // as kvcs_write_kernel
  ptx::grid_dep_launch();
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
      const long long ti = w.positions[i];   // both table loads in flight together
      live = slot >= 0;  // padding token
      if (live) {
        b = slot / bs;
        o = slot - b * bs;
        if (b >= w.num_blocks) {
          if (ci == 0 && hk == 0 && w.status) atomicOr(w.status, kStatusBadBlockId);
          live = false;
        } else {
          t = ti;
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

}  // namespace kvcs
