// kvcs_state.cuh -- the state-row kernel: Mamba state caches the bulk-copy
// kernel cannot stage (rows of any size, blocks not 16-byte aligned).
#pragma once

#include "kvcs_common.cuh"

namespace kvcs {

// Work items are (position, state cache) pairs, taken grid-stride by CTAs of
// 256 threads.  A state block lives at block position 0 only; its rows are
// its slices and its 2- or 4-byte elements the pieces, each weighted 2e+1
// by element index e.  Each item's sum is added with a 64-bit atomic into
// the pre-zeroed output word of its (position, column), so a few positions
// with large states still spread over the whole GPU.
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
    kvcs_state_kernel(const __grid_constant__ Params p) {
  __shared__ u64 red[kGenericThreads / 32];
  const int tid = threadIdx.x;
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
    long long q = 0, b = 0;
    bool ok = r >= 0;
    if (ok) {
      q = p.first_position[r] + (pos - p.pos_offsets[r]);
      b = p.block_ids[pos];
      if (p.first_position[r] < 0) ok = false;
    }
    if (tid == 0 && ci == 0) {
      if (!ok) set_status(p, kStatusBadRequests);
      else if (b < 0 || b >= p.min_num_blocks) set_status(p, kStatusBadBlockId);
    }
    if (ok && (b < 0 || b >= p.min_num_blocks)) ok = false;
    u64 acc = 0;
    if (ok && q == 0) {
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
    acc = warp_sum(acc);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      u64 total = 0;
      for (int w = 0; w < kGenericThreads / 32; ++w) total += red[w];
      if (total) {
        ptx::grid_dep_wait();   // the output is zeroed by the kernel before this one
        atomicAdd(p.out + pos * p.num_columns + C.column, total);
      }
    }
    __syncthreads();
  }
}

}  // namespace kvcs
