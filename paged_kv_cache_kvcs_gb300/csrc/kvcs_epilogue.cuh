// kvcs_epilogue.cuh -- row sums, tags and verification of offloaded KV, and
// the self-test of the bounded wait.
#pragma once

#include "kvcs_common.cuh"

namespace kvcs {

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

// Zeroes the n output words that the checksum kernels then add into, and the
// n_work work counters they take chunks from.  It is
// launched so that it may start while the stream's previous kernel ends, and
// first waits for all earlier work to finish.  Then it lets the next kernel
// of the stream start at once: that kernel reads its inputs meanwhile (all
// written by work that has finished) and waits for this grid before it
// writes an output word.
__global__ void __launch_bounds__(256)
    kvcs_zero_kernel(u64 *out, long long n, u64 *work, int n_work) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  for (long long i = t0; i < n; i += step) out[i] = 0ull;
  if (t0 < n_work) work[t0] = 0ull;   // the work counters of the launches
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
