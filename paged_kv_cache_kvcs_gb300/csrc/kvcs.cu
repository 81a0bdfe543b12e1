// kvcs.cu -- host side of the KV-cache block checksum library: argument
// validation, launch planning and the exported C ABI declared in kvcs.h.
//
// The library allocates no memory.  Every call validates its host arguments
// before touching CUDA, plans its kernel launches (the bulk-copy kernel per
// layout family; the direct-load kernel for KV caches it cannot stage; the
// state-row kernel for such state caches; the row-sum epilogue; or the write
// kernels) and enqueues them, plus, when CTAs or launches share positions,
// one kernel that zeroes the output first, on the caller's stream.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvcs.h"
#include "kvcs_bulk.cuh"
#include "kvcs_direct.cuh"
#include "kvcs_slots.cuh"
#include "kvcs_epilogue.cuh"
#include "kvcs_state.cuh"
#include "kvcs_write.cuh"

namespace kvcs {
namespace {

std::atomic<unsigned long long> g_launches{0};

constexpr u64 kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int kMaxDevices = 64;

struct DeviceState {
  std::mutex mu;
  std::atomic<bool> done{false};  // set only once the setup succeeded
  int sms = 0;
  std::atomic<u64 *> noalloc_scratch{nullptr};  // this device's g_noalloc_scratch
};
DeviceState g_dev[kMaxDevices];

// SM count of the current device; sets the bulk kernel's shared-memory
// attribute once per device.  A failed setup is not remembered: the next
// call on that device tries again.
cudaError_t device_setup(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceState &d = g_dev[dev];
  if (d.done.load(std::memory_order_acquire)) {
    *sms = d.sms;
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(d.mu);
  if (!d.done.load(std::memory_order_relaxed)) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    for (const void *fn : {reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamRows, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamHnd, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamXSplit, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamState, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamHndSub, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamRowsMis, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamHndMis, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamXSplitMis, false>),
                           reinterpret_cast<const void *>(kvcs_bulk_kernel<kFamRows, true>)})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    d.sms = n;
    d.done.store(true, std::memory_order_release);
  }
  *sms = d.sms;
  return cudaSuccess;
}

constexpr int kMaxColumns = 64;
// Positions of at most this many bytes, fewer than the SMs, are read one per
// CTA: split mode's memset and atomics would cost more than the imbalance.
constexpr long long kSmallPositionBytes = 128 * 1024;

// Bytes of one page: one block of K, of V, of latent rows, or of state rows.
long long page_bytes_of(const kvcs_cache &c, int block_size) {
  if (c.layout == KVCS_LAYOUT_STATE)
    return static_cast<long long>(c.num_heads) * c.head_bytes;
  return static_cast<long long>(block_size) * c.num_heads * c.head_bytes;
}

// NHD or latent rows of pages that may start 8 bytes past a 16-byte boundary
// (the base or a stride is 8 mod 16), rows whole 16-byte columns of one head:
// the bulk kernel's misaligned-rows instance stages them.
bool rows_misaligned(const kvcs_cache &c) {
  if (c.layout != KVCS_LAYOUT_NHD && c.layout != KVCS_LAYOUT_LATENT) return false;
  return reinterpret_cast<uintptr_t>(c.base) % 16 || c.half_stride % 16 || c.block_stride % 16;
}

// HND caches without kernel sub-blocks, and x-split caches, whose pages may
// start 8 bytes past a 16-byte boundary: a unit's heads, all slots of them,
// are one contiguous run, staged as misaligned rows are.
bool hnd_misaligned(const kvcs_cache &c, int block_size) {
  if (c.layout == KVCS_LAYOUT_HND) {
    if (c.kernel_block_size > 0 && c.kernel_block_size != block_size) return false;
  } else if (c.layout != KVCS_LAYOUT_XSPLIT) {
    return false;
  }
  return reinterpret_cast<uintptr_t>(c.base) % 16 || c.half_stride % 16 || c.block_stride % 16;
}

// Pages of the cache staged with the misaligned split (rows or HND heads).
bool staged_misaligned(const kvcs_cache &c, int block_size) {
  return rows_misaligned(c) || hnd_misaligned(c, block_size);
}

// The bulk kernel stages whole rows (NHD, latent, state) or whole heads
// (HND, x-split) with 16-byte-aligned bulk copies and reads 16-byte columns;
// NHD and latent pages 8 bytes off a 16-byte boundary too, their edge words
// by 8-byte asynchronous copies.
bool bulk_eligible(const kvcs_cache &c, int block_size) {
  if (c.head_bytes % 16) return false;
  if (!staged_misaligned(c, block_size) &&
      (reinterpret_cast<uintptr_t>(c.base) % 16 || c.half_stride % 16 || c.block_stride % 16))
    return false;
  const long long hb = c.head_bytes;
  switch (c.layout) {
    case KVCS_LAYOUT_NHD: return hb * c.num_heads <= kMaxUnitBytes;
    case KVCS_LAYOUT_HND:
    case KVCS_LAYOUT_XSPLIT: return hb * block_size <= kMaxUnitBytes;
    default: return hb <= kMaxUnitBytes;  // latent and state rows
  }
}

// Host-argument checks shared by every entry point.  Every column in
// [0, num_columns) must be named by at least one cache.  State caches (Mamba
// running states) cannot be mixed with KV caches in one call.
int validate_caches(const kvcs_cache *caches, int32_t num_caches,
                    int32_t block_size, int32_t num_columns) {
  if (!caches || num_caches < 1 || block_size <= 0) return KVCS_EINVAL;
  if (num_columns < 1 || num_columns > kMaxColumns) return KVCS_EINVAL;
  bool used[kMaxColumns] = {false};
  struct Span {
    int32_t layer;
    int64_t lo, hi;
  };
  std::vector<Span> spans;
  spans.reserve(num_caches);
  int states = 0;
  for (int32_t i = 0; i < num_caches; ++i) {
    const kvcs_cache &c = caches[i];
    if (!c.base || c.num_blocks < 0) return KVCS_EINVAL;
    if (c.layout < KVCS_LAYOUT_NHD || c.layout > KVCS_LAYOUT_STATE) return KVCS_EINVAL;
    if (c.column < 0 || c.column >= num_columns) return KVCS_EINVAL;
    used[c.column] = true;
    if (c.layer < 0 || c.head_offset < 0 || c.num_heads < 1) return KVCS_EINVAL;
    if (c.layout == KVCS_LAYOUT_STATE) {
      ++states;
      if (c.piece_bytes != 2 && c.piece_bytes != 4) return KVCS_EINVAL;
      if (c.head_bytes <= 0 || c.head_bytes % c.piece_bytes) return KVCS_EINVAL;
    } else {
      if (c.piece_bytes != 0) return KVCS_EINVAL;
      if (c.head_bytes <= 0 || c.head_bytes % 8) return KVCS_EINVAL;
    }
    if (c.layout == KVCS_LAYOUT_LATENT && c.num_heads != 1) return KVCS_EINVAL;
    if (c.layout == KVCS_LAYOUT_XSPLIT && c.head_bytes % 16) return KVCS_EINVAL;
    if (reinterpret_cast<uintptr_t>(c.base) % 8) return KVCS_EINVAL;
    if (static_cast<int64_t>(c.head_offset) + c.num_heads > KVCS_MAX_KV_HEADS_PER_LAYER)
      return KVCS_EUNSUPPORTED;
    // Bytes must stay addressable in 64 bits (always true for real pools;
    // guards absurd descriptors).
    const double page = static_cast<double>(page_bytes_of(c, block_size));
    if (page * 2.0 * static_cast<double>(c.num_blocks) > 9.0e18) return KVCS_EINVAL;
    // Strides: 8-byte multiples; pages of different blocks, and a block's K
    // and V pages, must not overlap.
    if (c.half_stride % 8 || c.block_stride % 8) return KVCS_EINVAL;
    if (c.block_stride != 0 && static_cast<double>(c.block_stride) < page) return KVCS_EINVAL;
    const bool two_halves = c.layout != KVCS_LAYOUT_LATENT && c.layout != KVCS_LAYOUT_STATE;
    if (two_halves && c.half_stride != 0 && std::fabs(static_cast<double>(c.half_stride)) < page)
      return KVCS_EINVAL;
    if (std::fabs(static_cast<double>(c.half_stride)) > 9.0e18 ||
        std::fabs(static_cast<double>(c.block_stride)) * static_cast<double>(c.num_blocks) > 9.0e18)
      return KVCS_EINVAL;
    if (c.kernel_block_size < 0 ||
        (c.kernel_block_size > 0 && block_size % c.kernel_block_size != 0))
      return KVCS_EINVAL;
    spans.push_back({c.layer, c.head_offset,
                     static_cast<int64_t>(c.head_offset) + c.num_heads});
  }
  if (states != 0 && states != num_caches) return KVCS_EINVAL;
  std::sort(spans.begin(), spans.end(), [](const Span &a, const Span &b) {
    return a.layer != b.layer ? a.layer < b.layer : a.lo < b.lo;
  });
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].layer == spans[i - 1].layer && spans[i].lo < spans[i - 1].hi)
      return KVCS_EINVAL;  // two caches weigh the same (layer, global head)
  for (int k = 0; k < num_columns; ++k)
    if (!used[k]) return KVCS_EINVAL;  // a column no cache adds into
  return KVCS_OK;
}

// The caches in column order (stable): a column's units are then
// consecutive within every position, which the kernels rely on.
std::vector<kvcs_cache> by_column(const kvcs_cache *caches, int32_t num_caches) {
  std::vector<kvcs_cache> v(caches, caches + num_caches);
  std::stable_sort(v.begin(), v.end(), [](const kvcs_cache &a, const kvcs_cache &b) {
    return a.column < b.column;
  });
  return v;
}

DevCache make_dev_cache(const kvcs_cache &c, int block_size) {
  DevCache d;
  std::memset(&d, 0, sizeof(d));
  d.base = static_cast<const unsigned char *>(c.base);
  d.m0 = 2ull * (static_cast<u64>(c.layer) * KVCS_MAX_KV_HEADS_PER_LAYER +
                 static_cast<u64>(c.head_offset)) + 1ull;
  d.layout = c.layout;
  d.heads = c.num_heads;
  d.hb = c.head_bytes;
  d.page_bytes = static_cast<u64>(page_bytes_of(c, block_size));
  d.half_stride = c.half_stride != 0
                      ? c.half_stride
                      : static_cast<long long>(c.num_blocks) * static_cast<long long>(d.page_bytes);
  d.block_stride = c.block_stride != 0 ? c.block_stride
                                       : static_cast<long long>(d.page_bytes);
  d.kbs = (c.layout == KVCS_LAYOUT_HND && c.kernel_block_size > 0) ? c.kernel_block_size
                                                                  : block_size;
  d.chunks = c.layout == KVCS_LAYOUT_XSPLIT ? c.head_bytes / 16 : 1;
  d.pbytes = c.layout == KVCS_LAYOUT_STATE ? c.piece_bytes : 8;
  d.halves = (c.layout == KVCS_LAYOUT_LATENT || c.layout == KVCS_LAYOUT_STATE) ? 1 : 2;
  d.P = c.layout == KVCS_LAYOUT_STATE
            ? c.head_bytes / c.piece_bytes
            : (c.layout == KVCS_LAYOUT_LATENT ? c.head_bytes : 2 * c.head_bytes) / 8;
  d.column = c.column;
  d.hb_shift = -1;
  for (int k = 0; k < 31; ++k)
    if (c.head_bytes == (1 << k)) d.hb_shift = k;
  // Units: cut a page into runs of about kUnitTargetBytes, as evenly as
  // possible, of whole rows (NHD, latent, state) or whole heads (HND,
  // x-split).
  if (c.layout == KVCS_LAYOUT_HND || c.layout == KVCS_LAYOUT_XSPLIT) {
    d.rowb = c.layout == KVCS_LAYOUT_HND ? c.head_bytes : 16;
    const long long head = static_cast<long long>(block_size) * c.head_bytes;
    const int fit = static_cast<int>(std::max<long long>(1, kUnitTargetBytes / head));
    d.upp = (c.num_heads + fit - 1) / fit;
    d.rpu = (c.num_heads + d.upp - 1) / d.upp;
  } else {
    d.rowb = c.layout == KVCS_LAYOUT_NHD ? c.num_heads * c.head_bytes : c.head_bytes;
    const int rows = c.layout == KVCS_LAYOUT_STATE ? c.num_heads : block_size;
    const int fit = std::max(1, kUnitTargetBytes / std::max(1, d.rowb));
    d.upp = (rows + fit - 1) / fit;
    d.rpu = (rows + d.upp - 1) / d.upp;
  }
  return d;
}

// Largest unit of one cache, in bytes of stage.
long long unit_bytes(const kvcs_cache &c, const DevCache &d, int block_size) {
  if (d.layout == KVCS_LAYOUT_HND || d.layout == KVCS_LAYOUT_XSPLIT)
    return static_cast<long long>(d.rpu) * block_size * d.hb +
           (hnd_misaligned(c, block_size) ? kMisPad : 0);
  return static_cast<long long>(d.rpu) * d.rowb + (rows_misaligned(c) ? kMisPad : 0);
}

// Shape of one bulk launch over caches [lo, hi): units per position,
// whether pages are packed several to a stage, stage size and count.
struct LaunchShape {
  long long units_per_pos = 0;
  int pack = 0;
  int full_pages = 1;
  int pages_per_pos = 0;
  int stage_bytes = 0;
  int stages = 0;
};

LaunchShape launch_shape(const kvcs_cache *caches, int lo, int hi, int block_size) {
  LaunchShape ls;
  bool uniform = true;
  long long biggest = 16;
  const DevCache d0 = make_dev_cache(caches[lo], block_size);
  for (int i = lo; i < hi; ++i) {
    const DevCache d = make_dev_cache(caches[i], block_size);
    ls.units_per_pos += static_cast<long long>(d.halves) * d.upp;
    ls.pages_per_pos += d.halves;
    biggest = std::max(biggest, unit_bytes(caches[i], d, block_size));
    uniform = uniform && d.upp == 1 && caches[i].layout == caches[lo].layout &&
              caches[i].column == caches[lo].column && d.kbs == d0.kbs &&
              caches[i].num_heads == caches[lo].num_heads &&
              caches[i].head_bytes == caches[lo].head_bytes &&
              caches[i].piece_bytes == caches[lo].piece_bytes;
  }
  if (uniform) {
    // Every page fits a unit and all pages look alike: each page is a unit,
    // and the producer packs consecutive pages of a position (e.g. a layer's
    // K and V) into one stage as far as their valid bytes fit.  The stage
    // holds as many whole pages as fit in the unit target.
    // (pages are counted against the target without the misaligned-rows
    // padding, so a stage packs as many pages as in an aligned pool)
    const long long page = static_cast<long long>(d0.page_bytes);
    long long ppu = std::max<long long>(
        1, std::min<long long>(ls.pages_per_pos, kUnitTargetBytes / page));
    const bool mis = staged_misaligned(caches[lo], block_size);
    if (mis) ppu = std::min<long long>(ppu, kMisMaxPages);
    ls.pack = 1;
    ls.full_pages = static_cast<int>(ppu);
    biggest = std::max(biggest, ppu * (page + (mis ? kMisPad : 0)));
  }
  ls.stage_bytes = static_cast<int>((biggest + 127) / 128 * 128);
  ls.stages = std::min(kMaxStages, (kSmemLimit - kHeaderBytes) / ls.stage_bytes);
  return ls;
}

// Consumer warps per group: the smallest of 1, 2, 4, 8 (at least
// kMinGroupWarps) that leaves no more groups than stages.
int group_warps_for(int stages) {
  int gw = kMinGroupWarps;
  while (gw < kConsumerWarps && kConsumerWarps / gw > stages) gw *= 2;
  return gw;
}

// Layout family of a cache (which instance of the bulk kernel stages it).
int family_of(const kvcs_cache &c, int block_size) {
  switch (c.layout) {
    case KVCS_LAYOUT_HND:
      return c.kernel_block_size > 0 && c.kernel_block_size != block_size ? kFamHndSub
             : hnd_misaligned(c, block_size)                               ? kFamHndMis
                                                                           : kFamHnd;
    case KVCS_LAYOUT_XSPLIT: return hnd_misaligned(c, block_size) ? kFamXSplitMis : kFamXSplit;
    case KVCS_LAYOUT_STATE: return kFamState;
    default: return rows_misaligned(c) ? kFamRowsMis : kFamRows;
  }
}

// One kernel launch: a kernel (the bulk instance of one layout family, the
// direct-load kernel or the state-row kernel) and a run of (column-sorted)
// caches.
constexpr int kKernelBulk = 0;
constexpr int kKernelDirect = 1;
constexpr int kKernelState = 2;
constexpr int kKernelSlots = 3;

struct Launch {
  int kernel;
  int family;
  std::vector<kvcs_cache> caches;
};

// How a call runs: caches the bulk kernel can stage go to its instance for
// their layout family (up to kMaxCachesPerLaunch per launch), the other KV
// caches to the direct-load kernel and the other state caches to the
// state-row kernel.  In a call whose blocks are mostly partial (at most two
// positions per request), a launch of alike latent or HND pages, or of NHD
// pages of at most kSlotsNhdPageBytes, goes to the valid-slot kernel
// instead.  With more than one launch, or a
// direct-load, state-row or valid-slot launch, every result is added
// atomically into an output zeroed first.
struct Plan {
  std::vector<Launch> launches;
  int kernel = 0;         // 0 bulk only, 1 direct loads only, 2 both
  int split = 0;          // bulk CTA ranges cut positions
  int bulk_grid = 0;
  int generic_grid = 0;   // direct-load or state-row kernel
  int stage_bytes = 0;    // of the first bulk launch
  int stages = 0;
  long long units = 0;    // units of the largest bulk launch
  long long kv_bytes_max = 0;
  bool all_atomic = false;
  bool memset = false;
  bool dynamic = false;   // bulk launches share the last units out by a counter
};

// Bulk launches with at least this many units per SM share the last part of
// their units out dynamically when the call has a workspace.  Below it a
// CTA's fixed share is only a few chunks long, and the CTAs that take the
// last chunks end later than an even fixed split would (one 70B-shaped
// request of 2048 tokens, 134 units per SM, ran 11% slower with them; from
// about 1000 units per SM on the share-out gains).
constexpr long long kDynamicUnitsPerSm = 1024;
// The part shared out dynamically (1 / kPoolShare of the units) and the
// chunks it is taken in (about kChunksPerCta chunks a CTA, at least
// kMinChunkUnits units).
constexpr long long kPoolShare = 16;
constexpr long long kChunksPerCta = 8;
constexpr long long kMinChunkUnits = 16;

// Caches of one launch the valid-slot kernel reads: latent or HND (no kernel
// sub-blocks) pages, and NHD pages of at most kSlotsNhdPageBytes, that the
// bulk kernel stages without the misaligned split, all of one geometry, each
// page under 2 GiB (its byte offsets fit 32 bits).  Larger NHD pages of such
// calls stay with the bulk kernel: a partial NHD page's valid slots are one
// contiguous run, which its bulk copies fetch with more bytes in flight than
// registers hold.  Measured on the newest blocks of 8192 requests of 1 to
// block_size - 1 tokens, 32 layers: pages of 4 and 8 KiB 6-38% faster on this
// kernel, pages of 16 and 32 KiB 2-7% faster on the bulk kernel (with one
// token a block this kernel was 41-97% faster at every page size).
constexpr long long kSlotsNhdPageBytes = 8192;
bool slots_eligible(int family, const kvcs_cache *c, size_t n, int32_t block_size) {
  if (family == kFamRows) {
    if (c[0].layout != KVCS_LAYOUT_LATENT && page_bytes_of(c[0], block_size) > kSlotsNhdPageBytes)
      return false;
  } else if (family != kFamHnd) {
    return false;
  }
  for (size_t i = 0; i < n; ++i) {
    if (c[i].layout != c[0].layout || c[i].num_heads != c[0].num_heads ||
        c[i].head_bytes != c[0].head_bytes)
      return false;
  }
  return page_bytes_of(c[0], block_size) < (1LL << 31);
}

// CTAs of a valid-slot launch over `pages` pages: kSlotsCtasPerSm a SM,
// fewer when there are few pages (a warp at least kSlotsPages of them).
long long slots_grid(long long pages, int sms) {
  const long long per_cta = static_cast<long long>(kSlotsWarps) * kSlotsPages;
  return std::max<long long>(1, std::min<long long>(static_cast<long long>(kSlotsCtasPerSm) * sms,
                                                    (pages + per_cta - 1) / per_cta));
}

// Window groups of a valid-slot launch of `grid` CTAs (slots_grid): a call
// whose pages leave SMs idle runs up to four times the CTAs, groups of them
// splitting each page's windows of valid chunks.
long long slots_window_groups(long long grid, int sms) {
  const long long full = static_cast<long long>(kSlotsCtasPerSm) * sms;
  return grid < full ? std::max<long long>(1, std::min<long long>(4, full / grid)) : 1;
}

// Whether a valid-slot launch with a work counter hands its last pages out
// from it: at least kSlotsDynamicPages pages a warp.
bool slots_dynamic(long long pages, long long grid) {
  return pages >= kSlotsDynamicPages * kSlotsWarps * grid;
}

// num_requests < 0: not known (kvcs_plan), planned as a call of whole blocks.
Plan make_plan(const std::vector<kvcs_cache> &sorted, int32_t block_size,
               int64_t total_positions, int sms, bool accumulate = false,
               bool workspace = false, long long num_requests = -1) {
  Plan pl;
  std::vector<kvcs_cache> fam[kNumFamilies], gen;
  std::vector<kvcs_cache> bulk;
  for (const kvcs_cache &c : sorted) {
    if (bulk_eligible(c, block_size)) {
      fam[family_of(c, block_size)].push_back(c);
      bulk.push_back(c);
    } else {
      gen.push_back(c);
    }
    const long long halves =
        (c.layout == KVCS_LAYOUT_LATENT || c.layout == KVCS_LAYOUT_STATE) ? 1 : 2;
    pl.kv_bytes_max += halves * page_bytes_of(c, block_size) * total_positions;
  }
  const bool partial = num_requests >= 0 && total_positions <= 2 * num_requests;
  bool has_bulk = false, has_slots = false;
  for (int f = 0; f <= kNumFamilies; ++f) {
    const std::vector<kvcs_cache> &set = f < kNumFamilies ? fam[f] : gen;
    for (size_t lo = 0; lo < set.size(); lo += kMaxCachesPerLaunch) {
      const size_t hi = std::min(set.size(), lo + kMaxCachesPerLaunch);
      int kernel = f < kNumFamilies ? kKernelBulk
                   : set[lo].layout == KVCS_LAYOUT_STATE ? kKernelState
                                                          : kKernelDirect;
      if (kernel == kKernelBulk && partial &&
          slots_eligible(f, set.data() + lo, hi - lo, block_size))
        kernel = kKernelSlots;
      has_bulk = has_bulk || kernel == kKernelBulk;
      has_slots = has_slots || kernel == kKernelSlots;
      pl.launches.push_back({kernel, f < kNumFamilies ? f : 0,
                             std::vector<kvcs_cache>(set.begin() + lo, set.begin() + hi)});
    }
  }
  pl.kernel = gen.empty() ? 0 : (bulk.empty() ? 1 : 2);
  // accumulating calls add every result into the caller's values
  pl.all_atomic = accumulate || pl.launches.size() > 1 || !gen.empty() || has_slots;
  if (sms < 1) sms = 1;
  if (has_bulk) {
    bool first = true;
    for (const Launch &l : pl.launches) {
      if (l.kernel != kKernelBulk) continue;
      const LaunchShape ls = launch_shape(l.caches.data(), 0,
                                          static_cast<int>(l.caches.size()), block_size);
      pl.units = std::max(pl.units, ls.units_per_pos * total_positions);
      if (first) {
        pl.stage_bytes = ls.stage_bytes;
        pl.stages = ls.stages;
        first = false;
      }
    }
    // With a workspace and enough units: every CTA a fixed share, the rest
    // taken in chunks from a counter; whole positions per CTA when that
    // balances well (>= 99% of the even split); otherwise split at unit
    // granularity.
    const double per = static_cast<double>(total_positions) / sms;
    const double eff = per / std::ceil(per > 0 ? per : 1.0);
    if (workspace && pl.units >= kDynamicUnitsPerSm * sms) {
      pl.dynamic = true;
      pl.split = 1;
      pl.bulk_grid = sms;
    } else if (total_positions >= sms && eff >= 0.99) {
      pl.split = 0;
      pl.bulk_grid = sms;
    } else if (total_positions < sms &&
               pl.kv_bytes_max <= kSmallPositionBytes * total_positions) {
      // few small positions: one CTA each, no memset and no atomics
      pl.split = 0;
      pl.bulk_grid = static_cast<int>(total_positions);
    } else {
      pl.split = 1;
      pl.bulk_grid = static_cast<int>(std::max<long long>(1, std::min<long long>(sms, pl.units)));
    }
  }
  if (!gen.empty()) {
    long long items = 0;
    for (const Launch &l : pl.launches) {
      if (l.kernel == kKernelBulk) continue;
      long long n = total_positions * static_cast<long long>(l.caches.size());
      // the direct-load kernel takes pages, a warp each, eight warps a CTA
      if (l.kernel == kKernelDirect) n = (2 * n + kDirectThreads / 32 - 1) / (kDirectThreads / 32);
      items = std::max<long long>(items, n);
    }
    // a state cache is all state or all KV, so one kind of kernel runs here
    const long long per_sm = gen[0].layout == KVCS_LAYOUT_STATE ? 8 : 4;
    pl.generic_grid = static_cast<int>(std::max<long long>(
        1, std::min<long long>(static_cast<long long>(sms) * per_sm, items)));
  }
  if (pl.dynamic) pl.all_atomic = true;
  pl.memset = !accumulate && total_positions > 0 &&
              (pl.all_atomic || (has_bulk && pl.split));
  return pl;
}

// Launch a checksum kernel.  Right after the zeroing kernel it is launched
// with programmatic stream serialization: it may start while the zeroing runs
// (every kernel waits for it before writing an output word; the zeroing
// kernel itself waited for all earlier work before letting it start).  Any
// other launch waits for the stream's earlier work as usual, so a kernel
// before it that lets its dependents start early can never have them read
// its inputs.
cudaError_t launch(void (*kernel)(Params), dim3 grid, int threads, size_t smem, cudaStream_t st,
                   bool after_zero, const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (after_zero) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// A write kernel, launched with programmatic stream serialization: it may be
// scheduled while the stream's previous kernel ends, and waits
// (griddepcontrol.wait) for all earlier work before it touches memory.  A
// run of one-layer calls, as a forward pass issues them, then pays the
// launch latency of each once, overlapped with the previous call.
cudaError_t launch_write(void (*kernel)(WriteParams), unsigned grid, cudaStream_t st,
                         const WriteParams &w) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(static_cast<unsigned>(kWriteThreads));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, w);
}

// Shared body of kvcs_block_checksums and kvcs_group_checksums.
int run_checksums(const kvcs_cache *caches_in, int32_t num_caches, int32_t block_size,
                  const kvcs_requests *reqs, int64_t total_positions,
                  const kvcs_outputs *outs, uint32_t *status, cudaStream_t st) {
  if (!outs || (outs->flags & ~(KVCS_OUT_ACCUMULATE | KVCS_OUT_WORKSPACE)) != 0)
    return KVCS_EINVAL;
  const bool accumulate = (outs->flags & KVCS_OUT_ACCUMULATE) != 0;
  // the workspace field exists only when the flag says so (ABI minor 3)
  u64 *workspace = (outs->flags & KVCS_OUT_WORKSPACE)
                       ? reinterpret_cast<u64 *>(outs->workspace) : nullptr;
  if ((outs->flags & KVCS_OUT_WORKSPACE) &&
      (!workspace || reinterpret_cast<uintptr_t>(workspace) % 8))
    return KVCS_EINVAL;
  const int ncols = outs->num_columns;
  int rc = validate_caches(caches_in, num_caches, block_size, ncols);
  if (rc != KVCS_OK) return rc;
  if (!reqs || total_positions < 0 || reqs->num_requests < 0) return KVCS_EINVAL;
  if ((outs->mismatch || outs->mismatch_count) && !outs->expected) return KVCS_EINVAL;
  if (total_positions == 0) return KVCS_OK;
  if (!outs->values || !reqs->pos_offsets || !reqs->first_position ||
      !reqs->num_tokens || !reqs->block_ids)
    return KVCS_EINVAL;
  if (reinterpret_cast<uintptr_t>(outs->values) % 8) return KVCS_EINVAL;

  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return KVCS_ECUDA;
  const Plan pl = make_plan(by_column(caches_in, num_caches), block_size, total_positions, sms,
                            accumulate, workspace != nullptr, reqs->num_requests);
  // one work counter per dynamic bulk launch, at most KVCS_WORKSPACE_WORDS
  // (and one per valid-slot launch, whose items are then handed out one at
  // a time)
  int n_work = 0;
  for (const Launch &l : pl.launches)
    if (((l.kernel == kKernelBulk && pl.dynamic) || (l.kernel == kKernelSlots && workspace)) &&
        n_work < KVCS_WORKSPACE_WORDS)
      ++n_work;

  if (pl.memset || n_work > 0) {
    // zero the output with a kernel that lets the first checksum launch start
    // at once (that launch waits for it before writing any output word)
    // (an accumulating call zeroes only the work counters)
    const long long words = pl.memset ? total_positions * static_cast<long long>(ncols) : 0;
    const long long blocks = std::max<long long>(
        1, std::min<long long>((words + 1023) / 1024, static_cast<long long>(sms)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kvcs_zero_kernel, reinterpret_cast<u64 *>(outs->values),
                           words, workspace, n_work) != cudaSuccess)
      return KVCS_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  bool after_zero = pl.memset || n_work > 0;
  int work_used = 0;

  long long min_nb = caches_in[0].num_blocks;
  for (int32_t i = 1; i < num_caches; ++i) min_nb = std::min<long long>(min_nb, caches_in[i].num_blocks);

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.pos_offsets = reinterpret_cast<const long long *>(reqs->pos_offsets);
  p.first_position = reinterpret_cast<const long long *>(reqs->first_position);
  p.num_tokens = reinterpret_cast<const long long *>(reqs->num_tokens);
  p.block_ids = reinterpret_cast<const int *>(reqs->block_ids);
  p.out = reinterpret_cast<u64 *>(outs->values);
  p.status = status;
  p.num_requests = reqs->num_requests;
  p.total_positions = total_positions;
  p.min_num_blocks = min_nb;
  p.timeout_ns = kTimeoutNs;
  p.block_size = block_size;
  p.all_atomic = pl.all_atomic ? 1 : 0;
  p.num_columns = ncols;
  p.state_call = caches_in[0].layout == KVCS_LAYOUT_STATE ? 1 : 0;

  for (const Launch &l : pl.launches) {
    const int n = static_cast<int>(l.caches.size());
    p.num_caches = n;
    long long U = 0;
    for (int i = 0; i < n; ++i) {
      p.caches[i] = make_dev_cache(l.caches[i], block_size);
      U += static_cast<long long>(p.caches[i].halves) * p.caches[i].upp;
    }
    for (int i = n - 1; i >= 0; --i)
      p.caches[i].run_end = i + 1 < n && p.caches[i + 1].column == p.caches[i].column
                                ? p.caches[i + 1].run_end : i + 1;
    p.pack = 0;
    p.full_pages = 1;
    p.pages_per_pos = 0;
    for (int i = 0; i < n; ++i) p.pages_per_pos += p.caches[i].halves;
    if (l.kernel == kKernelBulk) {
      const LaunchShape ls = launch_shape(l.caches.data(), 0, n, block_size);
      U = ls.units_per_pos;
      p.pack = ls.pack;
      p.full_pages = ls.full_pages;
      p.pages_per_pos = ls.pages_per_pos;
      p.stage_bytes = ls.stage_bytes;
      p.stages = ls.stages;
    }
    p.units_per_pos = U;
    p.total_units = U * total_positions;
    p.work = nullptr;
    p.pool_start = p.total_units;
    p.chunk_units = 1;
    if (l.kernel == kKernelBulk && pl.dynamic && work_used < n_work) {
      // the last 1/kPoolShare of the units go out in chunks of about
      // 1/kChunksPerCta of a CTA's share of them
      p.work = workspace + work_used++;
      const long long pool = p.total_units / kPoolShare;
      p.pool_start = p.total_units - pool;
      p.chunk_units = std::max<long long>(
          kMinChunkUnits, pool / (static_cast<long long>(pl.bulk_grid) * kChunksPerCta));
    }
    if (l.kernel == kKernelBulk) {
      // Calls whose blocks are mostly partial (at most one block of a
      // request is partial, so at most about two positions per request)
      // pack many pages into a unit; their NHD pages take the instance
      // whose whole producer warp issues the copies and whose consumers
      // reduce packed units at once.  Its producers, not DRAM, set the
      // pace, so it runs two CTAs a SM (two producers), each with half the
      // shared memory: its page-address table and a ring of fewer stages.
      // (Such calls' latent and HND pages, and NHD pages of at most
      // kSlotsNhdPageBytes, go to the valid-slot kernel.)
      const bool wide = p.pack && total_positions <= 2 * reqs->num_requests &&
                        l.family == kFamRows;
      if (wide)
        p.stages = std::max(1, std::min(p.stages, (kSmemLimit / 2 - 1024 - kHeaderBytes -
                                                    kWideTableBytes) / p.stage_bytes));
      p.split = pl.split;
      p.group_warps = group_warps_for(p.stages);
      p.groups = kConsumerWarps / p.group_warps;
      long long grid = pl.bulk_grid * (wide ? 2 : 1);
      if (p.split) grid = std::max<long long>(1, std::min<long long>(grid, p.total_units));
      const size_t smem = bulk_smem_bytes(p.stages, p.stage_bytes) + (wide ? kWideTableBytes : 0);
      const dim3 gd(static_cast<unsigned>(grid));
      cudaError_t e;
      switch (l.family) {
        case kFamHnd:
          e = launch(kvcs_bulk_kernel<kFamHnd, false>, gd, kBulkThreads, smem, st, after_zero, p);
          break;
        case kFamXSplit: e = launch(kvcs_bulk_kernel<kFamXSplit, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        case kFamState: e = launch(kvcs_bulk_kernel<kFamState, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        case kFamHndSub: e = launch(kvcs_bulk_kernel<kFamHndSub, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        case kFamRowsMis: e = launch(kvcs_bulk_kernel<kFamRowsMis, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        case kFamHndMis: e = launch(kvcs_bulk_kernel<kFamHndMis, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        case kFamXSplitMis: e = launch(kvcs_bulk_kernel<kFamXSplitMis, false>, gd, kBulkThreads, smem, st, after_zero, p); break;
        default:
          e = wide ? launch(kvcs_bulk_kernel<kFamRows, true>, gd, kBulkThreads, smem, st, after_zero, p)
                   : launch(kvcs_bulk_kernel<kFamRows, false>, gd, kBulkThreads, smem, st, after_zero, p);
          break;
      }
      if (e != cudaSuccess) return KVCS_ECUDA;
    } else if (l.kernel == kKernelSlots) {
      p.split = 0;
      const long long pages = total_positions * p.pages_per_pos;
      const long long g0 = slots_grid(pages, sms);
      const long long wg = slots_window_groups(g0, sms);
      const long long grid = g0 * wg;
      p.window_groups = static_cast<int>(wg);
      // with a work counter, on enough pages: the last pages handed out from
      // it (never with window groups: those calls have few pages)
      p.pool_start = pages;
      if (workspace && work_used < n_work) {
        p.work = workspace + work_used++;
        if (wg == 1 && slots_dynamic(pages, g0)) p.pool_start = pages / kSlotsFixedShare;
      }
      const dim3 gd(static_cast<unsigned>(grid));
      const cudaError_t e =
          l.family == kFamHnd
              ? launch(kvcs_slots_kernel<true>, gd, kSlotsThreads, 0, st, after_zero, p)
              : launch(kvcs_slots_kernel<false>, gd, kSlotsThreads, 0, st, after_zero, p);
      if (e != cudaSuccess) return KVCS_ECUDA;
    } else if (l.kernel == kKernelDirect) {
      p.split = 0;
      if (launch(kvcs_direct_kernel, dim3(static_cast<unsigned>(pl.generic_grid)), kDirectThreads,
                 0, st, after_zero, p) != cudaSuccess)
        return KVCS_ECUDA;
    } else {
      p.split = 0;
      if (launch(kvcs_state_kernel, dim3(static_cast<unsigned>(pl.generic_grid)), kGenericThreads,
                 0, st, after_zero, p) != cudaSuccess)
        return KVCS_ECUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return KVCS_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    after_zero = false;
  }

  if (outs->row_sums || outs->expected) {
    RowParams rp;
    rp.values = reinterpret_cast<const u64 *>(outs->values);
    rp.n = total_positions;
    rp.num_columns = ncols;
    rp.row_sums = reinterpret_cast<u64 *>(outs->row_sums);
    rp.tags = reinterpret_cast<const u64 *>(outs->tags);
    rp.expected = reinterpret_cast<const u64 *>(outs->expected);
    rp.mismatch = outs->mismatch;
    rp.mismatch_count = outs->mismatch_count;
    const long long blocks = std::min<long long>((total_positions + 255) / 256, 4LL * sms);
    kvcs_rows_kernel<<<static_cast<unsigned>(std::max<long long>(1, blocks)), 256, 0, st>>>(rp);
    if (cudaGetLastError() != cudaSuccess) return KVCS_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return KVCS_OK;
}

// Scratch of kvcs_block_checksums_noalloc: the bulk kernel's work counters
// for callers that cannot lend a workspace.  A module-scope device array,
// so every GPU that loads the library holds its 128 bytes until the process
// exits; on the host its name only stands for the symbol (its device
// address comes from cudaGetSymbolAddress).
static __device__ __align__(256) u64 g_noalloc_scratch[KVCS_WORKSPACE_WORDS];

// Within KVCS_NOALLOC_MAX_CACHES caches a call never has more bulk-copy
// launches (per layout family, groups of kMaxCachesPerLaunch) than counters.
static_assert(KVCS_NOALLOC_MAX_CACHES / kMaxCachesPerLaunch + kNumFamilies <=
                  KVCS_WORKSPACE_WORDS,
              "the no-alloc scratch must hold a counter per bulk launch");

// Device address of g_noalloc_scratch on the current device: looked up once
// per device, with that device current, and kept.
cudaError_t noalloc_scratch(u64 **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceState &d = g_dev[dev];
  u64 *p = d.noalloc_scratch.load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(d.mu);
    p = d.noalloc_scratch.load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_scratch);
      if (e != cudaSuccess || !p) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      d.noalloc_scratch.store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return cudaSuccess;
}

int columns_of(const kvcs_cache *caches, int32_t num_caches) {
  int m = 0;
  for (int32_t i = 0; caches && i < num_caches; ++i) m = std::max(m, caches[i].column + 1);
  return std::max(1, m);
}

}  // namespace
}  // namespace kvcs

using namespace kvcs;

extern "C" {

int kvcs_plan_requests(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
                       int64_t total_positions, int64_t num_requests, int32_t num_sms,
                       kvcs_plan_info *info) {
  if (!info || total_positions < 0) return KVCS_EINVAL;
  int rc = validate_caches(caches, num_caches, block_size, columns_of(caches, num_caches));
  if (rc != KVCS_OK) return rc;
  int sms = num_sms;
  if (sms <= 0) {
    if (device_setup(&sms) != cudaSuccess) return KVCS_ECUDA;
  }
  const std::vector<kvcs_cache> sorted = by_column(caches, num_caches);
  const Plan pl = make_plan(sorted, block_size, total_positions, sms, false, false,
                            num_requests);
  std::memset(info, 0, sizeof(*info));
  int n_slots = 0, n_other = 0, max_ipp = 0;
  for (const Launch &l : pl.launches) {
    if (l.kernel != kKernelSlots) {
      ++n_other;
      continue;
    }
    ++n_slots;
    int ipp = 0;
    for (const kvcs_cache &c : l.caches) ipp += c.layout == KVCS_LAYOUT_LATENT ? 1 : 2;
    max_ipp = std::max(max_ipp, ipp);
  }
  info->slot_launches = total_positions > 0 ? n_slots : 0;
  info->launches = total_positions > 0 ? static_cast<int32_t>(pl.launches.size()) : 0;
  info->memsets = pl.memset ? 1 : 0;
  info->kv_bytes_max = pl.kv_bytes_max;
  if (n_slots > 0 && n_other == 0) {
    // every launch on the valid-slot kernel
    const long long pages = total_positions * max_ipp;
    info->kernel = 3;
    const long long g0 = slots_grid(pages, sms);
    const long long wg = slots_window_groups(g0, sms);
    info->grid = static_cast<int32_t>(g0 * wg);
    info->threads = kSlotsThreads;
    info->units = pages;
    info->dynamic = total_positions > 0 && wg == 1 && slots_dynamic(pages, g0) ? 1 : 0;
    return KVCS_OK;
  }
  info->kernel = pl.kernel;
  info->split = pl.kernel != 1 ? pl.split : 0;
  info->grid = pl.kernel == 1 ? pl.generic_grid : pl.bulk_grid;
  info->threads = pl.kernel != 1 ? kBulkThreads
                  : caches[0].layout == KVCS_LAYOUT_STATE ? kGenericThreads
                                                           : kDirectThreads;
  info->smem_bytes = pl.kernel != 1 ? bulk_smem_bytes(pl.stages, pl.stage_bytes) : 0;
  info->stage_bytes = pl.kernel != 1 ? pl.stage_bytes : 0;
  info->stages = pl.kernel != 1 ? pl.stages : 0;
  info->units = pl.kernel == 1 ? total_positions : pl.units;
  info->dynamic = total_positions > 0 &&
                  make_plan(sorted, block_size, total_positions, sms, false, true,
                            num_requests).dynamic ? 1 : 0;
  return KVCS_OK;
}

int kvcs_plan(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
              int64_t total_positions, int32_t num_sms, kvcs_plan_info *info) {
  return kvcs_plan_requests(caches, num_caches, block_size, total_positions, -1, num_sms, info);
}

int kvcs_block_checksums(const kvcs_cache *caches, int32_t num_caches,
                         int32_t block_size, const kvcs_requests *reqs,
                         int64_t total_positions, uint64_t *out,
                         uint32_t *status, void *stream) {
  kvcs_outputs o;
  std::memset(&o, 0, sizeof(o));
  o.num_columns = 1;
  o.values = out;
  return run_checksums(caches, num_caches, block_size, reqs, total_positions, &o,
                       status, static_cast<cudaStream_t>(stream));
}

int kvcs_group_checksums(const kvcs_cache *caches, int32_t num_caches,
                         int32_t block_size, const kvcs_requests *reqs,
                         int64_t total_positions, const kvcs_outputs *outs,
                         uint32_t *status, void *stream) {
  return run_checksums(caches, num_caches, block_size, reqs, total_positions, outs,
                       status, static_cast<cudaStream_t>(stream));
}

int kvcs_block_checksums_noalloc(const kvcs_cache *caches, int32_t num_caches,
                                 int32_t block_size, const kvcs_requests *reqs,
                                 int64_t total_positions, uint64_t *out,
                                 uint32_t *status, void *stream) {
  // arguments first, with no CUDA call, as in kvcs_block_checksums
  if (num_caches > KVCS_NOALLOC_MAX_CACHES) return KVCS_ETOOLARGE;
  int rc = validate_caches(caches, num_caches, block_size, 1);
  if (rc != KVCS_OK) return rc;
  if (!reqs || total_positions < 0 || reqs->num_requests < 0) return KVCS_EINVAL;
  if (total_positions == 0) return KVCS_OK;
  if (!out || reinterpret_cast<uintptr_t>(out) % 8 || !reqs->pos_offsets ||
      !reqs->first_position || !reqs->num_tokens || !reqs->block_ids)
    return KVCS_EINVAL;
  u64 *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return KVCS_ECUDA;
  kvcs_outputs o;
  std::memset(&o, 0, sizeof(o));
  o.num_columns = 1;
  o.flags = KVCS_OUT_WORKSPACE;
  o.values = out;
  o.workspace = reinterpret_cast<uint64_t *>(scratch);
  return run_checksums(caches, num_caches, block_size, reqs, total_positions, &o,
                       status, static_cast<cudaStream_t>(stream));
}

int kvcs_block_checksum_tags(const void *block_hashes, int64_t hash_stride,
                             int64_t n, uint64_t fingerprint, uint64_t *tags,
                             void *stream) {
  if (n < 0 || hash_stride < 8) return KVCS_EINVAL;
  if (n == 0) return KVCS_OK;
  if (!block_hashes || !tags || reinterpret_cast<uintptr_t>(tags) % 8) return KVCS_EINVAL;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return KVCS_ECUDA;
  const long long blocks = std::min<long long>((n + 255) / 256, 4LL * sms);
  kvcs_tags_kernel<<<static_cast<unsigned>(std::max<long long>(1, blocks)), 256, 0,
                     static_cast<cudaStream_t>(stream)>>>(
      static_cast<const unsigned char *>(block_hashes), hash_stride, n, fingerprint,
      reinterpret_cast<u64 *>(tags));
  if (cudaGetLastError() != cudaSuccess) return KVCS_ECUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return KVCS_OK;
}

int kvcs_write_kv(const kvcs_cache *caches, int32_t num_caches, int32_t block_size,
                  int64_t num_tokens, const void *const *keys,
                  const void *const *values, const int64_t *slot_mapping,
                  const int64_t *positions, uint64_t *block_sums, uint32_t *status,
                  void *stream) {
  if (!caches || num_caches < 1 || num_tokens < 0 || !keys || !values) return KVCS_EINVAL;
  std::vector<kvcs_cache> plain(caches, caches + num_caches);
  for (kvcs_cache &c : plain) c.column = 0;  // running words are per block
  int rc = validate_caches(plain.data(), num_caches, block_size, 1);
  if (rc != KVCS_OK) return rc;
  auto al = [](const void *ptr, uintptr_t a) { return reinterpret_cast<uintptr_t>(ptr) % a == 0; };
  bool a16 = true;
  long long min_nb = caches[0].num_blocks;
  for (int32_t k = 0; k < num_caches; ++k) {
    const kvcs_cache &c = caches[k];
    if (c.layout == KVCS_LAYOUT_STATE) return KVCS_EINVAL;  // states are not per token
    const bool latent = c.layout == KVCS_LAYOUT_LATENT;
    if (num_tokens > 0 && (!keys[k] || (latent ? values[k] != nullptr : values[k] == nullptr)))
      return KVCS_EINVAL;
    if (!al(keys[k], 8) || (values[k] && !al(values[k], 8))) return KVCS_EINVAL;
    // the kernel indexes a token's row with 32-bit offsets
    if (static_cast<long long>(c.num_heads) * c.head_bytes >= (1LL << 30))
      return KVCS_EUNSUPPORTED;
    min_nb = std::min<long long>(min_nb, c.num_blocks);
    // 16-byte moves when every address involved stays 16-byte aligned
    a16 = a16 && al(c.base, 16) && al(keys[k], 16) && (!values[k] || al(values[k], 16)) &&
          c.head_bytes % 16 == 0 && c.half_stride % 16 == 0 && c.block_stride % 16 == 0;
  }
  if (block_sums && !al(block_sums, 8)) return KVCS_EINVAL;
  if (num_tokens == 0) return KVCS_OK;
  if (!slot_mapping || !positions) return KVCS_EINVAL;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return KVCS_ECUDA;
  WriteParams w;
  std::memset(&w, 0, sizeof(w));
  w.slots = reinterpret_cast<const long long *>(slot_mapping);
  w.positions = reinterpret_cast<const long long *>(positions);
  w.block_sums = reinterpret_cast<u64 *>(block_sums);
  w.status = status;
  w.num_tokens = num_tokens;
  w.num_blocks = min_nb;
  w.block_size = block_size;
  w.chunk = a16 ? 16 : 8;
  // caches by layout family (NHD and latent share one), each family in
  // launches of at most kMaxWriteCaches caches
  const int families[3] = {KVCS_LAYOUT_NHD, KVCS_LAYOUT_HND, KVCS_LAYOUT_XSPLIT};
  auto family = [](int layout) {
    return layout == KVCS_LAYOUT_LATENT ? static_cast<int>(KVCS_LAYOUT_NHD) : layout;
  };
  // a warp per item; CTAs beyond the resident ones start as others retire
  const long long warps_per_cta = kWriteThreads / 32;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int fam : families) {
    std::vector<int32_t> members;
    for (int32_t k = 0; k < num_caches; ++k)
      if (family(caches[k].layout) == fam) members.push_back(k);
    for (size_t lo = 0; lo < members.size(); lo += kMaxWriteCaches) {
      const int n = static_cast<int>(std::min<size_t>(kMaxWriteCaches, members.size() - lo));
      w.num_caches = n;
      for (int k = 0; k < n; ++k) {
        const int32_t m = members[lo + k];
        w.c[k] = make_dev_cache(caches[m], block_size);
        w.key[k] = static_cast<const unsigned char *>(keys[m]);
        w.value[k] = static_cast<const unsigned char *>(values[m]);
      }
      // enough (token, run of caches) items for about 64 warps per SM
      const long long want = 64LL * sms;
      const long long runs = std::min<long long>(n, std::max<long long>(
                                                        1, (want + num_tokens - 1) / num_tokens));
      w.caches_per_item = static_cast<int>((n + runs - 1) / runs);
      const long long witems = num_tokens * ((n + w.caches_per_item - 1) / w.caches_per_item);
      const unsigned grid = static_cast<unsigned>(std::max<long long>(
          1, std::min<long long>((witems + warps_per_cta - 1) / warps_per_cta, 32LL * sms)));
      // x-split: a warp per (cache, 32 tokens, run of heads) item, the runs
      // short enough for about 64 warps per SM
      int max_heads = 1;
      for (int k = 0; k < n; ++k) max_heads = std::max(max_heads, w.c[k].heads);
      const long long xbase = (num_tokens + 31) / 32 * n;
      const long long xruns = std::min<long long>(
          max_heads, std::max<long long>(1, (want + xbase - 1) / xbase));
      w.heads_per_item = static_cast<int>((max_heads + xruns - 1) / xruns);
      w.head_chunks = (max_heads + w.heads_per_item - 1) / w.heads_per_item;
      const unsigned xgrid = static_cast<unsigned>(std::max<long long>(
          1, std::min<long long>((xbase * w.head_chunks + warps_per_cta - 1) / warps_per_cta,
                                 32LL * sms)));
      cudaError_t e;
      if (fam == KVCS_LAYOUT_HND)
        e = launch_write(kvcs_write_kernel<kLayoutHND>, grid, st, w);
      else if (fam == KVCS_LAYOUT_XSPLIT)
        e = launch_write(kvcs_write_xsplit_kernel, xgrid, st, w);
      else
        e = launch_write(kvcs_write_kernel<kLayoutNHD>, grid, st, w);
      if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return KVCS_ECUDA;
      g_launches.fetch_add(1, std::memory_order_relaxed);
    }
  }
  return KVCS_OK;
}

int kvcs_selftest_wait_timeout(uint32_t *status, int64_t limit_ns, void *stream) {
  if (!status || limit_ns <= 0 || limit_ns > 2000000000LL) return KVCS_EINVAL;
  kvcs_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, static_cast<u64>(limit_ns));
  if (cudaGetLastError() != cudaSuccess) return KVCS_ECUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return KVCS_OK;
}

const char *kvcs_strerror(int code) {
  switch (code) {
    case KVCS_OK: return "success";
    case KVCS_EINVAL: return "invalid argument";
    case KVCS_EUNSUPPORTED:
      return "unsupported geometry (global heads past 65536 per layer, or a token row of 1 GiB "
             "or more in a write)";
    case KVCS_ECUDA: return "CUDA error";
    case KVCS_ETOOLARGE:
      return "beyond the fixed limit of kvcs_block_checksums_noalloc (more than "
             "KVCS_NOALLOC_MAX_CACHES = 1024 caches)";
    default: return "unknown error";
  }
}

uint64_t kvcs_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t kvcs_version(void) { return (1 << 16) | 4; }

}  // extern "C"
