/*
 * Scalar C oracle for the connector-agnostic KV-cache block checksum.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never includes, links or
 * calls this file; only the tests, the smoke check and the CPU-baseline legs
 * of the benchmark do, through oracle/c_oracle.py.  It shares no header,
 * helper or table with the CUDA library.
 *
 * Source: the page "vllm.distributed.kv_transfer.kv_checksum.checksum"
 * (vLLM API docs), module docstring item 1 (slice checksum
 * s = sum_j x_j*(2j+1) mod 2^64 with j = t*P + p) and item 2 (block checksum
 * c = sum m*s mod 2^64, m = 2*(layer*H + head) + 1, H = 1 << 16), the
 * dataclass KVChecksumBlocks (slots at or past num_tokens are skipped) and
 * the function num_valid_tokens.
 *
 * It computes the same thing as oracle/kvcs_oracle.py, in the same order
 * (slice checksums first, then the factor-weighted block sum), with plain
 * loops over logical indices (position, cache, head, slot, piece).  Pieces are
 * assembled byte by byte so host endianness does not matter.  The only
 * addition is that positions are shared out over POSIX threads; positions are
 * independent, so this changes no arithmetic.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_LAYOUT_NHD 0    /* pool [2][num_blocks][block_size][heads][head_bytes] */
#define ORACLE_LAYOUT_HND 1    /* pool [2][num_blocks][heads][block_size][head_bytes], or
                                  [2][num_blocks][block_size/kbs][heads][kbs][head_bytes] */
#define ORACLE_LAYOUT_LATENT 2 /* pool [num_blocks][block_size][row_bytes] */
#define ORACLE_LAYOUT_XSPLIT 3 /* pool [2][num_blocks][heads][head_bytes/16][block_size][16] */
#define ORACLE_LAYOUT_STATE 4  /* pool [num_blocks][rows][row_bytes]: Mamba state */

#define ORACLE_H 65536u /* MAX_KV_HEADS_PER_LAYER */
#define ORACLE_STATUS_BAD_BLOCK_ID 1u

typedef struct oracle_cache {
  const uint8_t *data; /* host bytes of the whole pool */
  int64_t data_bytes;  /* how many bytes `data` holds */
  int64_t num_blocks;
  int32_t layout;
  int32_t layer;
  int32_t head_offset;
  int32_t num_heads;
  int32_t head_bytes; /* K (= V) bytes per head per token; latent/state: row bytes */
  int32_t piece_bytes; /* state: element bytes (2 or 4); else ignored (8) */
  int32_t kernel_block_size; /* HND: slots per kernel sub-block; 0: none */
  int64_t half_stride;  /* bytes from a block's K page to its V page; 0: packed */
  int64_t block_stride; /* bytes between blocks' pages; 0: packed */
} oracle_cache;

/* Tokens of the request's first num_tokens that block `position` holds. */
static int64_t num_valid_tokens(int64_t position, int64_t block_size,
                                int64_t num_tokens) {
  int64_t first = position * block_size;
  if (num_tokens <= first) return 0;
  if (num_tokens - first >= block_size) return block_size;
  return num_tokens - first;
}

static int64_t pieces_per_token(const oracle_cache *c) {
  if (c->layout == ORACLE_LAYOUT_LATENT) return c->head_bytes / 8;
  return 2 * (int64_t)c->head_bytes / 8; /* K bytes then V bytes */
}

/* Piece p (little-endian u64) of slot `slot`'s slice for local head `head`. */
static uint64_t piece_at(const oracle_cache *c, int64_t block_size,
                         int64_t block, int64_t slot, int64_t head,
                         int64_t p) {
  int64_t hb = c->head_bytes;
  int64_t byte = 8 * p;
  int64_t kv = 0;
  if (c->layout != ORACLE_LAYOUT_LATENT && byte >= hb) {
    kv = 1;
    byte -= hb;
  }
  /* the page of (kv, block); explicit strides place it anywhere in the pool */
  int64_t page_bytes = block_size * c->num_heads * hb;
  int64_t half = c->half_stride ? c->half_stride : c->num_blocks * page_bytes;
  int64_t stride = c->block_stride ? c->block_stride : page_bytes;
  int64_t off = kv * half + block * stride;
  if (c->layout == ORACLE_LAYOUT_LATENT) {
    off += slot * hb + byte;
  } else if (c->layout == ORACLE_LAYOUT_NHD) {
    off += (slot * c->num_heads + head) * hb + byte;
  } else if (c->layout == ORACLE_LAYOUT_XSPLIT) {
    /* x elements make 16 bytes: [heads][head_bytes/16][block_size][16] */
    off += ((head * (hb / 16) + byte / 16) * block_size + slot) * 16 + byte % 16;
  } else {
    int64_t kbs = c->kernel_block_size > 0 ? c->kernel_block_size : block_size;
    off += ((slot / kbs * c->num_heads + head) * kbs + slot % kbs) * hb + byte;
  }
  uint64_t x = 0;
  for (int k = 0; k < 8; ++k) x |= (uint64_t)c->data[off + k] << (8 * k);
  return x;
}

/* s = sum_j x_j * (2j + 1) mod 2^64 over the first nv slots (item 1). */
static uint64_t slice_checksum(const oracle_cache *c, int64_t block_size,
                               int64_t block, int64_t position, int64_t nv,
                               int64_t head) {
  uint64_t P = (uint64_t)pieces_per_token(c);
  uint64_t s = 0;
  for (int64_t slot = 0; slot < nv; ++slot) {
    uint64_t t = (uint64_t)position * (uint64_t)block_size + (uint64_t)slot;
    for (uint64_t p = 0; p < P; ++p) {
      uint64_t j = t * P + p;
      s += piece_at(c, block_size, block, slot, head, (int64_t)p) * (2 * j + 1);
    }
  }
  return s;
}

/* Element p (little-endian, unsigned) of local row `row` of a state block. */
static uint64_t state_piece(const oracle_cache *c, int64_t block, int64_t row,
                            int64_t p) {
  int64_t stride = c->block_stride ? c->block_stride : (int64_t)c->num_heads * c->head_bytes;
  int64_t off = block * stride + row * c->head_bytes + p * c->piece_bytes;
  uint64_t x = 0;
  for (int k = 0; k < c->piece_bytes; ++k) x |= (uint64_t)c->data[off + k] << (8 * k);
  return x;
}

/* s of one global row of a Mamba state (paragraph on Mamba state): its
 * elements are the pieces and the piece index is the element index. */
static uint64_t state_slice_checksum(const oracle_cache *c, int64_t block,
                                     int64_t row) {
  uint64_t s = 0;
  int64_t n = c->head_bytes / c->piece_bytes;
  for (int64_t p = 0; p < n; ++p)
    s += state_piece(c, block, row, p) * (2 * (uint64_t)p + 1);
  return s;
}

/* m = 2 * (layer * H + head) + 1 (item 2). */
static uint64_t slice_factor(int64_t layer, int64_t global_head) {
  return 2 * ((uint64_t)layer * ORACLE_H + (uint64_t)global_head) + 1;
}

/* c = sum_{layer, head} m * s mod 2^64 (item 2). */
static uint64_t block_checksum(const oracle_cache *caches, int32_t num_caches,
                               int64_t block_size, int64_t block,
                               int64_t position, int64_t num_tokens) {
  int64_t nv = num_valid_tokens(position, block_size, num_tokens);
  uint64_t c = 0;
  for (int32_t k = 0; k < num_caches; ++k) {
    const oracle_cache *ca = &caches[k];
    if (ca->layout == ORACLE_LAYOUT_STATE) {
      /* a state block lives at position 0 only; its rows are its slices */
      if (position != 0) continue;
      for (int64_t r = 0; r < ca->num_heads; ++r)
        c += slice_factor(ca->layer, (int64_t)ca->head_offset + r) *
             state_slice_checksum(ca, block, r);
      continue;
    }
    for (int64_t h = 0; h < ca->num_heads; ++h) {
      uint64_t s = slice_checksum(ca, block_size, block, position, nv, h);
      c += slice_factor(ca->layer, (int64_t)ca->head_offset + h) * s;
    }
  }
  return c;
}

typedef struct job {
  const oracle_cache *caches;
  int32_t num_caches;
  int64_t block_size;
  int64_t num_requests;
  const int64_t *pos_offsets;
  const int64_t *first_position;
  const int64_t *num_tokens;
  const int32_t *block_ids;
  uint64_t *out;
  int64_t begin, end; /* global position indices of this thread */
  uint32_t status;
} job;

static void *run_job(void *arg) {
  job *jb = (job *)arg;
  /* request holding position index jb->begin */
  int64_t r = 0;
  while (r < jb->num_requests && jb->pos_offsets[r + 1] <= jb->begin) ++r;
  for (int64_t i = jb->begin; i < jb->end; ++i) {
    while (jb->pos_offsets[r + 1] <= i) ++r;
    int64_t position = jb->first_position[r] + (i - jb->pos_offsets[r]);
    int64_t block = jb->block_ids[i];
    int bad = 0;
    for (int32_t k = 0; k < jb->num_caches; ++k)
      if (block < 0 || block >= jb->caches[k].num_blocks) bad = 1;
    if (bad) {
      jb->out[i] = 0;
      jb->status |= ORACLE_STATUS_BAD_BLOCK_ID;
      continue;
    }
    jb->out[i] = block_checksum(jb->caches, jb->num_caches, jb->block_size,
                                block, position, jb->num_tokens[r]);
  }
  return NULL;
}

/* Bytes the pool must hold for every page its geometry addresses: up to the
 * end of the last block's last page (state: the last block's rows). */
static int64_t pool_bytes_needed(const oracle_cache *c, int64_t block_size) {
  if (c->num_blocks == 0) return 0;
  if (c->layout == ORACLE_LAYOUT_STATE) {
    int64_t state = (int64_t)c->num_heads * c->head_bytes;
    int64_t stride = c->block_stride ? c->block_stride : state;
    return (c->num_blocks - 1) * stride + state;
  }
  int64_t page_bytes = block_size * c->num_heads * (int64_t)c->head_bytes;
  int64_t half = c->half_stride ? c->half_stride : c->num_blocks * page_bytes;
  int64_t stride = c->block_stride ? c->block_stride : page_bytes;
  int64_t last_half = c->layout == ORACLE_LAYOUT_LATENT ? 0 : 1;
  return last_half * half + (c->num_blocks - 1) * stride + page_bytes;
}

/*
 * One uint64 per global position index into out[pos_offsets[num_requests]].
 * Returns 0, or -1 for arguments the definition does not cover or a pool
 * smaller than its declared geometry.  *status gets
 * ORACLE_STATUS_BAD_BLOCK_ID if some position's block id is outside
 * [0, num_blocks) of some cache (that position's output is 0).
 * num_threads <= 0 means one thread.
 */
int oracle_block_checksums(const oracle_cache *caches, int32_t num_caches,
                           int32_t block_size, int64_t num_requests,
                           const int64_t *pos_offsets,
                           const int64_t *first_position,
                           const int64_t *num_tokens,
                           const int32_t *block_ids, uint64_t *out,
                           uint32_t *status, int32_t num_threads) {
  if (block_size <= 0 || num_caches < 0 || num_requests < 0 || !pos_offsets)
    return -1;
  for (int32_t k = 0; k < num_caches; ++k) {
    const oracle_cache *c = &caches[k];
    if (c->num_blocks < 0 || c->data_bytes < 0 || (c->data_bytes > 0 && !c->data))
      return -1;
    if (c->layout == ORACLE_LAYOUT_STATE) {
      if ((c->piece_bytes != 2 && c->piece_bytes != 4) || c->head_bytes <= 0 ||
          c->head_bytes % c->piece_bytes || c->num_heads < 1 || c->head_offset < 0 ||
          (int64_t)c->head_offset + c->num_heads > (int64_t)ORACLE_H || c->block_stride < 0)
        return -1;
      if (pool_bytes_needed(c, block_size) > c->data_bytes) return -1;
      continue;
    }
    if (c->head_bytes <= 0 || c->head_bytes % 8 || c->num_heads < 1 ||
        c->head_offset < 0 ||
        (int64_t)c->head_offset + c->num_heads > (int64_t)ORACLE_H)
      return -1;
    if (c->layout == ORACLE_LAYOUT_LATENT && c->num_heads != 1) return -1;
    if (c->layout < 0 || c->layout > 3) return -1;
    if (c->half_stride < 0 || c->block_stride < 0) return -1;
    if (c->layout == ORACLE_LAYOUT_XSPLIT && c->head_bytes % 16) return -1;
    if (c->kernel_block_size != 0 &&
        (c->layout != ORACLE_LAYOUT_HND || c->kernel_block_size < 0 ||
         block_size % c->kernel_block_size))
      return -1;
    if (pool_bytes_needed(c, block_size) > c->data_bytes) return -1;
  }
  if (pos_offsets[0] != 0) return -1;
  for (int64_t r = 0; r < num_requests; ++r)
    if (pos_offsets[r + 1] < pos_offsets[r]) return -1;
  int64_t total = pos_offsets[num_requests];
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 1024) num_threads = 1024;
  if ((int64_t)num_threads > total) num_threads = total > 0 ? (int32_t)total : 1;

  job *jobs = (job *)calloc((size_t)num_threads, sizeof(job));
  pthread_t *tids = (pthread_t *)calloc((size_t)num_threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -1;
  }
  for (int32_t w = 0; w < num_threads; ++w) {
    job *jb = &jobs[w];
    jb->caches = caches;
    jb->num_caches = num_caches;
    jb->block_size = block_size;
    jb->num_requests = num_requests;
    jb->pos_offsets = pos_offsets;
    jb->first_position = first_position;
    jb->num_tokens = num_tokens;
    jb->block_ids = block_ids;
    jb->out = out;
    jb->begin = total * w / num_threads;
    jb->end = total * (w + 1) / num_threads;
    jb->status = 0;
  }
  int32_t started = 0;
  for (int32_t w = 1; w < num_threads; ++w) {
    if (pthread_create(&tids[w], NULL, run_job, &jobs[w]) != 0) break;
    started = w;
  }
  run_job(&jobs[0]);
  for (int32_t w = started + 1; w < num_threads; ++w) run_job(&jobs[w]);
  for (int32_t w = 1; w <= started; ++w) pthread_join(tids[w], NULL);
  uint32_t st = 0;
  for (int32_t w = 0; w < num_threads; ++w) st |= jobs[w].status;
  if (status) *status |= st;
  free(jobs);
  free(tids);
  return 0;
}
