/*
 * The library used from plain C through include/kvcs.h alone: no Python, no
 * torch.  Two NHD layers whose every 8-byte piece is 1, one request of 37
 * tokens in three 16-slot blocks at shuffled block ids.  With x_j = 1 the
 * slice sum over tokens [t0, t1) is sum_j (2j + 1) = (t1 P)^2 - (t0 P)^2, so
 * each block position's checksum has the closed form
 *   c = (t1^2 - t0^2) P^2 * sum_{layer, head} (2 (layer * 65536 + head) + 1)
 * mod 2^64, with t0 = position * 16 and t1 = min(t0 + 16, 37).  The program
 * also checks that bad arguments are refused before any CUDA work, that an
 * out-of-pool block id is flagged in the status word, and that writing the
 * same tokens into empty pools with kvcs_write_kv leaves each block's
 * running word at the same closed form.
 *
 * Build: nvcc -o c_abi_example c_abi_example.c -I<repo>/include -L<lib dir>
 *        -lkvcs -Xlinker -rpath,<lib dir>
 * Exit status 0 when every check passes.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvcs.h"

#define CHECK(cond, msg)                       \
  do {                                         \
    if (!(cond)) {                             \
      fprintf(stderr, "FAILED: %s\n", msg);    \
      return 1;                                \
    }                                          \
  } while (0)

int main(void) {
  const int layers = 2, heads = 2, head_bytes = 32, bs = 16, nb = 5;
  const int64_t ntok = 37;
  const uint64_t P = 2 * (uint64_t)head_bytes / 8;
  const size_t pool_bytes = (size_t)2 * nb * bs * heads * head_bytes;

  /* host pool: every little-endian 8-byte piece equals 1 */
  uint8_t *host = (uint8_t *)calloc(pool_bytes, 1);
  CHECK(host != NULL, "host allocation");
  for (size_t i = 0; i < pool_bytes; i += 8) host[i] = 1;

  void *pools[2];
  kvcs_cache caches[2];
  memset(caches, 0, sizeof(caches));
  for (int l = 0; l < layers; ++l) {
    CHECK(cudaMalloc(&pools[l], pool_bytes) == cudaSuccess, "cudaMalloc pool");
    CHECK(cudaMemcpy(pools[l], host, pool_bytes, cudaMemcpyHostToDevice) == cudaSuccess,
          "copy pool");
    caches[l].base = pools[l];
    caches[l].num_blocks = nb;
    caches[l].layout = KVCS_LAYOUT_NHD;
    caches[l].layer = l;
    caches[l].head_offset = 0;
    caches[l].num_heads = heads;
    caches[l].head_bytes = head_bytes;
  }

  /* one request, three block positions on blocks 3, 0, 4 */
  const int64_t h_po[2] = {0, 3}, h_fp[1] = {0}, h_nt[1] = {ntok};
  const int32_t h_ids[3] = {3, 0, 4};
  int64_t *d_po, *d_fp, *d_nt;
  int32_t *d_ids;
  uint64_t *d_out;
  uint32_t *d_status;
  CHECK(cudaMalloc((void **)&d_po, sizeof(h_po)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_fp, sizeof(h_fp)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_nt, sizeof(h_nt)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_ids, sizeof(h_ids)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_out, 3 * sizeof(uint64_t)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_status, sizeof(uint32_t)) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(d_po, h_po, sizeof(h_po), cudaMemcpyHostToDevice);
  cudaMemcpy(d_fp, h_fp, sizeof(h_fp), cudaMemcpyHostToDevice);
  cudaMemcpy(d_nt, h_nt, sizeof(h_nt), cudaMemcpyHostToDevice);
  cudaMemcpy(d_ids, h_ids, sizeof(h_ids), cudaMemcpyHostToDevice);
  cudaMemset(d_status, 0, sizeof(uint32_t));

  kvcs_requests reqs = {1, d_po, d_fp, d_nt, d_ids};

  /* bad arguments are refused before any CUDA work */
  CHECK(kvcs_block_checksums(NULL, 2, bs, &reqs, 3, d_out, d_status, NULL) == KVCS_EINVAL,
        "null caches refused");
  CHECK(kvcs_block_checksums(caches, 2, 0, &reqs, 3, d_out, d_status, NULL) == KVCS_EINVAL,
        "zero block_size refused");
  CHECK(kvcs_strerror(KVCS_EINVAL) != NULL, "strerror");

  int rc = kvcs_block_checksums(caches, layers, bs, &reqs, 3, d_out, d_status, NULL);
  CHECK(rc == KVCS_OK, "kvcs_block_checksums");
  uint64_t out[3];
  uint32_t status = 0;
  CHECK(cudaMemcpy(out, d_out, sizeof(out), cudaMemcpyDeviceToHost) == cudaSuccess,
        "copy out");
  CHECK(cudaMemcpy(&status, d_status, sizeof(status), cudaMemcpyDeviceToHost) ==
            cudaSuccess,
        "copy status");
  CHECK(status == 0, "status clear");

  uint64_t msum = 0;
  for (int l = 0; l < layers; ++l)
    for (int h = 0; h < heads; ++h) msum += 2 * ((uint64_t)l * 65536u + (uint64_t)h) + 1;
  for (int q = 0; q < 3; ++q) {
    const uint64_t t0 = (uint64_t)q * bs;
    const uint64_t t1 = t0 + bs < (uint64_t)ntok ? t0 + bs : (uint64_t)ntok;
    const uint64_t expect = (t1 * t1 - t0 * t0) * P * P * msum;
    if (out[q] != expect) {
      fprintf(stderr, "FAILED: position %d: %llu, closed form %llu\n", q,
              (unsigned long long)out[q], (unsigned long long)expect);
      return 1;
    }
  }

  /* a block id past the pool: that position reads 0 and the status says so */
  const int32_t bad_ids[3] = {3, 9, 4};
  cudaMemcpy(d_ids, bad_ids, sizeof(bad_ids), cudaMemcpyHostToDevice);
  rc = kvcs_block_checksums(caches, layers, bs, &reqs, 3, d_out, d_status, NULL);
  CHECK(rc == KVCS_OK, "second call");
  cudaMemcpy(out, d_out, sizeof(out), cudaMemcpyDeviceToHost);
  cudaMemcpy(&status, d_status, sizeof(status), cudaMemcpyDeviceToHost);
  CHECK(status & KVCS_STATUS_BAD_BLOCK_ID, "bad block id flagged");
  CHECK(out[1] == 0, "bad position reads 0");

  /* the fused write: the same 37 tokens (all pieces 1) into empty pools;
   * every written block's running word must be the same closed form */
  void *empty[2], *keys[2], *vals[2];
  const size_t tok_bytes = (size_t)ntok * heads * head_bytes;
  uint8_t *host_tok = (uint8_t *)calloc(tok_bytes, 1);
  CHECK(host_tok != NULL, "host allocation");
  for (size_t i = 0; i < tok_bytes; i += 8) host_tok[i] = 1;
  kvcs_cache wcaches[2];
  memcpy(wcaches, caches, sizeof(caches));
  for (int l = 0; l < layers; ++l) {
    CHECK(cudaMalloc(&empty[l], pool_bytes) == cudaSuccess, "cudaMalloc pool");
    cudaMemset(empty[l], 0, pool_bytes);
    CHECK(cudaMalloc(&keys[l], tok_bytes) == cudaSuccess, "cudaMalloc keys");
    CHECK(cudaMalloc(&vals[l], tok_bytes) == cudaSuccess, "cudaMalloc values");
    cudaMemcpy(keys[l], host_tok, tok_bytes, cudaMemcpyHostToDevice);
    cudaMemcpy(vals[l], host_tok, tok_bytes, cudaMemcpyHostToDevice);
    wcaches[l].base = empty[l];
  }
  int64_t h_slots[37], h_pos[37];
  for (int t = 0; t < ntok; ++t) {
    h_slots[t] = (int64_t)h_ids[t / bs] * bs + t % bs;
    h_pos[t] = t;
  }
  int64_t *d_slots, *d_pos;
  uint64_t *d_sums;
  CHECK(cudaMalloc((void **)&d_slots, sizeof(h_slots)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_pos, sizeof(h_pos)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void **)&d_sums, nb * sizeof(uint64_t)) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(d_slots, h_slots, sizeof(h_slots), cudaMemcpyHostToDevice);
  cudaMemcpy(d_pos, h_pos, sizeof(h_pos), cudaMemcpyHostToDevice);
  cudaMemset(d_sums, 0, nb * sizeof(uint64_t));
  cudaMemset(d_status, 0, sizeof(uint32_t));
  rc = kvcs_write_kv(wcaches, layers, bs, ntok, (const void *const *)keys,
                     (const void *const *)vals, d_slots, d_pos, d_sums, d_status, NULL);
  CHECK(rc == KVCS_OK, "kvcs_write_kv");
  uint64_t sums[5];
  cudaMemcpy(sums, d_sums, sizeof(sums), cudaMemcpyDeviceToHost);
  cudaMemcpy(&status, d_status, sizeof(status), cudaMemcpyDeviceToHost);
  CHECK(status == 0, "write status clear");
  for (int q = 0; q < 3; ++q) {
    const uint64_t t0 = (uint64_t)q * bs;
    const uint64_t t1 = t0 + bs < (uint64_t)ntok ? t0 + bs : (uint64_t)ntok;
    CHECK(sums[h_ids[q]] == (t1 * t1 - t0 * t0) * P * P * msum, "running word = closed form");
  }
  CHECK(sums[1] == 0 && sums[2] == 0, "unwritten blocks stay 0");

  printf("c abi ok: 3 block checksums and 3 fused-write block words equal the closed form "
         "(version %d.%d)\n", kvcs_version() >> 16, kvcs_version() & 0xffff);
  for (int l = 0; l < layers; ++l) {
    cudaFree(empty[l]);
    cudaFree(keys[l]);
    cudaFree(vals[l]);
  }
  cudaFree(d_slots);
  cudaFree(d_pos);
  cudaFree(d_sums);
  free(host_tok);
  for (int l = 0; l < layers; ++l) cudaFree(pools[l]);
  cudaFree(d_po);
  cudaFree(d_fp);
  cudaFree(d_nt);
  cudaFree(d_ids);
  cudaFree(d_out);
  cudaFree(d_status);
  free(host);
  return 0;
}
