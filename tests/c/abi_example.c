/*
 * abi_example.c -- the C ABI used from plain C (no Python, no torch): write
 * 64 tokens into a 2 x 64 x 352 nvfp4_ds_mla cache, gather 40 rows back, and
 * compare both with the CPU oracle linked beside it.  Exit status 0 on a
 * bit-exact match.  Built and run by tests/test_c_abi.py on a GPU host.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_oracle.h"

#define T 64
#define NB 2
#define BS 64
#define CHECK(x)                                                          \
  do {                                                                    \
    cudaError_t e_ = (x);                                                 \
    if (e_ != cudaSuccess) {                                              \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
      return 2;                                                           \
    }                                                                     \
  } while (0)

static uint32_t lcg = 12345u;
static uint16_t rand_bf16(void) {       /* finite bf16 values of modest magnitude */
  lcg = lcg * 1664525u + 1013904223u;
  uint16_t sign = (uint16_t)((lcg >> 31) << 15);
  uint16_t exp = (uint16_t)(120 + ((lcg >> 20) % 12));  /* 2^-7 .. 2^4 */
  uint16_t man = (uint16_t)((lcg >> 8) & 0x7F);
  return (uint16_t)(sign | (exp << 7) | man);
}

int main(void) {
  static uint16_t kv_c[T * 512], k_pe[T * 64];
  static int64_t slots[T];
  static uint8_t cache[NB * BS * 352], want_cache[NB * BS * 352];
  static uint16_t rows[40 * 576], want_rows[40 * 576];
  const int32_t table[2] = {1, 0}, ws[1] = {0}, starts[1] = {5};
  int i;
  for (i = 0; i < T * 512; ++i) kv_c[i] = rand_bf16();
  for (i = 0; i < T * 64; ++i) k_pe[i] = rand_bf16();
  for (i = 0; i < T; ++i) slots[i] = (i % 9 == 4) ? -1 : (int64_t)((i * 37) % (NB * BS));
  memset(want_cache, 0, sizeof want_cache);
  kvqo_write_nvfp4_ds_mla(kv_c, 512, k_pe, 64, slots, 0, T, want_cache, NB, BS, BS * 352, 352);
  memset(want_rows, 0, sizeof want_rows);
  kvqo_gather_nvfp4_ds_mla(want_cache, NB, BS, BS * 352, 352, want_rows, 576, 40, table, 2, 2, ws, starts, 1,
                           NULL, 40);

  void *d_kv, *d_pe, *d_slots, *d_cache, *d_rows, *d_table, *d_ws, *d_starts, *d_status;
  CHECK(cudaMalloc(&d_kv, sizeof kv_c));
  CHECK(cudaMalloc(&d_pe, sizeof k_pe));
  CHECK(cudaMalloc(&d_slots, sizeof slots));
  CHECK(cudaMalloc(&d_cache, sizeof cache));
  CHECK(cudaMalloc(&d_rows, sizeof rows));
  CHECK(cudaMalloc(&d_table, sizeof table));
  CHECK(cudaMalloc(&d_ws, sizeof ws));
  CHECK(cudaMalloc(&d_starts, sizeof starts));
  CHECK(cudaMalloc(&d_status, sizeof(int32_t)));
  CHECK(cudaMemcpy(d_kv, kv_c, sizeof kv_c, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_pe, k_pe, sizeof k_pe, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_slots, slots, sizeof slots, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_ws, ws, sizeof ws, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_starts, starts, sizeof starts, cudaMemcpyHostToDevice));
  CHECK(cudaMemset(d_cache, 0, sizeof cache));
  CHECK(cudaMemset(d_rows, 0, sizeof rows));
  CHECK(cudaMemset(d_status, 0, sizeof(int32_t)));

  kvq_status st = kvq_write_nvfp4_ds_mla(d_kv, 512, d_pe, 64, (const int64_t*)d_slots, T, (uint8_t*)d_cache,
                                         NB, BS, BS * 352, 352, (int32_t*)d_status, NULL);
  if (st != KVQ_OK) { fprintf(stderr, "write: %s\n", kvq_last_error_string()); return 3; }
  st = kvq_gather_upconvert_nvfp4_ds_mla((const uint8_t*)d_cache, NB, BS, BS * 352, 352, d_rows, 576, 40,
                                         (const int32_t*)d_table, 2, 2, (const int32_t*)d_ws,
                                         (const int32_t*)d_starts, 1, (int32_t*)d_status, NULL);
  if (st != KVQ_OK) { fprintf(stderr, "gather: %s\n", kvq_last_error_string()); return 3; }
  /* a host-side argument error: misaligned cache, nothing launched */
  st = kvq_write_nvfp4_ds_mla(d_kv, 512, d_pe, 64, (const int64_t*)d_slots, T, (uint8_t*)d_cache + 4, NB, BS,
                              BS * 352, 352, NULL, NULL);
  if (st != KVQ_ERR_INVALID_ARG) { fprintf(stderr, "expected KVQ_ERR_INVALID_ARG, got %d\n", st); return 4; }

  int32_t status = -1;
  CHECK(cudaMemcpy(cache, d_cache, sizeof cache, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(rows, d_rows, sizeof rows, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(&status, d_status, sizeof status, cudaMemcpyDeviceToHost));
  if (status != 0) { fprintf(stderr, "device status %d\n", status); return 5; }
  if (memcmp(cache, want_cache, sizeof cache) != 0) { fprintf(stderr, "cache differs\n"); return 6; }
  if (memcmp(rows, want_rows, sizeof rows) != 0) { fprintf(stderr, "rows differ\n"); return 7; }
  printf("C ABI: write (64 tokens) and gather (40 rows) match the oracle bit for bit\n");
  return 0;
}
