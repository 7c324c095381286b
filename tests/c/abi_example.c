/*
 * abi_example.c -- the C ABI used from plain C (no Python, no torch): write
 * 64 tokens into a 2 x 64 x 352 nvfp4_ds_mla cache, gather 40 rows back, run
 * the sparse MLA attention of 2 tokens x 16 heads over 48 of its slots, and
 * compare all three with the CPU oracle linked beside it (bit for bit for the
 * write and the gather, within the bound derived from the attention's
 * arithmetic for the attention).  Exit status 0 on success.  Built and run by
 * tests/test_c_abi.py on a GPU host.
 */
#include <math.h>
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

  /* attention: 2 tokens x 16 heads, 48 slots each (every 7th unused) */
  enum { AT = 2, AH = 16, AK = 48 };
  static uint16_t q[AT * AH * 576], o_bits[AT * AH * 512];
  static int32_t aidx[AT * AK];
  static float lse[AT * AH];
  static double want_o[AT * AH * 512], want_lse[AT * AH], keys[AK * 576];
  const float scale = 0.0416667f;
  for (i = 0; i < AT * AH * 576; ++i) q[i] = rand_bf16();
  for (i = 0; i < AT * AK; ++i) aidx[i] = (i % 7 == 3) ? -1 : (int32_t)((i * 29 + 3) % (NB * BS));
  kvqo_sparse_mla_attention_nvfp4_ds_mla(q, AH * 576, 576, 0, AT, AH, aidx, AK, AK, want_cache, NB, BS, BS * 352,
                                         352, scale, want_o, AH * 512, 512, want_lse, AH);
  void *d_q, *d_idx, *d_o, *d_lse;
  CHECK(cudaMalloc(&d_q, sizeof q));
  CHECK(cudaMalloc(&d_idx, sizeof aidx));
  CHECK(cudaMalloc(&d_o, sizeof o_bits));
  CHECK(cudaMalloc(&d_lse, sizeof lse));
  CHECK(cudaMemcpy(d_q, q, sizeof q, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(d_idx, aidx, sizeof aidx, cudaMemcpyHostToDevice));
  st = kvq_sparse_mla_attention_nvfp4_ds_mla(d_q, AH * 576, 576, AT, AH, (const int32_t*)d_idx, AK, AK,
                                             (const uint8_t*)d_cache, NB, BS, BS * 352, 352, scale, d_o,
                                             AH * 512, 512, (float*)d_lse, AH, (int32_t*)d_status, NULL);
  if (st != KVQ_OK) { fprintf(stderr, "attention: %s\n", kvq_last_error_string()); return 3; }
  CHECK(cudaMemcpy(o_bits, d_o, sizeof o_bits, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(lse, d_lse, sizeof lse, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(&status, d_status, sizeof status, cudaMemcpyDeviceToHost));
  if (status != 0) { fprintf(stderr, "attention device status %d\n", status); return 5; }
  for (int t = 0; t < AT; ++t) {
    int n = 0;
    double vmax = 0.0;
    for (int k = 0; k < AK; ++k) {
      const int32_t sl = aidx[t * AK + k];
      if (sl < 0) continue;
      kvqo_decode_nvfp4_ds_mla_entry(want_cache + (int64_t)sl * 352, keys + (int64_t)n * 576);
      for (int d = 0; d < 512; ++d) vmax = fmax(vmax, fabs(keys[(int64_t)n * 576 + d]));
      ++n;
    }
    for (int h = 0; h < AH; ++h) {
      /* the bound of the Python parity tests: score error e_s, weight error eps */
      double dmax = 0.0;
      for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < 576; ++d)
          acc += fabs((double)kvqo_bf16_value(q[(t * AH + h) * 576 + d])) * fabs(keys[(int64_t)j * 576 + d]);
        dmax = fmax(dmax, acc);
      }
      const double e_s = 576.0 * ldexp(1.0, -24) * scale * dmax;
      const double eps = ldexp(1.0, -9) + e_s + ldexp(1.0, -20);
      for (int d = 0; d < 512; ++d) {
        const double w = want_o[(t * AH + h) * 512 + d];
        const double got = kvqo_bf16_value(o_bits[(t * AH + h) * 512 + d]);
        if (fabs(got - w) > 2 * eps / (1 - eps) * vmax + ldexp(1.0, -9) * fabs(w)) {
          fprintf(stderr, "attention t%d h%d d%d: %g vs %g\n", t, h, d, got, w);
          return 8;
        }
      }
      if (fabs(lse[t * AH + h] - want_lse[t * AH + h]) > eps + e_s + ldexp(1.0, -22) * fabs(want_lse[t * AH + h])) {
        fprintf(stderr, "attention lse t%d h%d: %g vs %g\n", t, h, lse[t * AH + h], want_lse[t * AH + h]);
        return 9;
      }
    }
  }
  printf("C ABI: write (64 tokens) and gather (40 rows) match the oracle bit for bit; attention (2 x 16 x 48) "
         "within its bound\n");
  return 0;
}
