/*
 * kvq_oracle.h -- CPU oracle for the quantized paged KV-cache write and
 * gather-upconvert path (DeepSeek-style sparse MLA caches).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this library.  It shares no source,
 * header, table or constant with the CUDA library; neither includes the other.
 *
 * Every function is a plain scalar loop in token order.  Floating-point steps
 * that decide a quantised code run in fp32, because the kernels the pages
 * describe compute them in fp32 (an fp32 inverse scale feeds the
 * cvt.rn.satfinite.e2m1x2.f32 instruction); results that are exact
 * (e2m1 x e4m3 products) are formed in double.
 *
 * Sources, cited by page title and section:
 *   [P1] vLLM PR #51724, "Enable W4A16 DSA: NVFP4 DS-MLA KV cache format for
 *        the FlashMLA Sparse backend" -- sections "Implementation breakdown",
 *        "Key source snippets" (nvfp4_ds_mla_cache_kernels.cu, test_cache.py).
 *   [P2] vLLM PR #37332, "Add NVFP4 quantization to the KV cache, extending
 *        reshape_and_cache_flash" -- sections "Function and motivation",
 *        "Implementation breakdown", "Key source snippets" (torch_utils.py,
 *        flashinfer.py).
 *   [P3] vLLM PR #48642, "[Bugfix] Sparse MLA: enable fp8_ds_mla dense
 *        prefill" -- sections "Implementation breakdown", "Key source
 *        snippets" (mla_attention.py _compute_prefill_context).
 *   [OFP8] OCP 8-bit Floating Point Specification (OFP8) rev 1.0, E4M3.
 *   [MX]   OCP Microscaling Formats (MX) Specification v1.0, FP4 E2M1.
 *
 * Parity status: the per-head NVFP4 byte layout (region order inside a page),
 * the 656-byte fp8_ds_mla entry order and the sparse-decode index formula are
 * fixed by the written format spec, not by the pages: parity for those is
 * unpinned against the pages (the arithmetic is pinned).
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar number formats ------------------------------------------------ */
double   kvqo_e4m3_value(uint8_t code);      /* NaN for 0x7F / 0xFF            */
double   kvqo_e2m1_value(uint8_t nibble);    /* low 4 bits used                */
float    kvqo_bf16_value(uint16_t bits);
uint8_t  kvqo_e4m3_rn_sat(float f);
uint8_t  kvqo_e2m1_rn_sat(float f);
uint16_t kvqo_bf16_rn(float f);

/* Array forms, for sweeps over many inputs. */
void kvqo_encode_bits_range(uint32_t first_bits, int64_t count,
                            uint8_t* e4m3_out, uint8_t* e2m1_out);
void kvqo_bf16_rn_bits_range(uint32_t first_bits, int64_t count, uint16_t* out);
void kvqo_e4m3_rn_sat_array(const float* in, int64_t n, uint8_t* out);
void kvqo_e2m1_rn_sat_array(const float* in, int64_t n, uint8_t* out);
void kvqo_bf16_rn_array(const float* in, int64_t n, uint16_t* out);

/* ---- format constants (the oracle's own copy) ----------------------------- */
int32_t kvqo_nvfp4_ds_mla_entry_bytes(void);   /* 352 */
int32_t kvqo_fp8_ds_mla_entry_bytes(void);     /* 656 */
int32_t kvqo_nvfp4_full_dim(int32_t head_size);
int32_t kvqo_nvfp4_data_dim(int32_t full_dim);
int32_t kvqo_nvfp4_scale_dim(int32_t full_dim);

/* ---- operations ----------------------------------------------------------- */
/* All byte strides are in bytes; bf16 tensors are passed as uint16 bit
 * patterns with strides in elements.  Each op processes tokens / rows in the
 * half-open range given and returns how many it skipped because an index was
 * out of range (padding slots < 0 are not counted). */

int64_t kvqo_write_nvfp4_ds_mla(
    const uint16_t* kv_c, int64_t kv_c_stride,
    const uint16_t* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride);

int64_t kvqo_write_fp8_ds_mla(
    const uint16_t* kv_c, int64_t kv_c_stride,
    const uint16_t* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride);

/* Gathers: output row i of dst is workspace row rows[i] (rows == NULL means
 * row i itself).  Rows whose source cannot be resolved are left untouched. */
int64_t kvqo_gather_nvfp4_ds_mla(
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    uint16_t* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts,
    int32_t batch_size, const int64_t* rows, int64_t n_rows);

int64_t kvqo_gather_fp8_ds_mla(
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    uint16_t* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts,
    int32_t batch_size, const int64_t* rows, int64_t n_rows);

int64_t kvqo_reshape_and_cache_nvfp4(
    const uint16_t* key, const uint16_t* value,
    int64_t key_stride_t, int64_t key_stride_h,
    int64_t value_stride_t, int64_t value_stride_h,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    int32_t num_heads, int32_t head_size,
    uint8_t* cache, int64_t num_pages, int32_t block_size,
    float k_scale, float v_scale, int32_t layout);   /* layout: 0 = NHD, 1 = HND */

/* Reads K and V back out of the per-head cache at slot_mapping[t] into bf16
 * [T, H, D] (contiguous); rows for padding / out-of-range slots untouched. */
int64_t kvqo_dequant_nvfp4_per_head(
    const uint8_t* cache, int64_t num_pages, int32_t block_size,
    int32_t num_heads, int32_t head_size,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    float k_scale, float v_scale, int32_t layout, uint16_t* key_out, uint16_t* value_out);

/* Sparse-decode index conversion: out[i*topk+k] = global slot of position
 * token_indices[i*topk+k] of request req_id[i], or -1. */
int64_t kvqo_req_index_to_global_slot(
    const int32_t* req_id, const int32_t* token_indices, int64_t num_tokens,
    int32_t topk, const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width, int32_t num_requests, int32_t block_size,
    int64_t num_blocks, int32_t* out);

/* Sparse MLA attention (MQA form) of queries q bf16 [T, H, 576] over the
 * top-k global slots indices[t][0..topk) of the nvfp4_ds_mla cache: o[t,h]
 * [512] and lse[t,h] (natural log; may be NULL) in double.  Negative entries
 * are unused; out-of-range slots are skipped and counted; no valid entry
 * gives o = 0, lse = -inf.  Returns -1 if scratch memory runs out. */
int64_t kvqo_sparse_mla_attention_nvfp4_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t t_begin, int64_t t_end, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t);

/* The same over the 656-byte fp8_ds_mla cache (keys as the fp8 gather
 * upconverts them). */
int64_t kvqo_sparse_mla_attention_fp8_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t t_begin, int64_t t_end, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t);

/* Dense prefill of the query tokens [query_start[b], query_start[b+1]) of
 * requests b_begin <= b < b_end over their context positions [0,
 * context_lens[b]), read through block_table (the same attention as the
 * sparse form, with every context position listed).  Out-of-range block-table
 * columns or block ids are skipped and counted.  Returns -1 if scratch memory
 * runs out. */
int64_t kvqo_prefill_mla_attention_nvfp4_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int64_t b_begin, int64_t b_end,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t);
int64_t kvqo_prefill_mla_attention_fp8_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int64_t b_begin, int64_t b_end,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t);

/* Decodes one 656-byte fp8_ds_mla entry to its 576 bf16 values (as doubles). */
void kvqo_decode_fp8_ds_mla_entry(const uint8_t* entry, double* out576);

/* Decodes one 352-byte nvfp4_ds_mla entry to 576 values (NoPE then RoPE). */
void kvqo_decode_nvfp4_ds_mla_entry(const uint8_t* entry, double* out576);

#ifdef __cplusplus
}
#endif
#endif
