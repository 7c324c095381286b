/*
 * kvq.h -- C ABI of the GB300 (sm_103a) quantized paged KV-cache library.
 *
 * The library writes bf16 key/value activations into quantized paged caches
 * and gathers quantized pages back into contiguous bf16 workspaces, for
 * DeepSeek-style sparse MLA (352-byte nvfp4_ds_mla and 656-byte fp8_ds_mla
 * entries) and for a per-head NVFP4 K/V cache.
 *
 * Conventions shared by every entry point
 *   - Pointers named by a tensor are DEVICE pointers owned by the caller.  The
 *     library allocates and frees nothing and keeps no state between calls.
 *   - Calls are asynchronous and stream-ordered: the kernel is launched on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream) and the call
 *     returns without synchronising.
 *   - bf16 tensors are row-major with strides in ELEMENTS; caches are uint8
 *     with strides in BYTES.
 *   - Alignment: every bf16 row must start on a 16-byte boundary (base
 *     pointer 16-byte aligned, row strides multiples of 8 elements); cache base
 *     pointers 16-byte aligned and cache strides multiples of 16 bytes.  Cache
 *     entries that start on 32-byte boundaries are written in whole 32-byte
 *     sectors (352 = 11 x 32, 656 = 20.5 x 32).
 *   - Sizes of zero are valid no-ops (KVQ_OK, nothing launched, no device
 *     query).
 *   - Every index read from device memory is bounds-checked by the kernels:
 *     an out-of-range slot, block id or position is skipped (nothing is
 *     written for that token / row).  When `d_status` (a device int32, may be
 *     NULL) is given, the kernel ORs the KVQ_STATUS_* bits below into it; the
 *     caller zeroes it beforehand and reads it back when convenient.
 *   - Host-side argument errors return before anything is launched.  The text
 *     of the last error on the calling thread is kvq_last_error_string().
 *   - Duplicate non-negative slots within one write race (last writer wins,
 *     per byte); bytes of slots not named by a call are never touched.
 *
 * Sources, cited by page title and section:
 *   [P1] vLLM PR #51724 "Enable W4A16 DSA: NVFP4 DS-MLA KV cache format for
 *        the FlashMLA Sparse backend"
 *   [P2] vLLM PR #37332 "Add NVFP4 quantization to the KV cache, extending
 *        reshape_and_cache_flash"
 *   [P3] vLLM PR #48642 "[Bugfix] Sparse MLA: enable fp8_ds_mla dense
 *        prefill"
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kvq_status;
#define KVQ_OK                      0
#define KVQ_ERR_INVALID_ARG         1  /* null pointer, negative size, misalignment, ... */
#define KVQ_ERR_UNSUPPORTED_DEVICE  2  /* current device is not compute capability 10.3  */
#define KVQ_ERR_CUDA                3  /* a CUDA runtime call or launch failed           */

/* Bits a kernel ORs into *d_status. */
#define KVQ_STATUS_BAD_INDEX   0x1  /* slot, block id or position out of range (skipped) */
#define KVQ_STATUS_BAD_BATCH   0x2  /* workspace_starts not non-decreasing within [0, T],
                                       or a row before the first request (skipped)       */
#define KVQ_STATUS_TIMEOUT     0x4  /* a bounded wait of the attention kernel (on its own
                                       tensor-core work or on another of its warp roles)
                                       expired; the outputs concerned were not written  */

/* Entry geometry ([P1] "Implementation breakdown" items 2-3). */
#define KVQ_MLA_NOPE_DIM               512
#define KVQ_MLA_ROPE_DIM               64
#define KVQ_NVFP4_DS_MLA_ENTRY_BYTES   352  /* [0,256) e2m1 NoPE | [256,320) e4m3 RoPE |
                                               [320,352) e4m3 scale of NoPE group g at 320+g */
#define KVQ_FP8_DS_MLA_ENTRY_BYTES     656  /* [0,512) e4m3 NoPE | [512,528) 4 fp32 scales,
                                               one per 128 NoPE values | [528,656) bf16 RoPE */
#define KVQ_WORKSPACE_DIM              576  /* gathered row: NoPE 0..511, RoPE 512..575      */

/* Per-head cache layouts ([P2] "Key source snippets", _nvfp4_split_data_scale:
 * the split views keep the cache's NHD or HND layout). */
#define KVQ_LAYOUT_NHD   0  /* [num_pages, 2, block_size, num_heads, full_dim] */
#define KVQ_LAYOUT_HND   1  /* [num_pages, 2, num_heads, block_size, full_dim] */

typedef struct CUstream_st* kvq_stream_t;   /* identical to cudaStream_t */

/*
 * kvq_write_nvfp4_ds_mla -- concat_and_cache for the 352-byte nvfp4_ds_mla
 * cache.  [P1] "Key source snippets" (concat_and_cache_nvfp4_ds_mla_kernel)
 * and "Implementation breakdown" item 3.
 *
 * For each token t < num_tokens with slot s = slot_mapping[t]:
 *   s < 0                        padding: nothing is written for it (its
 *                                row may still be read);
 *   s >= num_blocks*block_size   out of range: skipped, KVQ_STATUS_BAD_INDEX;
 *   otherwise the entry at kv_cache + (s / block_size) * block_stride +
 *   (s % block_size) * entry_stride receives
 *     bytes [8g, 8g+8)  the 16 NoPE values of group g (g = 0..31) as e2m1
 *                       codes of x * (1 / sf_g), value 2k in the low nibble
 *                       of byte k, round-to-nearest-even, saturating;
 *     bytes [256, 320)  the 64 RoPE values as e4m3 (RN, saturating, unscaled);
 *     byte  320 + g     sf_g = e4m3_rn_sat(max|x| over group g / 6), computed
 *                       in fp32 (1/sf taken as 0 when sf is 0).
 * kv_c: bf16 [num_tokens, >=512], row stride kv_c_stride elements.
 * k_pe: bf16 [num_tokens, >=64],  row stride k_pe_stride elements.
 * slot_mapping: int64 [num_tokens].
 * kv_cache: uint8, num_blocks blocks of block_size entries; entry_stride >=
 *   352 bytes; strides in bytes.
 */
kvq_status kvq_write_nvfp4_ds_mla(
    const void* kv_c, int64_t kv_c_stride,
    const void* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t num_tokens,
    uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_gather_upconvert_nvfp4_ds_mla -- cp_gather_and_upconvert for the
 * 352-byte cache.  [P1] "Key source snippets"
 * (cp_gather_and_upconvert_nvfp4_kv_cache_kernel) with the seq_starts /
 * workspace_starts interface of [P3] "Implementation breakdown" item 2 and
 * "Key source snippets" (_compute_prefill_context).
 *
 * Output row w (0 <= w < num_out_tokens) belongs to request b, the largest b
 * with workspace_starts[b] <= w (request b owns rows [ws[b], ws[b+1]), the
 * last one up to num_out_tokens; zero-length requests are allowed).  Its
 * position is p = seq_starts[b] + (w - ws[b]); the source entry is at block
 * block_table[b * block_table_stride + p / block_size], offset p %
 * block_size.  Row w of dst receives bf16(e2m1 * sf) for the 512 NoPE values
 * and bf16(e4m3) for the 64 RoPE values -- both exact.  Rows whose source
 * cannot be resolved (p / block_size >= block_table_width, a block id outside
 * [0, num_blocks), a row before the first request) are skipped.
 * dst: bf16 [num_out_tokens, >=576], row stride dst_stride elements.
 * block_table: int32 [batch_size, >= block_table_width], row stride
 *   block_table_stride elements.
 * workspace_starts, seq_starts: int32 [batch_size] (a cu_seq_lens array of
 *   batch_size + 1 entries may be passed; its last entry is not read).
 */
kvq_status kvq_gather_upconvert_nvfp4_ds_mla(
    const uint8_t* src_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    void* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts, int32_t batch_size,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_gather_upconvert_fp8_ds_mla -- cp_gather_and_upconvert_fp8_kv_cache
 * with seq_starts (seq_lens removed).  [P3] "Implementation breakdown"
 * items 2 and 4, "Key source snippets".  Same index walk and arguments as
 * kvq_gather_upconvert_nvfp4_ds_mla; entry_stride >= 656.  NoPE value k =
 * bf16_rn(fp32(e4m3(byte k)) * scale[k / 128]) with one fp32 rounding; RoPE
 * bf16 copied bit for bit.
 */
kvq_status kvq_gather_upconvert_fp8_ds_mla(
    const uint8_t* src_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    void* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts, int32_t batch_size,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_write_fp8_ds_mla -- concat_and_cache for the 656-byte fp8_ds_mla cache
 * ([P1] "Implementation breakdown" item 2 gives the size; the recipe is the
 * format spec's).  Same slot rules and arguments as kvq_write_nvfp4_ds_mla;
 * entry_stride >= 656.  Per 128-value tile j: s_j = max|x| / 448 in fp32 (1
 * when the tile is all zero), NoPE byte = e4m3_rn_sat(x / s_j) with IEEE
 * division, scale j stored as fp32 at 512 + 4j, RoPE bf16 bits at 528.
 */
kvq_status kvq_write_fp8_ds_mla(
    const void* kv_c, int64_t kv_c_stride,
    const void* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t num_tokens,
    uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_reshape_and_cache_nvfp4 -- reshape_and_cache_flash into a per-head
 * NVFP4 K/V cache.  [P2] "Function and motivation" and "Implementation
 * breakdown" item 4 (layout [K_data | K_scale | V_data | V_scale], per-tensor
 * scale), "Key source snippets" (cache shape (num_pages, 2, block_size,
 * num_kv_heads, full_dim) with full_dim = head_size/2 + head_size/16, data_dim
 * = full_dim*8/9).
 *
 * kv_cache is a contiguous uint8 [num_pages, 2, block_size, num_heads,
 * full_dim] allocation (layout KVQ_LAYOUT_NHD) or [num_pages, 2, num_heads,
 * block_size, full_dim] (KVQ_LAYOUT_HND).  Inside page p and side s (K = 0,
 * V = 1) its block_size*num_heads*full_dim bytes hold one head_size/2-byte
 * data row per (offset, head), then one head_size/16-byte scale row per
 * (offset, head); rows in the layout's order: offset * num_heads + head
 * (NHD) or head * block_size + offset (HND).
 * Token t with slot s = slot_mapping[t] >= 0 goes to page s / block_size,
 * offset s % block_size: each 16-value group of y = x * (1 / scale) (fp32;
 * scale = *k_scale or *v_scale, device fp32 scalars) is quantized exactly as
 * an nvfp4_ds_mla NoPE group.  head_size must be a multiple of 16.
 * key, value: bf16 [num_tokens, num_heads, head_size] with token and head
 * strides in elements (unit inner stride).
 */
kvq_status kvq_reshape_and_cache_nvfp4(
    const void* key, const void* value,
    int64_t key_stride_t, int64_t key_stride_h,
    int64_t value_stride_t, int64_t value_stride_h,
    const int64_t* slot_mapping, int64_t num_tokens,
    int32_t num_heads, int32_t head_size,
    uint8_t* kv_cache, int64_t num_pages, int32_t block_size, int32_t layout,
    const float* k_scale, const float* v_scale,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_dequant_nvfp4_per_head -- reads the per-head NVFP4 cache back into bf16
 * (the GPU counterpart of [P2] "Implementation breakdown" item 5,
 * dequant_nvfp4_kv_cache; the decode consumer [P2] leaves unimplemented).
 * For each token t with slot s = slot_mapping[t] >= 0 (in range), every
 * 16-value group of head h and side (K -> key_out, V -> value_out) becomes
 * bf16_rn((e2m1 * sf) * scale): the first product exact, one fp32 rounding
 * for the per-tensor scale (*k_scale / *v_scale).  Rows of padding and
 * out-of-range slots are not written.  Cache layouts and argument rules as in
 * kvq_reshape_and_cache_nvfp4; key_out / value_out are bf16 [num_tokens,
 * num_heads, head_size] outputs with token and head strides in elements.
 */
kvq_status kvq_dequant_nvfp4_per_head(
    const uint8_t* kv_cache, int64_t num_pages, int32_t block_size, int32_t layout,
    int32_t num_heads, int32_t head_size,
    const int64_t* slot_mapping, int64_t num_tokens,
    const float* k_scale, const float* v_scale,
    void* key_out, int64_t key_stride_t, int64_t key_stride_h,
    void* value_out, int64_t value_stride_t, int64_t value_stride_h,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_sparse_mla_attention_nvfp4_ds_mla -- sparse MLA attention read straight
 * from the 352-byte nvfp4_ds_mla cache, the consumer that makes the bf16
 * workspace unnecessary.  [P1] "Key source snippets" (flashmla_sparse.py: the
 * sparse decode path serves the quantized DS-MLA formats and reads the cache
 * itself) and [P3] "Implementation breakdown" item 3 (that decode is MQA over
 * the latent cache).  For token t < num_tokens, head h < num_heads and the
 * valid entries j of indices[t * indices_stride + 0 .. topk) (global slots as
 * kvq_req_index_to_global_slot produces them; < 0 = unused, >= num_blocks *
 * block_size = out of range: skipped, KVQ_STATUS_BAD_INDEX):
 *   s_j = softmax_scale * (q[t,h] . k_j)     k_j = the slot's 576 decoded
 *                                            values (NoPE then RoPE, exact)
 *   out[t,h] = sum_j exp(s_j - m) k_j[0:512] / sum_j exp(s_j - m)
 *   lse[t,h] = m + ln(sum_j exp(s_j - m)),   m = max_j s_j
 * A token with no valid entry gets out = 0 and lse = -inf.
 * Arithmetic: q . k on the tensor cores (bf16 products, fp32 accumulation);
 * exp in base 2 in fp32; the weights rounded to bf16 for the weighted sum
 * (fp32 accumulation), and the denominator summed from those rounded
 * weights; out rounded once to bf16.
 * q: bf16 [num_tokens, num_heads, 576] (token / head strides in elements,
 * multiples of 8, head stride >= 576, unit inner stride); 1 <= num_heads <=
 * 128.  out: bf16 [num_tokens, num_heads, 512] (strides multiples of 8, head
 * stride >= 512, token stride >= (num_heads - 1) * head stride + 512).  lse:
 * fp32 [num_tokens, num_heads] with token stride lse_stride_t >= num_heads,
 * or NULL.  indices: int32, indices_stride >= topk.  The cache follows the
 * nvfp4 gather's rules.  Every wait of the kernel is bounded (about 2 s):
 * if one expires (not expected), the kernel sets KVQ_STATUS_TIMEOUT, leaves
 * the outputs of the query rows concerned unwritten (each of the two CTAs of
 * a token writes its own 256 output columns) and still returns, with nothing
 * of it left running on the device.
 */
kvq_status kvq_sparse_mla_attention_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_sparse_mla_attention_fp8_ds_mla -- the same attention read straight
 * from the 656-byte fp8_ds_mla cache ([P1] "Key source snippets": the sparse
 * decode path serves both quantized DS-MLA formats; [P3] is about this
 * cache).  The key of a slot is what kvq_gather_upconvert_fp8_ds_mla writes
 * for it: NoPE value k = bf16_rn(fp32(e4m3) * s_{k/128}) (one fp32 product
 * rounding), RoPE the stored bf16.  Arguments, arithmetic, outputs and status
 * as kvq_sparse_mla_attention_nvfp4_ds_mla; entry_stride >= 656.
 */
kvq_status kvq_sparse_mla_attention_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream);

#define KVQ_ATTN_MAX_SPLITS 32         /* key ranges per token of the split-key decode */

/*
 * kvq_sparse_mla_attention_split_workspace_bytes -- bytes of device workspace
 * the split-key decode below needs for num_tokens x num_heads query rows cut
 * into num_splits key ranges: num_tokens * num_heads * num_splits * 514 * 4,
 * rounded up to 16.  -1 for a negative or zero argument or a size past
 * INT64_MAX.
 */
int64_t kvq_sparse_mla_attention_split_workspace_bytes(int64_t num_tokens, int32_t num_heads,
                                                       int32_t num_splits);

/*
 * kvq_sparse_mla_attention_split_nvfp4_ds_mla,
 * kvq_sparse_mla_attention_split_fp8_ds_mla -- the sparse MLA attention of
 * kvq_sparse_mla_attention_nvfp4_ds_mla / _fp8_ds_mla (the same definition,
 * [P1] "Key source snippets" and [P3] "Implementation breakdown" item 3; the
 * same arguments, arithmetic rules, outputs and status), scheduled for decode
 * batches too small to fill the GPU: no passage of the pages defines the
 * schedule, which is a split over the keys.  Each token's list is cut into
 * num_splits ranges of whole 64-key tiles (the last ranges may be empty); a
 * pair of CTAs per (token, range) writes the range's normalised partial output
 * o_r (fp32) and its base-2 log-sum-exp L_r into the workspace, and a second
 * launch on the same stream combines them:
 *   out = sum_r w_r o_r / sum_r w_r,   lse = (M + log2 sum_r w_r) ln 2,
 *   w_r = 2^(L_r - M),   M = max_r L_r.
 * Each range's weights are relative to its own maximum before their bf16
 * rounding, so the result differs from the one-range result within the same
 * error bound.  1 <= num_splits <= KVQ_ATTN_MAX_SPLITS; num_splits = 1 is
 * the plain entry point (the workspace is not used and may be NULL).
 * workspace: device memory owned by the caller, 16-byte aligned, at least
 * kvq_sparse_mla_attention_split_workspace_bytes(num_tokens, num_heads,
 * num_splits) bytes (workspace_bytes says how many there are), overwritten:
 * fp32 partial rows [num_tokens, num_heads, num_splits, 512], then the fp32
 * range lse values (two per row and range, one per value half); no other
 * call may use it while this one runs.  The range lse values are set to NaN
 * before the partial launch, and the combine leaves a row untouched if any
 * of its ranges was not written (as after a KVQ_STATUS_TIMEOUT), as the
 * plain entry point leaves the rows of a CTA that timed out.
 */
kvq_status kvq_sparse_mla_attention_split_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t num_splits, void* workspace, int64_t workspace_bytes,
    int32_t* d_status, kvq_stream_t stream);
kvq_status kvq_sparse_mla_attention_split_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t num_splits, void* workspace, int64_t workspace_bytes,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_prefill_mla_attention_split_nvfp4_ds_mla,
 * kvq_prefill_mla_attention_split_fp8_ds_mla -- the dense prefill of
 * kvq_prefill_mla_attention_nvfp4_ds_mla / _fp8_ds_mla (the same definition,
 * [P3] "Function and motivation" and "Key source snippets",
 * _compute_prefill_context; the same arguments, arithmetic rules, outputs and
 * status) split over the context, as the split-key decode above splits a
 * token's list, for batches with few query rows over long contexts.  Each
 * request's context is cut into num_splits ranges of whole 64-position
 * tiles sized from max_context_len (ceil(ceil(max_context_len / 64) /
 * num_splits) tiles; the last range of a request also takes every position
 * past the others, so a context longer than max_context_len is still
 * attended in full, only less evenly split).  workspace as for the split
 * decode, sized by kvq_sparse_mla_attention_split_workspace_bytes(num_tokens,
 * num_heads, num_splits) (num_tokens = all query tokens).  Rows of query
 * tokens that belong to no request, or to a skipped one, are left
 * untouched, as by the plain entry point.
 */
kvq_status kvq_prefill_mla_attention_split_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t max_context_len, int32_t num_splits, void* workspace, int64_t workspace_bytes,
    int32_t* d_status, kvq_stream_t stream);
kvq_status kvq_prefill_mla_attention_split_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t max_context_len, int32_t num_splits, void* workspace, int64_t workspace_bytes,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_prefill_mla_attention_workspace -- the dense prefill attention of
 * kvq_prefill_mla_attention_nvfp4_ds_mla over the bf16 workspace that
 * kvq_gather_upconvert_nvfp4_ds_mla / _fp8_ds_mla fill: the pages' own
 * prefill flow ([P3] "Key source snippets", _compute_prefill_context: the
 * context gathered into the bf16 workspace, then attention over it).
 * Request b's context position p is workspace row workspace_starts[b] + p
 * (576 bf16 values, NoPE then RoPE), p < context_lens[b].  Same definition,
 * arithmetic, outputs and status as the quantized-cache prefill; over the
 * workspace that the gather wrote from the same cache the results are equal
 * bit for bit.  The keys arrive by tensor-map copies (no decode in the
 * attention), so the pair of calls pays off when many query rows share a
 * context: the gather decodes it once, the fused prefill once per CTA.
 * workspace: bf16, 16-byte aligned, workspace_rows rows (< 2^31) of
 * workspace_stride >= 576 elements (a multiple of 8).  Rows that a tile
 * reads past a request's context (up to 63 more, or up to the end of the
 * workspace, past which zeros are read) must hold finite values, as the
 * gather's packed output does.  A request whose context does not lie inside
 * the workspace is skipped (KVQ_STATUS_BAD_BATCH, its rows untouched).
 */
kvq_status kvq_prefill_mla_attention_workspace(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, const int32_t* workspace_starts,
    int32_t batch_size, int32_t max_query_len,
    const void* workspace, int64_t workspace_stride, int64_t workspace_rows,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream);

#define KVQ_NOALLOC_SCRATCH_BYTES (24LL << 20)   /* fixed partial-result array, per GPU */

/*
 * kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc -- the split-key decode
 * of kvq_sparse_mla_attention_split_nvfp4_ds_mla (same arguments except the
 * workspace, same results bit for bit) for callers that cannot allocate
 * device memory when they call in: an engine that reserved the GPU's memory
 * for its own pools at start-up, or host code on a latency-critical path
 * where an allocation can synchronise the device.  The paper has no
 * counterpart: this is an addition of this library.  The partial results go
 * to one array of KVQ_NOALLOC_SCRATCH_BYTES (24 MiB) that the library holds
 * on every GPU that loads it, until the process exits; a call whose
 * num_tokens x num_heads x num_splits rows need more
 * (kvq_sparse_mla_attention_split_workspace_bytes) returns
 * KVQ_ERR_INVALID_ARG and launches nothing.  num_splits = 1 uses no array.
 * The first call on a device (with that device current) looks up the array's
 * device address and keeps it: make that first call before any stream
 * capture.  Every call shares the array, which keeps the last call's
 * contents; nothing in it has to start at zero (a call writes every partial
 * row it reads before reading it), but calls that overlap on the GPU (other
 * streams, other host threads) race on it, so the caller orders them.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 */
kvq_status kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t num_splits,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_prefill_mla_attention_nvfp4_ds_mla -- dense prefill over the 352-byte
 * cache: the query tokens of each request attend to every position of its
 * context, read straight from the quantized pages through the block table
 * ([P3] "Function and motivation" and "Key source snippets",
 * _compute_prefill_context, which otherwise gathers that context into the
 * bf16 workspace first).  Request b < batch_size owns the query tokens
 * [query_start[b], query_start[b+1]) (rows of q / out / lse; at most
 * max_query_len of them) and the context positions p < context_lens[b];
 * position p is entry p % block_size of block block_table[b *
 * block_table_stride + p / block_size].  For each of its query tokens t and
 * heads h, out[t,h] and lse[t,h] are the attention of
 * kvq_sparse_mla_attention_nvfp4_ds_mla with the key list = all of those
 * positions, with the same arithmetic.  (token, head) rows of a request are
 * processed 128 at a time, so a decoded page feeds the heads of every query
 * token in such a block.  A position whose block-table column is >=
 * block_table_width or whose block id is outside [0, num_blocks) is skipped
 * (KVQ_STATUS_BAD_INDEX); a request whose query range is not inside [0,
 * num_tokens) or is longer than max_query_len is skipped (KVQ_STATUS_BAD_BATCH);
 * a request with no context position gets out = 0, lse = -inf.
 * q, out, lse: as kvq_sparse_mla_attention_nvfp4_ds_mla, num_heads >= 1
 * (max_query_len * num_heads < 2^31).  query_start: int32 [batch_size + 1];
 * context_lens: int32 [batch_size]; block_table: int32 [batch_size, >=
 * block_table_width]; batch_size <= 65535.  Waits are bounded as in the
 * sparse form (KVQ_STATUS_TIMEOUT).
 */
kvq_status kvq_prefill_mla_attention_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_prefill_mla_attention_fp8_ds_mla -- the same dense prefill over the
 * 656-byte fp8_ds_mla cache (keys as kvq_gather_upconvert_fp8_ds_mla writes
 * them); entry_stride >= 656.
 */
kvq_status kvq_prefill_mla_attention_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h,
    float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_req_index_to_global_slot -- sparse-decode index conversion feeding the
 * sparse MLA decode ([P3] "Implementation breakdown" item 1:
 * triton_convert_req_index_to_global_index and its length check).  For decode
 * token i < num_tokens of request r = req_id[i] and each k < topk, position
 * p = token_indices[i * token_indices_stride + k] becomes
 * out[i * out_stride + k] = block_table[r][p / block_size] * block_size +
 * p % block_size, or -1 when p < 0 (an unused top-k entry).  An out-of-range
 * request, column or block id also gives -1 and sets KVQ_STATUS_BAD_INDEX.
 * As on the page, a call whose req_id length (num_req_ids) differs from the
 * number of token_indices rows (num_tokens) is rejected with
 * KVQ_ERR_INVALID_ARG before anything is launched.  All arrays int32;
 * num_blocks * block_size must fit an int32 slot.
 */
kvq_status kvq_req_index_to_global_slot(
    const int32_t* req_id, int64_t num_req_ids,
    const int32_t* token_indices, int64_t num_tokens, int32_t topk,
    int64_t token_indices_stride,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int32_t num_requests, int32_t block_size, int64_t num_blocks,
    int32_t* out, int64_t out_stride,
    int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_selftest_convert -- exposes the device number-format converters the
 * kernels above use, for exhaustive testing.  For i < count and f the float
 * whose bit pattern is first_bits + i (mod 2^32):
 *   e4m3_lo[i] / e4m3_hi[i]  e4m3 code of f placed in the low / high lane of
 *                            the packed two-value conversion;
 *   e2m1_lo[i] / e2m1_hi[i]  the same for e2m1 (code in the low 4 bits);
 *   bf16_out[i]              bf16 bits of f rounded to nearest even.
 * Any output pointer may be NULL.  Not part of the cache path.
 */
kvq_status kvq_selftest_convert(
    uint32_t first_bits, int64_t count,
    uint8_t* e4m3_lo, uint8_t* e4m3_hi, uint8_t* e2m1_lo, uint8_t* e2m1_hi,
    uint16_t* bf16_out, kvq_stream_t stream);

/* Text of the last error returned on the calling thread ("" if none). */
const char* kvq_last_error_string(void);

/* Library ABI version (major * 100 + minor). */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
