// kvq_launch.h -- host launchers of the kernels (one per .cu file), called by
// the C ABI in kvq_abi.cu after it has validated the arguments.  Each returns
// the cudaError_t of its launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvq_device.cuh"

namespace kvq {


struct WriteArgs {
  const void* kv_c;
  int64_t kv_c_stride;
  const void* k_pe;
  int64_t k_pe_stride;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  uint8_t* cache;
  int64_t num_slots;     // num_blocks * block_size, < 2^32
  int32_t block_size;
  FastDiv block_div;     // divides a slot by block_size
  int64_t block_stride;
  int64_t entry_stride;
  int32_t* status;
};

struct GatherArgs {
  const uint8_t* cache;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride;
  int64_t entry_stride;
  void* dst;
  int64_t dst_stride;
  int64_t num_out;
  const int32_t* block_table;
  int64_t block_table_stride;
  int32_t block_table_width;
  const int32_t* workspace_starts;
  const int32_t* seq_starts;
  int32_t batch_size;
  int32_t* status;
  FastDiv block_div;     // divides a position by block_size
};

struct PerHeadArgs {
  const void* key;
  const void* value;
  int64_t key_stride_t, key_stride_h, value_stride_t, value_stride_h;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t head_size;
  uint8_t* cache;
  int64_t num_slots;
  int32_t block_size;
  int32_t layout;        // KVQ_LAYOUT_NHD or KVQ_LAYOUT_HND
  const float* k_scale;
  const float* v_scale;
  int32_t* status;
  FastDiv block_div;     // slot -> page
  // Set by the launcher for the groups-per-thread g it picks:
  FastDiv unit_div;      // flat thread index -> token (2 * H * D/16/g threads per token)
  FastDiv side_div;      // thread within token -> side (H * D/16/g)
  FastDiv head_div;      // thread within side -> head (D/16/g)
};

struct AttentionArgs {
  const void* q;                 // bf16 [num_tokens, num_heads, 576]
  int64_t q_stride_t, q_stride_h;
  int64_t num_tokens;
  int32_t num_heads;             // 1 .. 128 (sparse decode), >= 1 (dense prefill)
  FastDiv head_div;              // divides a packed (token, head) row by num_heads
  // sparse decode: each token's own list of global slots
  const int32_t* indices;        // global slots [num_tokens, topk], < 0 unused
  int64_t indices_stride;
  int32_t topk;
  // dense prefill: request b's query tokens [query_start[b], query_start[b+1])
  // attend to its context positions [0, context_lens[b]) through block_table
  const int32_t* query_start;    // [batch_size + 1]
  const int32_t* context_lens;   // [batch_size]
  const int32_t* block_table;    // [batch_size, >= block_table_width]
  int64_t block_table_stride;
  int32_t block_table_width;
  int32_t batch_size;
  int32_t max_query_len;         // bounds the grid (row blocks per request)
  const uint8_t* cache;
  int64_t num_blocks;
  int64_t num_slots;             // num_blocks * block_size
  int32_t block_size;
  FastDiv block_div;             // slot (or context position) -> block (or block-table column)
  int64_t block_stride, entry_stride;
  float scale_log2;              // softmax_scale * log2(e)
  void* out;                     // bf16 [num_tokens, num_heads, 512]
  int64_t out_stride_t, out_stride_h;
  float* lse;                    // fp32 [num_tokens, num_heads] or nullptr
  int64_t lse_stride_t;
  int32_t* status;
  int32_t wave;                  // set by the launcher: CTAs resident at once (one per SM)
  int32_t q_tma;                 // set by the launcher: query rows loaded through its tensor map
  // split over the keys: each token's list (sparse) or each request's context
  // (dense) cut into num_splits ranges of split_keys keys (whole 64-key
  // tiles), one CTA pair per range, each writing its normalised partial
  // output and base-2 lse to part_o / part_lse (nullptr: no split,
  // num_splits = 1, results straight to out / lse)
  int32_t num_splits;
  int32_t split_keys;
  // dense prefill over a gathered bf16 workspace: request b's context
  // positions are rows ws_starts[b] .. + context_lens[b] of ws
  const void* ws;                // bf16 [ws_rows, >= 576], row stride ws_stride elements
  int64_t ws_stride;
  int64_t ws_rows;
  const int32_t* ws_starts;      // [batch_size]
  float* part_o;                 // fp32 [num_tokens, num_heads, num_splits, 512]
  float* part_lse;               // fp32 [num_tokens, num_heads, num_splits, 2] (one per value half)
};

int64_t write_max_tokens();     // grid.x bound of the write launches
cudaError_t launch_write_nvfp4_ds_mla(const WriteArgs& a, cudaStream_t stream);
cudaError_t launch_write_fp8_ds_mla(const WriteArgs& a, cudaStream_t stream);
cudaError_t launch_gather_nvfp4_ds_mla(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_fp8_ds_mla(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_reshape_and_cache_nvfp4(const PerHeadArgs& a, cudaStream_t stream);
// Read-back: key / value are the bf16 OUTPUTS (written through const_cast).
cudaError_t launch_dequant_nvfp4_per_head(const PerHeadArgs& a, cudaStream_t stream);
cudaError_t launch_sparse_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_sparse_mla_attention_fp8(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream);
// Split-key sparse decode: the partial launch, then the combine into out / lse.
cudaError_t launch_sparse_mla_attention_split_nvfp4(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_sparse_mla_attention_split_fp8(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_mla_attention_split_nvfp4(const AttentionArgs& a, cudaStream_t stream);
// Dense prefill whose keys are rows of a gathered bf16 workspace.
cudaError_t launch_prefill_mla_attention_workspace(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_mla_attention_split_fp8(const AttentionArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_mla_attention_fp8(const AttentionArgs& a, cudaStream_t stream);

struct IndexArgs {
  const int32_t* req_id;
  const int32_t* token_indices;
  int64_t token_indices_stride;   // elements between rows
  int64_t num_tokens;
  int32_t topk;
  const int32_t* block_table;
  int64_t block_table_stride;
  int32_t block_table_width;
  int32_t num_requests;
  int32_t block_size;
  int64_t num_blocks;
  int32_t* out;
  int64_t out_stride;
  int32_t* status;
  FastDiv block_div;              // position -> table column
  int32_t block_shift;            // log2(block_size) when it is a power of two (set by the launcher)
};
cudaError_t launch_req_index_to_global_slot(const IndexArgs& a, cudaStream_t stream);
cudaError_t launch_selftest_convert(uint32_t first_bits, int64_t count, uint8_t* e4m3_lo,
                                    uint8_t* e4m3_hi, uint8_t* e2m1_lo, uint8_t* e2m1_hi,
                                    uint16_t* bf16_out, int num_sms, cudaStream_t stream);

}  // namespace kvq
