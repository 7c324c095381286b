// kvq_abi.cu -- the extern "C" entry points declared in include/kvq.h:
// host-side validation, device check, launch on the caller's stream, status.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <mutex>
#include <string>

#include "kvq.h"
#include "kvq_launch.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

kvq_status ok() {
  g_last_error.clear();
  return KVQ_OK;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// The kernels are built for sm_103a only (GB300); the pages gate the NVFP4
// DS-MLA format on compute capability 10.x.
kvq_status check_device(const char* fn, int* num_sms = nullptr) {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess && num_sms != nullptr)
    e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(KVQ_ERR_UNSUPPORTED_DEVICE,
                "%s: this library is built for sm_103a (GB300); device %d is sm_%d%d", fn, dev,
                major, minor);
  return KVQ_OK;
}

kvq_status launched(const char* fn, cudaError_t e) {
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

#define KVQ_REQUIRE(cond, ...) \
  do {                         \
    if (!(cond)) return fail(KVQ_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

// Shared checks of a [num_blocks, block_size, entry] cache.
kvq_status check_mla_cache(const char* fn, const void* cache, int64_t num_blocks,
                           int32_t block_size, int64_t block_stride, int64_t entry_stride,
                           int64_t entry_bytes) {
  KVQ_REQUIRE(cache != nullptr, "%s: cache is NULL", fn);
  KVQ_REQUIRE(aligned(cache, 16), "%s: cache base must be 16-byte aligned", fn);
  KVQ_REQUIRE(num_blocks > 0 && block_size > 0, "%s: num_blocks and block_size must be positive", fn);
  KVQ_REQUIRE(num_blocks <= (int64_t{1} << 32) / block_size,
              "%s: num_blocks * block_size must not exceed 2^32 slots", fn);
  KVQ_REQUIRE(entry_stride >= entry_bytes && entry_stride % 16 == 0,
              "%s: entry_stride must be >= %lld and a multiple of 16 (got %lld)", fn,
              static_cast<long long>(entry_bytes), static_cast<long long>(entry_stride));
  KVQ_REQUIRE(block_stride > 0 && block_stride % 16 == 0,
              "%s: block_stride must be a positive multiple of 16 (got %lld)", fn,
              static_cast<long long>(block_stride));
  return KVQ_OK;
}

kvq_status check_bf16_rows(const char* fn, const char* name, const void* p, int64_t stride,
                           int64_t width) {
  KVQ_REQUIRE(p != nullptr, "%s: %s is NULL", fn, name);
  KVQ_REQUIRE(aligned(p, 16), "%s: %s must be 16-byte aligned", fn, name);
  KVQ_REQUIRE(stride >= width && stride % 8 == 0,
              "%s: %s row stride must be >= %lld and a multiple of 8 elements (got %lld)", fn, name,
              static_cast<long long>(width), static_cast<long long>(stride));
  return KVQ_OK;
}

kvq_status write_common(const char* fn, int64_t entry_bytes,
                        cudaError_t (*launch)(const kvq::WriteArgs&, cudaStream_t),
                        const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                        int64_t k_pe_stride, const int64_t* slot_mapping, int64_t num_tokens,
                        uint8_t* kv_cache, int64_t num_blocks, int32_t block_size,
                        int64_t block_stride, int64_t entry_stride, int32_t* d_status,
                        kvq_stream_t stream) {
  KVQ_REQUIRE(num_tokens >= 0, "%s: num_tokens < 0", fn);
  if (num_tokens == 0) return ok();
  KVQ_REQUIRE(num_tokens <= kvq::write_max_tokens(), "%s: num_tokens exceeds %lld (grid limit)", fn,
              static_cast<long long>(kvq::write_max_tokens()));
  if (kvq_status s = check_bf16_rows(fn, "kv_c", kv_c, kv_c_stride, KVQ_MLA_NOPE_DIM)) return s;
  if (kvq_status s = check_bf16_rows(fn, "k_pe", k_pe, k_pe_stride, KVQ_MLA_ROPE_DIM)) return s;
  KVQ_REQUIRE(slot_mapping != nullptr, "%s: slot_mapping is NULL", fn);
  KVQ_REQUIRE(aligned(slot_mapping, 8), "%s: slot_mapping must be 8-byte aligned", fn);
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (kvq_status s = check_mla_cache(fn, kv_cache, num_blocks, block_size, block_stride,
                                     entry_stride, entry_bytes))
    return s;
  if (kvq_status s = check_device(fn)) return s;
  const kvq::WriteArgs a{kv_c,       kv_c_stride,  k_pe,         k_pe_stride,
                         slot_mapping, num_tokens, kv_cache,   num_blocks * block_size,
                         block_size, kvq::FastDiv::make(static_cast<uint32_t>(block_size)),
                         block_stride, entry_stride, d_status};
  return launched(fn, launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status gather_common(const char* fn, int64_t entry_bytes,
                         cudaError_t (*launch)(const kvq::GatherArgs&, cudaStream_t),
                         const uint8_t* src_cache, int64_t num_blocks, int32_t block_size,
                         int64_t block_stride, int64_t entry_stride, void* dst, int64_t dst_stride,
                         int64_t num_out_tokens, const int32_t* block_table,
                         int64_t block_table_stride, int32_t block_table_width,
                         const int32_t* workspace_starts, const int32_t* seq_starts,
                         int32_t batch_size, int32_t* d_status, kvq_stream_t stream) {
  KVQ_REQUIRE(num_out_tokens >= 0, "%s: num_out_tokens < 0", fn);
  if (num_out_tokens == 0) return ok();
  KVQ_REQUIRE(num_out_tokens <= INT32_MAX, "%s: num_out_tokens exceeds int32 workspace_starts", fn);
  if (kvq_status s = check_mla_cache(fn, src_cache, num_blocks, block_size, block_stride,
                                     entry_stride, entry_bytes))
    return s;
  if (kvq_status s = check_bf16_rows(fn, "dst", dst, dst_stride, KVQ_WORKSPACE_DIM)) return s;
  KVQ_REQUIRE(batch_size > 0, "%s: batch_size must be positive", fn);
  KVQ_REQUIRE(block_table != nullptr && workspace_starts != nullptr && seq_starts != nullptr,
              "%s: block_table, workspace_starts and seq_starts must be non-NULL", fn);
  KVQ_REQUIRE(aligned(block_table, 4) && aligned(workspace_starts, 4) && aligned(seq_starts, 4),
              "%s: int32 arrays must be 4-byte aligned", fn);
  KVQ_REQUIRE(block_table_width > 0 && block_table_stride >= block_table_width,
              "%s: need block_table_width > 0 and block_table_stride >= block_table_width", fn);
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (kvq_status s = check_device(fn)) return s;
  const kvq::GatherArgs a{src_cache,        num_blocks,       block_size,        block_stride,
                          entry_stride,     dst,              dst_stride,        num_out_tokens,
                          block_table,      block_table_stride, block_table_width, workspace_starts,
                          seq_starts,       batch_size,       d_status,
                          kvq::FastDiv::make(static_cast<uint32_t>(block_size))};
  return launched(fn, launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status per_head_common(const char* fn, bool read_back,
                           cudaError_t (*launch)(const kvq::PerHeadArgs&, cudaStream_t),
                           const void* key, const void* value, int64_t key_stride_t,
                           int64_t key_stride_h, int64_t value_stride_t, int64_t value_stride_h,
                           const int64_t* slot_mapping, int64_t num_tokens, int32_t num_heads,
                           int32_t head_size, const uint8_t* kv_cache, int64_t num_pages,
                           int32_t block_size, int32_t layout, const float* k_scale,
                           const float* v_scale, int32_t* d_status, kvq_stream_t stream) {
  KVQ_REQUIRE(num_tokens >= 0, "%s: num_tokens < 0", fn);
  KVQ_REQUIRE(layout == KVQ_LAYOUT_NHD || layout == KVQ_LAYOUT_HND,
              "%s: layout must be KVQ_LAYOUT_NHD (0) or KVQ_LAYOUT_HND (1)", fn);
  if (num_tokens == 0) return ok();
  KVQ_REQUIRE(num_heads > 0 && head_size >= 16 && head_size % 16 == 0,
              "%s: need num_heads > 0 and head_size a positive multiple of 16", fn);
  KVQ_REQUIRE(num_tokens * 2 * num_heads * (head_size / 16) < (int64_t{1} << 32) - 256,
              "%s: num_tokens * 2 * num_heads * head_size / 16 must stay below 2^32 - 256", fn);
  KVQ_REQUIRE(key != nullptr && value != nullptr, "%s: key / value is NULL", fn);
  KVQ_REQUIRE(aligned(key, 16) && aligned(value, 16), "%s: key / value must be 16-byte aligned", fn);
  KVQ_REQUIRE(key_stride_t % 8 == 0 && key_stride_h % 8 == 0 && value_stride_t % 8 == 0 &&
                  value_stride_h % 8 == 0 && key_stride_t >= 0 && key_stride_h >= 0 &&
                  value_stride_t >= 0 && value_stride_h >= 0,
              "%s: key / value strides must be non-negative multiples of 8 elements", fn);
  if (read_back)
    KVQ_REQUIRE(key_stride_h >= head_size && key_stride_t >= num_heads * key_stride_h &&
                    value_stride_h >= head_size && value_stride_t >= num_heads * value_stride_h,
                "%s: output strides must not overlap rows", fn);
  KVQ_REQUIRE(slot_mapping != nullptr && aligned(slot_mapping, 8), "%s: bad slot_mapping", fn);
  KVQ_REQUIRE(k_scale != nullptr && v_scale != nullptr && aligned(k_scale, 4) && aligned(v_scale, 4),
              "%s: k_scale / v_scale must be device fp32 scalars", fn);
  KVQ_REQUIRE(kv_cache != nullptr && aligned(kv_cache, 16), "%s: kv_cache must be 16-byte aligned", fn);
  KVQ_REQUIRE(num_pages > 0 && block_size > 0, "%s: num_pages and block_size must be positive", fn);
  KVQ_REQUIRE(num_pages <= (int64_t{1} << 32) / block_size,
              "%s: num_pages * block_size must not exceed 2^32 slots", fn);
  const int64_t full_dim = head_size / 2 + head_size / 16;
  KVQ_REQUIRE((int64_t{block_size} * num_heads * full_dim) % 8 == 0 &&
                  (int64_t{block_size} * num_heads * (head_size / 2)) % 8 == 0,
              "%s: block_size * num_heads * full_dim must be a multiple of 8", fn);
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (kvq_status s = check_device(fn)) return s;
  // the launcher sets the index dividers for the groups-per-thread it picks
  const kvq::PerHeadArgs a{key,          value,     key_stride_t, key_stride_h, value_stride_t,
                           value_stride_h, slot_mapping, num_tokens, num_heads, head_size,
                           const_cast<uint8_t*>(kv_cache), num_pages * block_size, block_size,
                           layout, k_scale, v_scale, d_status,
                           kvq::FastDiv::make(static_cast<uint32_t>(block_size)), {}, {}, {}};
  return launched(fn, launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

kvq_status kvq_write_nvfp4_ds_mla(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                                  int64_t k_pe_stride, const int64_t* slot_mapping,
                                  int64_t num_tokens, uint8_t* kv_cache, int64_t num_blocks,
                                  int32_t block_size, int64_t block_stride, int64_t entry_stride,
                                  int32_t* d_status, kvq_stream_t stream) {
  return write_common("kvq_write_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                      kvq::launch_write_nvfp4_ds_mla, kv_c, kv_c_stride, k_pe, k_pe_stride,
                      slot_mapping, num_tokens, kv_cache, num_blocks, block_size, block_stride,
                      entry_stride, d_status, stream);
}

kvq_status kvq_write_fp8_ds_mla(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                                int64_t k_pe_stride, const int64_t* slot_mapping,
                                int64_t num_tokens, uint8_t* kv_cache, int64_t num_blocks,
                                int32_t block_size, int64_t block_stride, int64_t entry_stride,
                                int32_t* d_status, kvq_stream_t stream) {
  return write_common("kvq_write_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                      kvq::launch_write_fp8_ds_mla, kv_c, kv_c_stride, k_pe, k_pe_stride,
                      slot_mapping, num_tokens, kv_cache, num_blocks, block_size, block_stride,
                      entry_stride, d_status, stream);
}

kvq_status kvq_gather_upconvert_nvfp4_ds_mla(
    const uint8_t* src_cache, int64_t num_blocks, int32_t block_size, int64_t block_stride,
    int64_t entry_stride, void* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts, int32_t batch_size,
    int32_t* d_status, kvq_stream_t stream) {
  return gather_common("kvq_gather_upconvert_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                       kvq::launch_gather_nvfp4_ds_mla, src_cache, num_blocks, block_size,
                       block_stride, entry_stride, dst, dst_stride, num_out_tokens, block_table,
                       block_table_stride, block_table_width, workspace_starts, seq_starts,
                       batch_size, d_status, stream);
}

kvq_status kvq_gather_upconvert_fp8_ds_mla(
    const uint8_t* src_cache, int64_t num_blocks, int32_t block_size, int64_t block_stride,
    int64_t entry_stride, void* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts, int32_t batch_size,
    int32_t* d_status, kvq_stream_t stream) {
  return gather_common("kvq_gather_upconvert_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                       kvq::launch_gather_fp8_ds_mla, src_cache, num_blocks, block_size,
                       block_stride, entry_stride, dst, dst_stride, num_out_tokens, block_table,
                       block_table_stride, block_table_width, workspace_starts, seq_starts,
                       batch_size, d_status, stream);
}

kvq_status kvq_reshape_and_cache_nvfp4(const void* key, const void* value, int64_t key_stride_t,
                                       int64_t key_stride_h, int64_t value_stride_t,
                                       int64_t value_stride_h, const int64_t* slot_mapping,
                                       int64_t num_tokens, int32_t num_heads, int32_t head_size,
                                       uint8_t* kv_cache, int64_t num_pages, int32_t block_size,
                                       int32_t layout, const float* k_scale, const float* v_scale,
                                       int32_t* d_status, kvq_stream_t stream) {
  return per_head_common("kvq_reshape_and_cache_nvfp4", false, kvq::launch_reshape_and_cache_nvfp4,
                         key, value, key_stride_t, key_stride_h, value_stride_t, value_stride_h,
                         slot_mapping, num_tokens, num_heads, head_size, kv_cache, num_pages,
                         block_size, layout, k_scale, v_scale, d_status, stream);
}

kvq_status kvq_dequant_nvfp4_per_head(const uint8_t* kv_cache, int64_t num_pages,
                                      int32_t block_size, int32_t layout, int32_t num_heads,
                                      int32_t head_size, const int64_t* slot_mapping, int64_t num_tokens,
                                      const float* k_scale, const float* v_scale, void* key_out,
                                      int64_t key_stride_t, int64_t key_stride_h, void* value_out,
                                      int64_t value_stride_t, int64_t value_stride_h,
                                      int32_t* d_status, kvq_stream_t stream) {
  return per_head_common("kvq_dequant_nvfp4_per_head", true, kvq::launch_dequant_nvfp4_per_head,
                         key_out, value_out, key_stride_t, key_stride_h, value_stride_t,
                         value_stride_h, slot_mapping, num_tokens, num_heads, head_size, kv_cache,
                         num_pages, block_size, layout, k_scale, v_scale, d_status, stream);
}

kvq_status kvq_req_index_to_global_slot(const int32_t* req_id, int64_t num_req_ids,
                                        const int32_t* token_indices, int64_t num_tokens,
                                        int32_t topk, int64_t token_indices_stride,
                                        const int32_t* block_table, int64_t block_table_stride,
                                        int32_t block_table_width, int32_t num_requests,
                                        int32_t block_size, int64_t num_blocks, int32_t* out,
                                        int64_t out_stride, int32_t* d_status,
                                        kvq_stream_t stream) {
  const char* fn = "kvq_req_index_to_global_slot";
  KVQ_REQUIRE(num_tokens >= 0 && topk >= 0, "%s: num_tokens / topk < 0", fn);
  KVQ_REQUIRE(num_req_ids == num_tokens,
              "%s: req_id has %lld entries but token_indices has %lld rows", fn,
              static_cast<long long>(num_req_ids), static_cast<long long>(num_tokens));
  if (num_tokens == 0 || topk == 0) return ok();
  KVQ_REQUIRE(num_tokens < (int64_t{1} << 31) && topk <= (1 << 24),
              "%s: num_tokens must be below 2^31 and topk at most 2^24", fn);   // grid x / y
  KVQ_REQUIRE(req_id != nullptr && token_indices != nullptr && out != nullptr && block_table != nullptr,
              "%s: req_id, token_indices, block_table and out must be non-NULL", fn);
  KVQ_REQUIRE(aligned(req_id, 4) && aligned(token_indices, 4) && aligned(out, 4) && aligned(block_table, 4),
              "%s: int32 arrays must be 4-byte aligned", fn);
  KVQ_REQUIRE(token_indices_stride >= topk && out_stride >= topk,
              "%s: row strides must be >= topk", fn);
  KVQ_REQUIRE(num_requests > 0 && block_table_width > 0 && block_table_stride >= block_table_width,
              "%s: need num_requests > 0, block_table_width > 0, stride >= width", fn);
  KVQ_REQUIRE(block_size > 0 && num_blocks > 0 && num_blocks <= INT32_MAX / block_size,
              "%s: num_blocks * block_size must fit an int32 slot", fn);
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (kvq_status s = check_device(fn)) return s;
  const kvq::IndexArgs a{req_id,        token_indices, token_indices_stride, num_tokens,
                         topk,          block_table,   block_table_stride,   block_table_width,
                         num_requests,  block_size,    num_blocks,           out,
                         out_stride,    d_status,
                         kvq::FastDiv::make(static_cast<uint32_t>(block_size))};
  return launched(fn, kvq::launch_req_index_to_global_slot(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

kvq_status attention_common(
    const char* fn, int64_t entry_bytes, cudaError_t (*launch)(const kvq::AttentionArgs&, cudaStream_t),
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    float softmax_scale, void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse,
    int64_t lse_stride_t, int32_t* d_status, kvq_stream_t stream, int32_t num_splits = 1,
    void* workspace = nullptr, int64_t workspace_bytes = 0) {
  KVQ_REQUIRE(num_tokens >= 0 && topk >= 0, "%s: num_tokens / topk < 0", fn);
  KVQ_REQUIRE(num_splits >= 1 && num_splits <= KVQ_ATTN_MAX_SPLITS, "%s: num_splits must be in [1, %d] (got %d)",
              fn, KVQ_ATTN_MAX_SPLITS, num_splits);
  if (num_tokens == 0) return ok();
  KVQ_REQUIRE(num_tokens * num_splits < (int64_t{1} << 30), "%s: num_tokens x num_splits too large", fn);
  KVQ_REQUIRE(num_heads >= 1 && num_heads <= 128, "%s: num_heads must be in [1, 128] (got %d)", fn,
              num_heads);
  KVQ_REQUIRE(q != nullptr && out != nullptr, "%s: q and out must be non-NULL", fn);
  KVQ_REQUIRE(aligned(q, 16) && aligned(out, 16), "%s: q and out must be 16-byte aligned", fn);
  KVQ_REQUIRE(q_stride_h >= KVQ_WORKSPACE_DIM && q_stride_h % 8 == 0 && q_stride_t % 8 == 0 &&
                  q_stride_t >= 0,
              "%s: q strides must be multiples of 8 elements with head stride >= 576", fn);
  KVQ_REQUIRE(out_stride_h >= KVQ_MLA_NOPE_DIM && out_stride_h % 8 == 0 && out_stride_t % 8 == 0 &&
                  out_stride_t >= (num_heads - 1) * out_stride_h + KVQ_MLA_NOPE_DIM,
              "%s: out strides must be multiples of 8 elements and rows must not overlap "
              "(head stride >= 512, token stride >= (num_heads - 1) * head stride + 512)", fn);
  KVQ_REQUIRE(lse == nullptr || (aligned(lse, 4) && lse_stride_t >= num_heads),
              "%s: lse must be 4-byte aligned with token stride >= num_heads", fn);
  KVQ_REQUIRE(topk == 0 || (indices != nullptr && aligned(indices, 4) && indices_stride >= topk),
              "%s: indices must be non-NULL, 4-byte aligned, with stride >= topk", fn);
  KVQ_REQUIRE(softmax_scale == softmax_scale && softmax_scale > -3.0e38f && softmax_scale < 3.0e38f,
              "%s: softmax_scale must be finite", fn);
  if (kvq_status s = check_mla_cache(fn, kv_cache, num_blocks, block_size, block_stride,
                                     entry_stride, entry_bytes))
    return s;
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (num_splits > 1) {
    const int64_t need = kvq_sparse_mla_attention_split_workspace_bytes(num_tokens, num_heads, num_splits);
    KVQ_REQUIRE(workspace != nullptr && aligned(workspace, 16) && workspace_bytes >= need,
                "%s: workspace must be non-NULL, 16-byte aligned and at least %lld bytes (got %lld)", fn,
                static_cast<long long>(need), static_cast<long long>(workspace_bytes));
  }
  if (kvq_status s = check_device(fn)) return s;
  kvq::AttentionArgs a{};
  a.num_splits = num_splits;
  if (num_splits > 1) {
    // whole 64-key tiles per range; ranges past the list are empty
    const int64_t tiles = (int64_t{topk} + 63) / 64;
    a.split_keys = static_cast<int32_t>((tiles + num_splits - 1) / num_splits * 64);
    const int64_t rows = num_tokens * num_heads * num_splits;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = static_cast<float*>(workspace) + rows * KVQ_MLA_NOPE_DIM;
  }
  a.q = q;
  a.q_stride_t = q_stride_t;
  a.q_stride_h = q_stride_h;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.indices = indices;
  a.indices_stride = indices_stride;
  a.topk = topk;
  a.cache = kv_cache;
  a.num_blocks = num_blocks;
  a.num_slots = num_blocks * block_size;
  a.block_size = block_size;
  a.block_div = kvq::FastDiv::make(static_cast<uint32_t>(block_size));
  a.block_stride = block_stride;
  a.entry_stride = entry_stride;
  a.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  a.out = out;
  a.out_stride_t = out_stride_t;
  a.out_stride_h = out_stride_h;
  a.lse = lse;
  a.lse_stride_t = lse_stride_t;
  a.status = d_status;
  return launched(fn, launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status prefill_common(
    const char* fn, int64_t entry_bytes, cudaError_t (*launch)(const kvq::AttentionArgs&, cudaStream_t),
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t* d_status,
    kvq_stream_t stream, int32_t num_splits = 1,
    int32_t max_context_len = 0, void* workspace = nullptr, int64_t workspace_bytes = 0) {
  KVQ_REQUIRE(num_tokens >= 0 && batch_size >= 0 && max_query_len >= 0,
              "%s: num_tokens, batch_size and max_query_len must be >= 0", fn);
  if (num_tokens == 0 || batch_size == 0 || max_query_len == 0) return ok();
  KVQ_REQUIRE(num_heads >= 1, "%s: num_heads must be >= 1 (got %d)", fn, num_heads);
  KVQ_REQUIRE(batch_size <= 65535, "%s: batch_size must be at most 65535 (grid.y)", fn);
  KVQ_REQUIRE(int64_t{max_query_len} * num_heads < (int64_t{1} << 31) && num_tokens < (int64_t{1} << 31),
              "%s: max_query_len * num_heads and num_tokens must stay below 2^31", fn);
  KVQ_REQUIRE(q != nullptr && out != nullptr, "%s: q and out must be non-NULL", fn);
  KVQ_REQUIRE(aligned(q, 16) && aligned(out, 16), "%s: q and out must be 16-byte aligned", fn);
  KVQ_REQUIRE(q_stride_h >= KVQ_WORKSPACE_DIM && q_stride_h % 8 == 0 && q_stride_t % 8 == 0 &&
                  q_stride_t >= 0,
              "%s: q strides must be multiples of 8 elements with head stride >= 576", fn);
  KVQ_REQUIRE(out_stride_h >= KVQ_MLA_NOPE_DIM && out_stride_h % 8 == 0 && out_stride_t % 8 == 0 &&
                  out_stride_t >= (num_heads - 1) * out_stride_h + KVQ_MLA_NOPE_DIM,
              "%s: out strides must be multiples of 8 elements and rows must not overlap "
              "(head stride >= 512, token stride >= (num_heads - 1) * head stride + 512)", fn);
  KVQ_REQUIRE(lse == nullptr || (aligned(lse, 4) && lse_stride_t >= num_heads),
              "%s: lse must be 4-byte aligned with token stride >= num_heads", fn);
  KVQ_REQUIRE(query_start != nullptr && context_lens != nullptr && block_table != nullptr,
              "%s: query_start, context_lens and block_table must be non-NULL", fn);
  KVQ_REQUIRE(aligned(query_start, 4) && aligned(context_lens, 4) && aligned(block_table, 4),
              "%s: int32 arrays must be 4-byte aligned", fn);
  KVQ_REQUIRE(block_table_width > 0 && block_table_stride >= block_table_width,
              "%s: need block_table_width > 0 and block_table_stride >= block_table_width", fn);
  KVQ_REQUIRE(softmax_scale == softmax_scale && softmax_scale > -3.0e38f && softmax_scale < 3.0e38f,
              "%s: softmax_scale must be finite", fn);
  if (kvq_status s = check_mla_cache(fn, kv_cache, num_blocks, block_size, block_stride,
                                     entry_stride, entry_bytes))
    return s;
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  KVQ_REQUIRE(num_splits >= 1 && num_splits <= KVQ_ATTN_MAX_SPLITS, "%s: num_splits must be in [1, %d] (got %d)",
              fn, KVQ_ATTN_MAX_SPLITS, num_splits);
  if (num_splits > 1) {
    const int64_t need = kvq_sparse_mla_attention_split_workspace_bytes(num_tokens, num_heads, num_splits);
    KVQ_REQUIRE(max_context_len >= 0, "%s: max_context_len must be >= 0", fn);
    KVQ_REQUIRE((int64_t{max_query_len} * num_heads + 127) / 128 * 2 * num_splits < (int64_t{1} << 31),
                "%s: too many CTAs (grid.x)", fn);
    KVQ_REQUIRE(workspace != nullptr && aligned(workspace, 16) && need >= 0 && workspace_bytes >= need,
                "%s: workspace must be non-NULL, 16-byte aligned and at least %lld bytes (got %lld)", fn,
                static_cast<long long>(need), static_cast<long long>(workspace_bytes));
  }
  if (kvq_status s = check_device(fn)) return s;
  kvq::AttentionArgs a{};
  a.num_splits = num_splits;
  if (num_splits > 1) {
    // whole 64-key tiles per range, sized from max_context_len; the last range
    // of a request also takes every position past num_splits ranges
    const int64_t tiles = (int64_t{max_context_len} + 63) / 64;
    a.split_keys = static_cast<int32_t>(std::max<int64_t>(1, (tiles + num_splits - 1) / num_splits) * 64);
    const int64_t rows = num_tokens * num_heads * num_splits;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = static_cast<float*>(workspace) + rows * KVQ_MLA_NOPE_DIM;
  }
  a.q = q;
  a.q_stride_t = q_stride_t;
  a.q_stride_h = q_stride_h;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.head_div = kvq::FastDiv::make(static_cast<uint32_t>(num_heads));
  a.query_start = query_start;
  a.context_lens = context_lens;
  a.block_table = block_table;
  a.block_table_stride = block_table_stride;
  a.block_table_width = block_table_width;
  a.batch_size = batch_size;
  a.max_query_len = max_query_len;
  a.cache = kv_cache;
  a.num_blocks = num_blocks;
  a.num_slots = num_blocks * block_size;
  a.block_size = block_size;
  a.block_div = kvq::FastDiv::make(static_cast<uint32_t>(block_size));
  a.block_stride = block_stride;
  a.entry_stride = entry_stride;
  a.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  a.out = out;
  a.out_stride_t = out_stride_t;
  a.out_stride_h = out_stride_h;
  a.lse = lse;
  a.lse_stride_t = lse_stride_t;
  a.status = d_status;
  return launched(fn, launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

kvq_status kvq_prefill_mla_attention_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t* d_status,
    kvq_stream_t stream) {
  return prefill_common("kvq_prefill_mla_attention_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                        kvq::launch_prefill_mla_attention_nvfp4, q, q_stride_t, q_stride_h, num_tokens, num_heads,
                        query_start, context_lens, batch_size, max_query_len, block_table, block_table_stride,
                        block_table_width, kv_cache, num_blocks, block_size, block_stride, entry_stride,
                        softmax_scale, out, out_stride_t, out_stride_h, lse, lse_stride_t, d_status, stream);
}

kvq_status kvq_prefill_mla_attention_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t* d_status,
    kvq_stream_t stream) {
  return prefill_common("kvq_prefill_mla_attention_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                        kvq::launch_prefill_mla_attention_fp8, q, q_stride_t, q_stride_h, num_tokens, num_heads,
                        query_start, context_lens, batch_size, max_query_len, block_table, block_table_stride,
                        block_table_width, kv_cache, num_blocks, block_size, block_stride, entry_stride,
                        softmax_scale, out, out_stride_t, out_stride_h, lse, lse_stride_t, d_status, stream);
}

kvq_status kvq_prefill_mla_attention_split_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t,
    int32_t max_context_len, int32_t num_splits, void* workspace, int64_t workspace_bytes, int32_t* d_status,
    kvq_stream_t stream) {
  return prefill_common("kvq_prefill_mla_attention_split_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                        num_splits > 1 ? kvq::launch_prefill_mla_attention_split_nvfp4
                                       : kvq::launch_prefill_mla_attention_nvfp4,
                        q, q_stride_t, q_stride_h, num_tokens, num_heads, query_start, context_lens, batch_size,
                        max_query_len, block_table, block_table_stride, block_table_width, kv_cache, num_blocks,
                        block_size, block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h, lse,
                        lse_stride_t, d_status, stream, num_splits, max_context_len, workspace, workspace_bytes);
}

kvq_status kvq_prefill_mla_attention_split_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, int32_t batch_size, int32_t max_query_len,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale,
    void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t,
    int32_t max_context_len, int32_t num_splits, void* workspace, int64_t workspace_bytes, int32_t* d_status,
    kvq_stream_t stream) {
  return prefill_common("kvq_prefill_mla_attention_split_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                        num_splits > 1 ? kvq::launch_prefill_mla_attention_split_fp8
                                       : kvq::launch_prefill_mla_attention_fp8,
                        q, q_stride_t, q_stride_h, num_tokens, num_heads, query_start, context_lens, batch_size,
                        max_query_len, block_table, block_table_stride, block_table_width, kv_cache, num_blocks,
                        block_size, block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h, lse,
                        lse_stride_t, d_status, stream, num_splits, max_context_len, workspace, workspace_bytes);
}

kvq_status kvq_prefill_mla_attention_workspace(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens, const int32_t* workspace_starts, int32_t batch_size,
    int32_t max_query_len, const void* workspace, int64_t workspace_stride, int64_t workspace_rows,
    float softmax_scale, void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t,
    int32_t* d_status, kvq_stream_t stream) {
  const char* fn = "kvq_prefill_mla_attention_workspace";
  KVQ_REQUIRE(num_tokens >= 0 && batch_size >= 0 && max_query_len >= 0 && workspace_rows >= 0,
              "%s: num_tokens, batch_size, max_query_len and workspace_rows must be >= 0", fn);
  if (num_tokens == 0 || batch_size == 0 || max_query_len == 0) return ok();
  KVQ_REQUIRE(num_heads >= 1, "%s: num_heads must be >= 1 (got %d)", fn, num_heads);
  KVQ_REQUIRE(batch_size <= 65535, "%s: batch_size must be at most 65535 (grid.y)", fn);
  KVQ_REQUIRE(int64_t{max_query_len} * num_heads < (int64_t{1} << 31) && num_tokens < (int64_t{1} << 31),
              "%s: max_query_len * num_heads and num_tokens must stay below 2^31", fn);
  KVQ_REQUIRE(q != nullptr && out != nullptr, "%s: q and out must be non-NULL", fn);
  KVQ_REQUIRE(aligned(q, 16) && aligned(out, 16), "%s: q and out must be 16-byte aligned", fn);
  KVQ_REQUIRE(q_stride_h >= KVQ_WORKSPACE_DIM && q_stride_h % 8 == 0 && q_stride_t % 8 == 0 && q_stride_t >= 0,
              "%s: q strides must be multiples of 8 elements with head stride >= 576", fn);
  KVQ_REQUIRE(out_stride_h >= KVQ_MLA_NOPE_DIM && out_stride_h % 8 == 0 && out_stride_t % 8 == 0 &&
                  out_stride_t >= (num_heads - 1) * out_stride_h + KVQ_MLA_NOPE_DIM,
              "%s: out strides must be multiples of 8 elements and rows must not overlap", fn);
  KVQ_REQUIRE(lse == nullptr || (aligned(lse, 4) && lse_stride_t >= num_heads),
              "%s: lse must be 4-byte aligned with token stride >= num_heads", fn);
  KVQ_REQUIRE(query_start != nullptr && context_lens != nullptr && workspace_starts != nullptr,
              "%s: query_start, context_lens and workspace_starts must be non-NULL", fn);
  KVQ_REQUIRE(aligned(query_start, 4) && aligned(context_lens, 4) && aligned(workspace_starts, 4),
              "%s: int32 arrays must be 4-byte aligned", fn);
  KVQ_REQUIRE(workspace_rows == 0 || (workspace != nullptr && aligned(workspace, 16)),
              "%s: workspace must be non-NULL and 16-byte aligned", fn);
  KVQ_REQUIRE(workspace_stride >= KVQ_WORKSPACE_DIM && workspace_stride % 8 == 0 && workspace_rows < (int64_t{1} << 31),
              "%s: workspace row stride must be >= 576 and a multiple of 8 elements, workspace_rows below 2^31", fn);
  KVQ_REQUIRE(softmax_scale == softmax_scale && softmax_scale > -3.0e38f && softmax_scale < 3.0e38f,
              "%s: softmax_scale must be finite", fn);
  KVQ_REQUIRE(d_status == nullptr || aligned(d_status, 4), "%s: d_status misaligned", fn);
  if (kvq_status st = check_device(fn)) return st;
  kvq::AttentionArgs a{};
  a.q = q;
  a.q_stride_t = q_stride_t;
  a.q_stride_h = q_stride_h;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.head_div = kvq::FastDiv::make(static_cast<uint32_t>(num_heads));
  a.query_start = query_start;
  a.context_lens = context_lens;
  a.batch_size = batch_size;
  a.max_query_len = max_query_len;
  a.ws = workspace;
  a.ws_stride = workspace_stride;
  a.ws_rows = workspace_rows;
  a.ws_starts = workspace_starts;
  a.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  a.out = out;
  a.out_stride_t = out_stride_t;
  a.out_stride_h = out_stride_h;
  a.lse = lse;
  a.lse_stride_t = lse_stride_t;
  a.status = d_status;
  if (workspace_rows == 0) a.ws = q;   // no rows: every context must be empty; the map's one row is never read
  return launched(fn, kvq::launch_prefill_mla_attention_workspace(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_sparse_mla_attention_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    float softmax_scale, void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse,
    int64_t lse_stride_t, int32_t* d_status, kvq_stream_t stream) {
  return attention_common("kvq_sparse_mla_attention_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                          kvq::launch_sparse_mla_attention_nvfp4, q, q_stride_t, q_stride_h, num_tokens,
                          num_heads, indices, indices_stride, topk, kv_cache, num_blocks, block_size,
                          block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h, lse,
                          lse_stride_t, d_status, stream);
}

kvq_status kvq_sparse_mla_attention_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache,
    int64_t num_blocks, int32_t block_size, int64_t block_stride, int64_t entry_stride,
    float softmax_scale, void* out, int64_t out_stride_t, int64_t out_stride_h, float* lse,
    int64_t lse_stride_t, int32_t* d_status, kvq_stream_t stream) {
  return attention_common("kvq_sparse_mla_attention_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                          kvq::launch_sparse_mla_attention_fp8, q, q_stride_t, q_stride_h, num_tokens,
                          num_heads, indices, indices_stride, topk, kv_cache, num_blocks, block_size,
                          block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h, lse,
                          lse_stride_t, d_status, stream);
}

int64_t kvq_sparse_mla_attention_split_workspace_bytes(int64_t num_tokens, int32_t num_heads, int32_t num_splits) {
  constexpr int64_t kRowBytes = (KVQ_MLA_NOPE_DIM + 2) * 4;
  if (num_tokens < 0 || num_heads < 1 || num_splits < 1 ||
      num_tokens > (INT64_MAX - 15) / kRowBytes / num_heads / num_splits)
    return -1;
  const int64_t rows = num_tokens * num_heads * num_splits;
  return (rows * kRowBytes + 15) / 16 * 16;
}

kvq_status kvq_sparse_mla_attention_split_nvfp4_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache, int64_t num_blocks,
    int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale, void* out,
    int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t num_splits,
    void* workspace, int64_t workspace_bytes, int32_t* d_status, kvq_stream_t stream) {
  return attention_common("kvq_sparse_mla_attention_split_nvfp4_ds_mla", KVQ_NVFP4_DS_MLA_ENTRY_BYTES,
                          num_splits > 1 ? kvq::launch_sparse_mla_attention_split_nvfp4
                                         : kvq::launch_sparse_mla_attention_nvfp4,
                          q, q_stride_t, q_stride_h, num_tokens, num_heads, indices, indices_stride, topk, kv_cache,
                          num_blocks, block_size, block_stride, entry_stride, softmax_scale, out, out_stride_t,
                          out_stride_h, lse, lse_stride_t, d_status, stream, num_splits, workspace, workspace_bytes);
}

kvq_status kvq_sparse_mla_attention_split_fp8_ds_mla(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache, int64_t num_blocks,
    int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale, void* out,
    int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t num_splits,
    void* workspace, int64_t workspace_bytes, int32_t* d_status, kvq_stream_t stream) {
  return attention_common("kvq_sparse_mla_attention_split_fp8_ds_mla", KVQ_FP8_DS_MLA_ENTRY_BYTES,
                          num_splits > 1 ? kvq::launch_sparse_mla_attention_split_fp8
                                         : kvq::launch_sparse_mla_attention_fp8,
                          q, q_stride_t, q_stride_h, num_tokens, num_heads, indices, indices_stride, topk, kv_cache,
                          num_blocks, block_size, block_stride, entry_stride, softmax_scale, out, out_stride_t,
                          out_stride_h, lse, lse_stride_t, d_status, stream, num_splits, workspace, workspace_bytes);
}

kvq_status kvq_selftest_convert(uint32_t first_bits, int64_t count, uint8_t* e4m3_lo,
                                uint8_t* e4m3_hi, uint8_t* e2m1_lo, uint8_t* e2m1_hi,
                                uint16_t* bf16_out, kvq_stream_t stream) {
  const char* fn = "kvq_selftest_convert";
  KVQ_REQUIRE(count >= 0 && count <= (int64_t{1} << 32), "%s: count out of range", fn);
  if (count == 0) return ok();
  int num_sms = 0;
  if (kvq_status s = check_device(fn, &num_sms)) return s;
  return launched(fn, kvq::launch_selftest_convert(first_bits, count, e4m3_lo, e4m3_hi, e2m1_lo,
                                                   e2m1_hi, bf16_out, num_sms,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The split-key decode without a caller workspace
// ---------------------------------------------------------------------------
//
// Some callers cannot allocate device memory when they call in: a serving
// engine that reserved the GPU's memory for its own pools at start-up (a
// cudaMalloc would fail, or take memory its key-value cache counts on), or
// host code on a latency-critical path, where an allocation can synchronise
// the device and stall its other streams.  For them the partial results of
// the split-key decode live in one fixed array that the library holds on
// every GPU that loads it, for the life of the process.

// Device storage of the partial results; in host code this name is only a
// stand-in for the symbol, never a device address.
static __device__ __align__(256) unsigned char g_split_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of g_split_scratch on the current device, looked up on
// the first call made with that device current and kept.
cudaError_t split_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

kvq_status kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, int64_t num_tokens, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk, const uint8_t* kv_cache, int64_t num_blocks,
    int32_t block_size, int64_t block_stride, int64_t entry_stride, float softmax_scale, void* out,
    int64_t out_stride_t, int64_t out_stride_h, float* lse, int64_t lse_stride_t, int32_t num_splits,
    int32_t* d_status, kvq_stream_t stream) {
  const char* fn = "kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc";
  KVQ_REQUIRE(num_tokens >= 0 && num_heads >= 1 && num_splits >= 1,
              "%s: num_tokens must be >= 0, num_heads and num_splits >= 1", fn);
  const int64_t need =
      num_splits > 1 ? kvq_sparse_mla_attention_split_workspace_bytes(num_tokens, num_heads, num_splits) : 0;
  KVQ_REQUIRE(need >= 0 && need <= KVQ_NOALLOC_SCRATCH_BYTES,
              "%s: %lld tokens x %d heads x %d key ranges need %lld bytes of partial results, more than the "
              "library's fixed %lld-byte array holds (at most %lld (token, head, range) rows); use fewer ranges "
              "or tokens, or kvq_sparse_mla_attention_split_nvfp4_ds_mla with a workspace",
              fn, static_cast<long long>(num_tokens), num_heads, num_splits, static_cast<long long>(need),
              static_cast<long long>(KVQ_NOALLOC_SCRATCH_BYTES),
              static_cast<long long>(KVQ_NOALLOC_SCRATCH_BYTES / ((KVQ_MLA_NOPE_DIM + 2) * 4)));
  void* scratch = nullptr;
  if (need > 0) {
    if (kvq_status st = check_device(fn)) return st;
    const cudaError_t e = split_scratch(&scratch);
    if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: the scratch array's address: %s", fn, cudaGetErrorString(e));
  }
  return kvq_sparse_mla_attention_split_nvfp4_ds_mla(
      q, q_stride_t, q_stride_h, num_tokens, num_heads, indices, indices_stride, topk, kv_cache, num_blocks,
      block_size, block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h, lse, lse_stride_t,
      num_splits, scratch, need > 0 ? KVQ_NOALLOC_SCRATCH_BYTES : 0, d_status, stream);
}

const char* kvq_last_error_string(void) { return g_last_error.c_str(); }

int32_t kvq_version(void) { return 100; }

}  // extern "C"
