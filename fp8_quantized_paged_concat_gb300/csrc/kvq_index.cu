// kvq_index.cu -- sparse-decode index conversion: per decode token i and
// top-k slot k, position token_indices[i][k] of request req_id[i] -> global
// cache slot block_table[r][p / block_size] * block_size + p % block_size,
// -1 for unused (negative) positions and for anything out of range.
//
// One thread per (token, k): int32 reads and writes, fully coalesced along k;
// the block-table read is a gather into a small, L2-resident table.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) req_index_to_global_slot_kernel(const IndexArgs a) {
  const uint32_t idx = blockIdx.x * kThreads + threadIdx.x;      // < 2^32 - 256 (host check)
  const uint32_t i = a.topk_div.div(idx);
  if (i >= a.num_tokens) return;
  const uint32_t k = idx - i * a.topk_div.d;
  const int32_t p = __ldg(a.token_indices + static_cast<int64_t>(i) * a.token_indices_stride + k);
  int32_t slot = -1;
  if (p >= 0) {
    const int32_t r = __ldg(a.req_id + i);
    const uint32_t col = a.block_div.div(static_cast<uint32_t>(p));
    bool ok = r >= 0 && r < a.num_requests && col < static_cast<uint32_t>(a.block_table_width);
    if (ok) {
      const int32_t blk = __ldg(a.block_table + static_cast<int64_t>(r) * a.block_table_stride + col);
      ok = blk >= 0 && blk < a.num_blocks;
      if (ok) slot = blk * a.block_size + static_cast<int32_t>(static_cast<uint32_t>(p) - col * a.block_div.d);
    }
    if (!ok) report(a.status, KVQ_STATUS_BAD_INDEX);
  }
  a.out[static_cast<int64_t>(i) * a.out_stride + k] = slot;
}

}  // namespace

cudaError_t launch_req_index_to_global_slot(const IndexArgs& a, cudaStream_t stream) {
  const int64_t threads = a.num_tokens * a.topk;
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  req_index_to_global_slot_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
