// kvq_index.cu -- sparse-decode index conversion: per decode token i and
// top-k slot k, position token_indices[i][k] of request req_id[i] -> global
// cache slot block_table[r][p / block_size] * block_size + p % block_size,
// -1 for unused (negative) positions and for anything out of range.
//
// One thread per 4 consecutive (token, k) pairs (16-byte loads and stores;
// one per pair when rows are not 16-byte aligned): int32 reads and writes,
// coalesced along k; the block-table read is a gather into a small,
// L2-resident table.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

// Slot of position p of request r, or -1 (with a status bit when out of range).
__device__ __forceinline__ int32_t global_slot(const IndexArgs& a, int32_t r, int32_t p) {
  if (p < 0) return -1;
  const uint32_t col = a.block_div.div(static_cast<uint32_t>(p));
  if (r >= 0 && r < a.num_requests && col < static_cast<uint32_t>(a.block_table_width)) {
    const int32_t blk = __ldg(a.block_table + static_cast<int64_t>(r) * a.block_table_stride + col);
    if (blk >= 0 && blk < a.num_blocks)
      return blk * a.block_size + static_cast<int32_t>(static_cast<uint32_t>(p) - col * a.block_div.d);
  }
  report(a.status, KVQ_STATUS_BAD_INDEX);
  return -1;
}

// kVec consecutive positions per thread (16-byte loads and stores when 4).
template <int kVec>
__global__ void __launch_bounds__(kThreads) req_index_to_global_slot_kernel(const IndexArgs a) {
  const uint32_t idx = blockIdx.x * kThreads + threadIdx.x;      // < 2^32 - 256 (host check)
  const uint32_t i = a.topk_div.div(idx);                        // topk_div divides by topk / kVec
  if (i >= a.num_tokens) return;
  const uint32_t k = (idx - i * a.topk_div.d) * kVec;
  const int32_t r = __ldg(a.req_id + i);
  const int32_t* src = a.token_indices + static_cast<int64_t>(i) * a.token_indices_stride + k;
  int32_t* dst = a.out + static_cast<int64_t>(i) * a.out_stride + k;
  if constexpr (kVec == 4) {
    const int4 p = __ldcs(reinterpret_cast<const int4*>(src));
    *reinterpret_cast<int4*>(dst) =
        make_int4(global_slot(a, r, p.x), global_slot(a, r, p.y), global_slot(a, r, p.z), global_slot(a, r, p.w));
  } else {
    *dst = global_slot(a, r, __ldg(src));
  }
}

}  // namespace

cudaError_t launch_req_index_to_global_slot(const IndexArgs& a, cudaStream_t stream) {
  // four positions per thread when rows are 16-byte aligned and topk % 4 == 0
  const bool vec = a.topk % 4 == 0 && a.token_indices_stride % 4 == 0 && a.out_stride % 4 == 0 &&
                   reinterpret_cast<uintptr_t>(a.token_indices) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.out) % 16 == 0;
  IndexArgs b = a;
  const int per_thread = vec ? 4 : 1;
  b.topk_div = FastDiv::make(static_cast<uint32_t>(a.topk / per_thread));
  const int64_t threads = a.num_tokens * (a.topk / per_thread);
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  if (vec)
    req_index_to_global_slot_kernel<4><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(b);
  else
    req_index_to_global_slot_kernel<1><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace kvq
