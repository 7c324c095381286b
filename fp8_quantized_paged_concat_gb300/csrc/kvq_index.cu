// kvq_index.cu -- sparse-decode index conversion: per decode token i and
// top-k slot k, position token_indices[i][k] of request req_id[i] -> global
// cache slot block_table[r][p / block_size] * block_size + p % block_size,
// -1 for unused (negative) positions and for anything out of range.
//
// One CTA per (token, chunk of 2048 positions): every position of a token
// belongs to the same request, so the CTA stages that request's block-table
// row in shared memory once and resolves its positions there (a 4-byte
// gather per position from L2 would move a 32-byte sector each).  Threads
// take 4 x 4 consecutive positions (16-byte loads and stores, all four loads
// in flight together; 4 x 1 position when rows are not 16-byte aligned).
// Rows wider than the staging limit read the table from global memory.
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

// Launch shape (compile-time tuning knobs; the defaults are the measured best).
#ifndef KVQ_INDEX_THREADS
#define KVQ_INDEX_THREADS 128
#endif
#ifndef KVQ_INDEX_LOADS
#define KVQ_INDEX_LOADS 4
#endif
constexpr int kThreads = KVQ_INDEX_THREADS;
constexpr int kLoads = KVQ_INDEX_LOADS;       // independent accesses per thread
constexpr int kMaxStagedWidth = 12288;        // 48 KB of int32: no opt-in shared memory needed

// Slot of position p given the request's table row (or -1, with a status
// bit when out of range; row == nullptr marks an out-of-range request).
template <typename Row>
__device__ __forceinline__ int32_t global_slot(const IndexArgs& a, Row row, int32_t p) {
  if (p < 0) return -1;
  const uint32_t col = a.block_div.div(static_cast<uint32_t>(p));
  if (row != nullptr && col < static_cast<uint32_t>(a.block_table_width)) {
    const int32_t blk = row[col];
    if (blk >= 0 && blk < a.num_blocks)
      return blk * a.block_size + static_cast<int32_t>(static_cast<uint32_t>(p) - col * a.block_div.d);
  }
  report(a.status, KVQ_STATUS_BAD_INDEX);
  return -1;
}

template <int kVec, bool kStaged>
__global__ void __launch_bounds__(kThreads) req_index_to_global_slot_kernel(const IndexArgs a) {
  extern __shared__ int32_t s_row[];
  const int64_t i = blockIdx.x;                                   // token
  // kLoads accesses of kVec positions per thread, kThreads * kVec apart
  // (coalesced).  They do not depend on the request, so they are issued
  // first and their latency overlaps the block-table staging.
  const int64_t k0 = (static_cast<int64_t>(blockIdx.y) * kThreads * kLoads + threadIdx.x) * kVec;
  const int32_t* src = a.token_indices + i * a.token_indices_stride;
  int32_t* dst = a.out + i * a.out_stride;
  using Vec = typename std::conditional<kVec == 4, int4, int32_t>::type;
  Vec p[kLoads];
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int64_t k = k0 + u * kThreads * kVec;
    if (k < a.topk) p[u] = __ldcs(reinterpret_cast<const Vec*>(src + k));
  }
  const int32_t r = __ldg(a.req_id + i);
  const bool valid_req = r >= 0 && r < a.num_requests;
  const int32_t* g_row = valid_req ? a.block_table + static_cast<int64_t>(r) * a.block_table_stride : nullptr;
  if constexpr (kStaged) {
    if (valid_req) {
#pragma unroll 4
      for (int c = threadIdx.x; c < a.block_table_width; c += kThreads) s_row[c] = __ldg(g_row + c);
    }
    __syncthreads();
  }
  const int32_t* row = valid_req ? (kStaged ? s_row : g_row) : nullptr;
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int64_t k = k0 + u * kThreads * kVec;
    if (k >= a.topk) continue;
    if constexpr (kVec == 4) {
      __stcs(reinterpret_cast<int4*>(dst + k),
             make_int4(global_slot(a, row, p[u].x), global_slot(a, row, p[u].y), global_slot(a, row, p[u].z),
                       global_slot(a, row, p[u].w)));
    } else {
      __stcs(dst + k, global_slot(a, row, p[u]));
    }
  }
}

template <int kVec>
cudaError_t launch(const IndexArgs& a, cudaStream_t stream) {
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kLoads * kVec;
  const dim3 grid(static_cast<unsigned>(a.num_tokens), static_cast<unsigned>((a.topk + per_cta - 1) / per_cta));
  if (a.block_table_width <= kMaxStagedWidth)
    req_index_to_global_slot_kernel<kVec, true>
        <<<grid, kThreads, a.block_table_width * sizeof(int32_t), stream>>>(a);
  else
    req_index_to_global_slot_kernel<kVec, false><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_req_index_to_global_slot(const IndexArgs& a, cudaStream_t stream) {
  // four positions per thread when rows are 16-byte aligned and topk % 4 == 0
  const bool vec = a.topk % 4 == 0 && a.token_indices_stride % 4 == 0 && a.out_stride % 4 == 0 &&
                   reinterpret_cast<uintptr_t>(a.token_indices) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.out) % 16 == 0;
  return vec ? launch<4>(a, stream) : launch<1>(a, stream);
}

}  // namespace kvq
