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
// Rows wider than the staging limit read the table from global memory.  A
// power-of-two block size (the usual case) splits a position with a shift and
// a mask; the checks are branch-free and a warp reports a bad index once.
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
#ifndef KVQ_INDEX_TOKENS
#define KVQ_INDEX_TOKENS 1
#endif
constexpr int kThreads = KVQ_INDEX_THREADS;
constexpr int kLoads = KVQ_INDEX_LOADS;       // independent accesses per thread and token
constexpr int kTokens = KVQ_INDEX_TOKENS;     // tokens per CTA
constexpr int kMaxStagedWidth = 12288;        // 48 KB of int32: no opt-in shared memory needed

// Block-table column and offset of position p >= 0: a shift and a mask when
// the block size is a power of two, else the multiply-high divider.
template <bool kPow2>
__device__ __forceinline__ uint32_t column_of(const IndexArgs& a, uint32_t p, uint32_t& off) {
  if constexpr (kPow2) {
    off = p & (a.block_div.d - 1);
    return p >> a.block_shift;
  } else {
    const uint32_t col = a.block_div.div(p);
    off = p - col * a.block_div.d;
    return col;
  }
}

// Slot of position p given the request's table row (or -1; row == nullptr
// marks an out-of-range request).  A position >= 0 that cannot be resolved
// sets `bad` (reported once per warp by the caller).
template <bool kPow2, typename Row>
__device__ __forceinline__ int32_t global_slot(const IndexArgs& a, Row row, int32_t p, int32_t num_blocks, bool& bad) {
  // branch-free: a negative (unused) position gives -1 and is not an error
  uint32_t off;
  const uint32_t col = column_of<kPow2>(a, static_cast<uint32_t>(p), off);   // huge for p < 0
  const int32_t blk = (row != nullptr && col < static_cast<uint32_t>(a.block_table_width)) ? row[col] : -1;
  const bool ok = blk >= 0 && blk < num_blocks;
  bad |= !ok && p >= 0;
  return ok ? blk * a.block_size + static_cast<int32_t>(off) : -1;
}

template <int kVec, bool kStaged, bool kPow2>
__global__ void __launch_bounds__(kThreads) req_index_to_global_slot_kernel(const IndexArgs a) {
  extern __shared__ int32_t s_rows[];                             // [kTokens][block_table_width]
  // kTokens tokens per CTA (consecutive), kLoads accesses of kVec positions
  // per thread and token, kThreads * kVec apart (coalesced).  The position
  // loads do not depend on the request, so all of them are issued first and
  // their latency overlaps the block-table staging.
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTokens;
  const int64_t k0 = (static_cast<int64_t>(blockIdx.y) * kThreads * kLoads + threadIdx.x) * kVec;
  using Vec = typename std::conditional<kVec == 4, int4, int32_t>::type;
  Vec p[kTokens][kLoads];
#pragma unroll
  for (int j = 0; j < kTokens; ++j) {
    if (i0 + j >= a.num_tokens) continue;
    const int32_t* src = a.token_indices + (i0 + j) * a.token_indices_stride;
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int64_t k = k0 + u * kThreads * kVec;
      if (k < a.topk) p[j][u] = __ldcs(reinterpret_cast<const Vec*>(src + k));
    }
  }
  const int32_t* rows[kTokens];
#pragma unroll
  for (int j = 0; j < kTokens; ++j) {
    rows[j] = nullptr;
    if (i0 + j >= a.num_tokens) continue;
    const int32_t r = __ldg(a.req_id + i0 + j);
    if (r >= 0 && r < a.num_requests) {
      const int32_t* g_row = a.block_table + static_cast<int64_t>(r) * a.block_table_stride;
      if constexpr (kStaged) {
        int32_t* s_row = s_rows + j * a.block_table_width;
#pragma unroll 4
        for (int c = threadIdx.x; c < a.block_table_width; c += kThreads) s_row[c] = __ldg(g_row + c);
        rows[j] = s_row;
      } else {
        rows[j] = g_row;
      }
    }
  }
  if constexpr (kStaged) __syncthreads();
  bool bad = false;
  const int32_t nb = static_cast<int32_t>(a.num_blocks);         // < 2^31 (host check)
#pragma unroll
  for (int j = 0; j < kTokens; ++j) {
    if (i0 + j >= a.num_tokens) continue;
    int32_t* dst = a.out + (i0 + j) * a.out_stride;
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int64_t k = k0 + u * kThreads * kVec;
      if (k >= a.topk) continue;
      if constexpr (kVec == 4) {
        __stcs(reinterpret_cast<int4*>(dst + k),
               make_int4(global_slot<kPow2>(a, rows[j], p[j][u].x, nb, bad),
                         global_slot<kPow2>(a, rows[j], p[j][u].y, nb, bad),
                         global_slot<kPow2>(a, rows[j], p[j][u].z, nb, bad),
                         global_slot<kPow2>(a, rows[j], p[j][u].w, nb, bad)));
      } else {
        __stcs(dst + k, global_slot<kPow2>(a, rows[j], p[j][u], nb, bad));
      }
    }
  }
  if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
}

template <int kVec, bool kPow2>
cudaError_t launch(const IndexArgs& a, cudaStream_t stream) {
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kLoads * kVec;
  const dim3 grid(static_cast<unsigned>((a.num_tokens + kTokens - 1) / kTokens),
                  static_cast<unsigned>((a.topk + per_cta - 1) / per_cta));
  if (a.block_table_width <= kMaxStagedWidth / kTokens)
    req_index_to_global_slot_kernel<kVec, true, kPow2>
        <<<grid, kThreads, kTokens * a.block_table_width * sizeof(int32_t), stream>>>(a);
  else
    req_index_to_global_slot_kernel<kVec, false, kPow2><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_req_index_to_global_slot(const IndexArgs& a, cudaStream_t stream) {
  // four positions per thread when rows are 16-byte aligned and topk % 4 == 0
  const bool vec = a.topk % 4 == 0 && a.token_indices_stride % 4 == 0 && a.out_stride % 4 == 0 &&
                   reinterpret_cast<uintptr_t>(a.token_indices) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.out) % 16 == 0;
  const bool pow2 = (a.block_size & (a.block_size - 1)) == 0;
  if (pow2) {
    IndexArgs b = a;
    b.block_shift = 0;
    while ((1 << b.block_shift) < a.block_size) ++b.block_shift;
    return vec ? launch<4, true>(b, stream) : launch<1, true>(b, stream);
  }
  return vec ? launch<4, false>(a, stream) : launch<1, false>(a, stream);
}

}  // namespace kvq
