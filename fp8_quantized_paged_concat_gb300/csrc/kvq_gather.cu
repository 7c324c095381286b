// kvq_gather.cu -- prefill gather-upconvert of quantized MLA pages into a
// contiguous bf16 [T, 576] workspace (nvfp4_ds_mla and fp8_ds_mla).
//
// Design (GB300): small CTAs, warps independent of each other.  A CTA first
// stages workspace_starts in shared memory (one coalesced load; batches
// larger than kMaxSmemBatch search global memory instead) -- the only CTA
// barrier.  Each warp then owns kRowsPerWarp consecutive workspace rows: lane
// r < kRowsPerWarp resolves row r (binary search over the staged starts, then
// seq_starts and block_table) into the byte offset of its source entry and
// the warp shares the offsets by shuffle.  NoPE: one row at a time across the
// warp, lane l converting 16 values (one NVFP4 group / a 16-byte fp8 slice)
// and storing 32 contiguous bytes, so each row is one 1024-byte segment; the
// loads of all the warp's rows are issued before any conversion.  RoPE: 8
// lanes per row.  Consecutive rows of a request read consecutive entries of a
// page, so reads stay in runs of up to block_size entries.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

#ifndef KVQ_GATHER_WARPS_PER_BLOCK
#define KVQ_GATHER_WARPS_PER_BLOCK 4
#endif
#ifndef KVQ_GATHER_ROWS_PER_WARP
#define KVQ_GATHER_ROWS_PER_WARP 4
#endif
#ifndef KVQ_GATHER_MIN_BLOCKS
#define KVQ_GATHER_MIN_BLOCKS 12
#endif
constexpr int kWarps = KVQ_GATHER_WARPS_PER_BLOCK;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = KVQ_GATHER_ROWS_PER_WARP;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
constexpr int kMinBlocks = KVQ_GATHER_MIN_BLOCKS;
constexpr int kRopeItems = kRowsPerWarp * 8 / 32;          // RoPE pieces per lane (4 rows each)
constexpr int kMaxSmemBatch = 1024;                         // starts staged in smem
static_assert(kRowsPerWarp <= 32 && (kRowsPerWarp * 8) % 32 == 0, "row tiling");

// Largest b with starts[b] <= w (starts non-decreasing), or -1.
template <typename Load>
__device__ __forceinline__ int find_request(int64_t w, int batch, Load starts) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(starts(mid)) <= w) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

// Byte offset of the source entry of workspace row w, or -1.
__device__ __forceinline__ int64_t resolve_row(int64_t w, const GatherArgs& a, const int32_t* s_ws) {
  const int b = a.batch_size <= kMaxSmemBatch
                    ? find_request(w, a.batch_size, [&](int i) { return s_ws[i]; })
                    : find_request(w, a.batch_size, [&](int i) { return __ldg(a.workspace_starts + i); });
  if (b < 0) {
    report(a.status, KVQ_STATUS_BAD_BATCH);
    return -1;
  }
  const int64_t ws_b = a.batch_size <= kMaxSmemBatch ? s_ws[b] : __ldg(a.workspace_starts + b);
  const int64_t p = static_cast<int64_t>(__ldg(a.seq_starts + b)) + (w - ws_b);
  // 0 <= p < 2^32: an int32 start plus a row offset below 2^31
  if (p < 0) {
    report(a.status, KVQ_STATUS_BAD_INDEX);
    return -1;
  }
  const uint32_t col = a.block_div.div(static_cast<uint32_t>(p));
  const uint32_t off = static_cast<uint32_t>(p) - col * static_cast<uint32_t>(a.block_size);
  if (col >= static_cast<uint32_t>(a.block_table_width)) {
    report(a.status, KVQ_STATUS_BAD_INDEX);
    return -1;
  }
  const int64_t blk = __ldg(a.block_table + b * a.block_table_stride + col);
  if (blk < 0 || blk >= a.num_blocks) {
    report(a.status, KVQ_STATUS_BAD_INDEX);
    return -1;
  }
  return blk * a.block_stride + static_cast<int64_t>(off) * a.entry_stride;
}

// Stages workspace_starts in shared memory (CTA 0 also validates them when a
// status word is given), then gives every lane the source offsets of its
// warp's rows: offs[k] is row w0 + k's offset (or -1), also held by lane k in
// `mine`.  Returns w0.
__device__ __forceinline__ int64_t resolve_warp_rows(const GatherArgs& a, int32_t* s_ws,
                                                     int64_t (&offs)[kRowsPerWarp], int64_t& mine) {
  if (a.batch_size <= kMaxSmemBatch)
    for (int b = threadIdx.x; b < a.batch_size; b += kThreads) s_ws[b] = __ldg(a.workspace_starts + b);
  if (a.status != nullptr && blockIdx.x == 0) {
    for (int b = threadIdx.x; b < a.batch_size; b += kThreads) {
      const int32_t v = __ldg(a.workspace_starts + b);
      const bool bad = v < 0 || v > a.num_out ||
                       (b + 1 < a.batch_size && v > __ldg(a.workspace_starts + b + 1));
      if (bad) report(a.status, KVQ_STATUS_BAD_BATCH);
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
  mine = -1;
  if (lane < kRowsPerWarp && w0 + lane < a.num_out) mine = resolve_row(w0 + lane, a, s_ws);
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) offs[k] = __shfl_sync(kFull, mine, k);
  return w0;
}

// 8 e4m3 codes -> 8 bf16 (exact), as 4 packed words.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 c) {
  const float2 f0 = __half22float2(e4m3x2_to_half2(c.x));
  const float2 f1 = __half22float2(e4m3x2_to_half2(c.x >> 16));
  const float2 f2 = __half22float2(e4m3x2_to_half2(c.y));
  const float2 f3 = __half22float2(e4m3x2_to_half2(c.y >> 16));
  return make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y), pack_bf16x2(f2.x, f2.y),
                    pack_bf16x2(f3.x, f3.y));
}

// ---------------------------------------------------------------------------
// nvfp4_ds_mla
// ---------------------------------------------------------------------------
template <bool kWide>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gather_nvfp4_ds_mla_kernel(const GatherArgs a) {
  __shared__ int32_t s_ws[kMaxSmemBatch];
  int64_t offs[kRowsPerWarp], mine;
  const int64_t w0 = resolve_warp_rows(a, s_ws, offs, mine);
  // RoPE piece k of this lane: row (lane / 8) + 4k, piece lane % 8
  int64_t roff[kRopeItems];
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) roff[k] = __shfl_sync(kFull, mine, ((threadIdx.x & 31) >> 3) + 4 * k);
  const int lane = threadIdx.x & 31;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);

  // Issue every load of the warp's rows first: NoPE group `lane` (8 bytes and
  // its scale byte) and RoPE pieces (8 bytes each).
  uint2 q[kRowsPerWarp];
  uint32_t sf[kRowsPerWarp];
  uint2 rp[kRopeItems];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    if (offs[k] >= 0) {
      q[k] = ld_stream8(a.cache + offs[k] + 8 * lane);
      sf[k] = ld_byte(a.cache + offs[k] + kNvSfOff + lane);
    }
  }
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k)
    if (roff[k] >= 0) rp[k] = ld_stream8(a.cache + roff[k] + kNvRopeOff + 8 * (lane & 7));

#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    if (offs[k] < 0) continue;
    const float scale = e4m3_to_float(sf[k]);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = (i < 4 ? q[k].x : q[k].y) >> (8 * (i & 3));
      const float2 v = __half22float2(e2m1x2_to_half2(byte));
      o[i] = pack_bf16x2(v.x * scale, v.y * scale);     // exact products
    }
    store32<kWide>(dst + (w0 + k) * a.dst_stride + 16 * lane, make_uint4(o[0], o[1], o[2], o[3]),
                   make_uint4(o[4], o[5], o[6], o[7]));
  }
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) {
    if (roff[k] < 0) continue;
    const int r = (lane >> 3) + 4 * k;
    st16(dst + (w0 + r) * a.dst_stride + kNopeDim + 8 * (lane & 7), e4m3x8_to_bf16x8(rp[k]));
  }
}

// ---------------------------------------------------------------------------
// fp8_ds_mla
// ---------------------------------------------------------------------------
template <bool kWide>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gather_fp8_ds_mla_kernel(const GatherArgs a) {
  __shared__ int32_t s_ws[kMaxSmemBatch];
  int64_t offs[kRowsPerWarp], mine;
  const int64_t w0 = resolve_warp_rows(a, s_ws, offs, mine);
  // RoPE piece k of this lane: row (lane / 8) + 4k, piece lane % 8
  int64_t roff[kRopeItems];
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) roff[k] = __shfl_sync(kFull, mine, ((threadIdx.x & 31) >> 3) + 4 * k);
  const int lane = threadIdx.x & 31;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);

  // NoPE: lane converts bytes [16 lane, 16 lane + 16) with scale lane / 8;
  // RoPE: bf16 bits copied, 8 pieces of 16 bytes per row.
  uint4 q[kRowsPerWarp];
  float s[kRowsPerWarp];
  uint4 rp[kRopeItems];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    if (offs[k] >= 0) {
      q[k] = ld_stream16(a.cache + offs[k] + 16 * lane);
      s[k] = __uint_as_float(__ldg(reinterpret_cast<const unsigned int*>(
          a.cache + offs[k] + kF8ScaleOff + 4 * (lane >> 3))));
    }
  }
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k)
    if (roff[k] >= 0) rp[k] = ld_stream16(a.cache + roff[k] + kF8RopeOff + 16 * (lane & 7));

#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    if (offs[k] < 0) continue;
    const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v0 = __half22float2(e4m3x2_to_half2(w[i]));
      const float2 v1 = __half22float2(e4m3x2_to_half2(w[i] >> 16));
      const float2 p0 = fmul2(v0, make_float2(s[k], s[k]));   // packed pairs, each rounded as __fmul_rn
      const float2 p1 = fmul2(v1, make_float2(s[k], s[k]));
      o[2 * i] = pack_bf16x2(p0.x, p0.y);
      o[2 * i + 1] = pack_bf16x2(p1.x, p1.y);
    }
    store32<kWide>(dst + (w0 + k) * a.dst_stride + 16 * lane, make_uint4(o[0], o[1], o[2], o[3]),
                   make_uint4(o[4], o[5], o[6], o[7]));
  }
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) {
    if (roff[k] < 0) continue;
    const int r = (lane >> 3) + 4 * k;
    st16(dst + (w0 + r) * a.dst_stride + kNopeDim + 8 * (lane & 7), rp[k]);
  }
}

// Workspace rows that start on 32-byte boundaries are written with 32-byte
// stores.
bool wide_rows(const GatherArgs& a) {
  return reinterpret_cast<uintptr_t>(a.dst) % 32 == 0 && (a.dst_stride * 2) % 32 == 0;
}

cudaError_t launch_gather(void (*kernel)(GatherArgs), const GatherArgs& a, cudaStream_t stream) {
  const int64_t blocks = (a.num_out + kRowsPerBlock - 1) / kRowsPerBlock;
  kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_nvfp4_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(wide_rows(a) ? gather_nvfp4_ds_mla_kernel<true> : gather_nvfp4_ds_mla_kernel<false>,
                       a, stream);
}

cudaError_t launch_gather_fp8_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(wide_rows(a) ? gather_fp8_ds_mla_kernel<true> : gather_fp8_ds_mla_kernel<false>,
                       a, stream);
}

}  // namespace kvq
