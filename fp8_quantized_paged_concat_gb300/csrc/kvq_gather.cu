// kvq_gather.cu -- prefill gather-upconvert of quantized MLA pages into a
// contiguous bf16 [T, 576] workspace (nvfp4_ds_mla and fp8_ds_mla).
//
// Design (GB300): a CTA owns kRowsPerBlock consecutive workspace rows.  First
// kRowsPerBlock threads resolve one row each (binary search of
// workspace_starts, then seq_starts and block_table) into the byte offset of
// its source entry, kept in shared memory; the whole CTA then streams the
// entries.  NoPE: one warp per row, lane l converts 16 values (one NVFP4
// group / a 16-byte fp8 slice) and stores 32 contiguous bytes, so a warp
// writes a 1024-byte row segment.  RoPE: 8 lanes per row.  Each warp issues
// the loads of all its rows before converting any of them.  Consecutive rows
// of one request read consecutive entries of a page, so reads stay in runs of
// up to block_size entries.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kRowsPerBlock = 64;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kRowsPerBlock / kWarps;   // NoPE rows per warp
constexpr int kRopeItems = kRowsPerBlock * 8 / kThreads;  // RoPE pieces per thread

// Byte offset of the source entry of workspace row w, or -1.
__device__ __forceinline__ int64_t resolve_row(int64_t w, const GatherArgs& a) {
  // largest b with workspace_starts[b] <= w (binary search; ws non-decreasing)
  int lo = 0, hi = a.batch_size;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(__ldg(a.workspace_starts + mid)) <= w) lo = mid + 1; else hi = mid;
  }
  const int b = lo - 1;
  if (b < 0) {
    report(a.status, KVQ_STATUS_BAD_BATCH);
    return -1;
  }
  const int64_t p = static_cast<int64_t>(__ldg(a.seq_starts + b)) +
                    (w - static_cast<int64_t>(__ldg(a.workspace_starts + b)));
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

// Fills s_off for this CTA's rows; CTA 0 also checks that workspace_starts is
// non-decreasing inside [0, num_out] when a status word is given.
__device__ __forceinline__ void resolve_rows(const GatherArgs& a, int64_t w0, int64_t* s_off) {
  if (threadIdx.x < kRowsPerBlock) {
    const int64_t w = w0 + threadIdx.x;
    s_off[threadIdx.x] = w < a.num_out ? resolve_row(w, a) : -1;
  }
  if (a.status != nullptr && blockIdx.x == 0) {
    for (int b = threadIdx.x; b < a.batch_size; b += kThreads) {
      const int32_t v = __ldg(a.workspace_starts + b);
      const bool bad = v < 0 || v > a.num_out ||
                       (b + 1 < a.batch_size && v > __ldg(a.workspace_starts + b + 1));
      if (bad) report(a.status, KVQ_STATUS_BAD_BATCH);
    }
  }
  __syncthreads();
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
__global__ void __launch_bounds__(kThreads) gather_nvfp4_ds_mla_kernel(const GatherArgs a) {
  __shared__ int64_t s_off[kRowsPerBlock];
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  resolve_rows(a, w0, s_off);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);

  // NoPE: warp handles rows warp, warp + 8, ...; lane = NVFP4 group.
  uint2 q[kRowsPerWarp];
  uint32_t sf[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int64_t off = s_off[warp + kWarps * k];
    if (off >= 0) {
      q[k] = ld_stream8(a.cache + off + 8 * lane);
      sf[k] = ld_byte(a.cache + off + kNvSfOff + lane);
    }
  }
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = warp + kWarps * k;
    if (s_off[r] < 0) continue;
    const float scale = e4m3_to_float(sf[k]);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = (i < 4 ? q[k].x : q[k].y) >> (8 * (i & 3));
      const float2 v = __half22float2(e2m1x2_to_half2(byte));
      o[i] = pack_bf16x2(v.x * scale, v.y * scale);     // exact products
    }
    __nv_bfloat16* out = dst + (w0 + r) * a.dst_stride + 16 * lane;
    st16(out, make_uint4(o[0], o[1], o[2], o[3]));
    st16(out + 8, make_uint4(o[4], o[5], o[6], o[7]));
  }

  // RoPE: 8 pieces of 8 values per row.
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) {
    const int item = threadIdx.x + kThreads * k;
    const int r = item >> 3, piece = item & 7;
    const int64_t off = s_off[r];
    if (off < 0) continue;
    const uint2 c = ld_stream8(a.cache + off + kNvRopeOff + 8 * piece);
    st16(dst + (w0 + r) * a.dst_stride + kNopeDim + 8 * piece, e4m3x8_to_bf16x8(c));
  }
}

// ---------------------------------------------------------------------------
// fp8_ds_mla
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) gather_fp8_ds_mla_kernel(const GatherArgs a) {
  __shared__ int64_t s_off[kRowsPerBlock];
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock;
  resolve_rows(a, w0, s_off);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);

  // NoPE: lane converts bytes [16 lane, 16 lane + 16), scale lane / 8.
  uint4 q[kRowsPerWarp];
  float s[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int64_t off = s_off[warp + kWarps * k];
    if (off >= 0) {
      q[k] = ld_stream16(a.cache + off + 16 * lane);
      s[k] = __uint_as_float(__ldg(reinterpret_cast<const unsigned int*>(
          a.cache + off + kF8ScaleOff + 4 * (lane >> 3))));
    }
  }
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = warp + kWarps * k;
    if (s_off[r] < 0) continue;
    const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v0 = __half22float2(e4m3x2_to_half2(w[i]));
      const float2 v1 = __half22float2(e4m3x2_to_half2(w[i] >> 16));
      o[2 * i] = pack_bf16x2(__fmul_rn(v0.x, s[k]), __fmul_rn(v0.y, s[k]));
      o[2 * i + 1] = pack_bf16x2(__fmul_rn(v1.x, s[k]), __fmul_rn(v1.y, s[k]));
    }
    __nv_bfloat16* out = dst + (w0 + r) * a.dst_stride + 16 * lane;
    st16(out, make_uint4(o[0], o[1], o[2], o[3]));
    st16(out + 8, make_uint4(o[4], o[5], o[6], o[7]));
  }

  // RoPE: bf16 bits copied, 8 pieces of 16 bytes per row.
#pragma unroll
  for (int k = 0; k < kRopeItems; ++k) {
    const int item = threadIdx.x + kThreads * k;
    const int r = item >> 3, piece = item & 7;
    const int64_t off = s_off[r];
    if (off < 0) continue;
    st16(dst + (w0 + r) * a.dst_stride + kNopeDim + 8 * piece,
         ld_stream16(a.cache + off + kF8RopeOff + 16 * piece));
  }
}

cudaError_t launch_gather(void (*kernel)(GatherArgs), const GatherArgs& a, cudaStream_t stream) {
  const int64_t blocks = (a.num_out + kRowsPerBlock - 1) / kRowsPerBlock;
  kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_nvfp4_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(gather_nvfp4_ds_mla_kernel, a, stream);
}

cudaError_t launch_gather_fp8_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(gather_fp8_ds_mla_kernel, a, stream);
}

}  // namespace kvq
