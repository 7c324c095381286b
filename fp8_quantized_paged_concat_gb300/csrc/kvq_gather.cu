// kvq_gather.cu -- prefill gather-upconvert of quantized MLA pages into a
// contiguous bf16 [T, 576] workspace (nvfp4_ds_mla and fp8_ds_mla).
//
// Design (GB300): a persistent grid of small CTAs (every SM filled to its
// occupancy), warps independent of each other.  A CTA stages
// workspace_starts in shared memory once (one coalesced load; batches larger
// than kMaxSmemBatch search global memory instead) -- its only barrier.  Each
// warp then walks groups of kRowsPerWarp consecutive workspace rows with a
// grid stride.  For a group, lane r < kRowsPerWarp resolves row r (binary
// search over the staged starts, then seq_starts and block_table) into the
// byte offset of its source entry, and the warp shares the offsets by
// shuffle.  The loop is software-pipelined: the group's entry loads are
// issued, then the NEXT group's rows are resolved while those loads are in
// flight, then the group is converted and stored.  NoPE: one row at a time
// across the warp, lane l converting 16 values (one NVFP4 group / a 16-byte
// fp8 slice) and storing 32 contiguous bytes, so a row is one 1024-byte
// segment.  RoPE: 8 lanes per row.  Consecutive rows of a request read
// consecutive entries of a page, so reads stay in runs of up to block_size
// entries.
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
#ifndef KVQ_GATHER_NVFP4_MIN_BLOCKS
#define KVQ_GATHER_NVFP4_MIN_BLOCKS 12
#endif
#ifndef KVQ_GATHER_FP8_MIN_BLOCKS
#define KVQ_GATHER_FP8_MIN_BLOCKS 8
#endif
constexpr int kWarps = KVQ_GATHER_WARPS_PER_BLOCK;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = KVQ_GATHER_ROWS_PER_WARP;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
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

// Stages workspace_starts in shared memory; CTA 0 also validates them when a
// status word is given.
__device__ __forceinline__ void stage_starts(const GatherArgs& a, int32_t* s_ws) {
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

// Source offsets of one group: offs[k] for the NoPE of row k, roff[k] for
// RoPE piece k of this lane (row lane / 8 + 4k, piece lane % 8).
struct GroupOffsets {
  int64_t offs[kRowsPerWarp];
  int64_t roff[kRopeItems];

  __device__ __forceinline__ void share(int64_t mine) {
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) offs[k] = __shfl_sync(kFull, mine, k);
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k)
      roff[k] = __shfl_sync(kFull, mine, ((threadIdx.x & 31) >> 3) + 4 * k);
  }
};

// nvfp4_ds_mla: per lane, NoPE group `lane` (8 bytes + scale byte) of each
// row and 8-byte RoPE pieces.
struct Nvfp4Rows {
  static constexpr int kMinBlocks = KVQ_GATHER_NVFP4_MIN_BLOCKS;
  uint2 q[kRowsPerWarp];
  uint32_t sf[kRowsPerWarp];
  uint2 rp[kRopeItems];

  __device__ __forceinline__ void load(const uint8_t* cache, const GroupOffsets& o, int lane) {
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (o.offs[k] >= 0) {
        q[k] = ld_stream8(cache + o.offs[k] + 8 * lane);
        sf[k] = ld_byte(cache + o.offs[k] + kNvSfOff + lane);
      }
    }
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k)
      if (o.roff[k] >= 0) rp[k] = ld_stream8(cache + o.roff[k] + kNvRopeOff + 8 * (lane & 7));
  }

  __device__ __forceinline__ void store(__nv_bfloat16* dst, int64_t stride, int64_t w0,
                                        const GroupOffsets& o, int lane) const {
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (o.offs[k] < 0) continue;
      const float scale = e4m3_to_float(sf[k]);
      uint32_t v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = (i < 4 ? q[k].x : q[k].y) >> (8 * (i & 3));
        const float2 f = __half22float2(e2m1x2_to_half2(byte));
        v[i] = pack_bf16x2(f.x * scale, f.y * scale);     // exact products
      }
      __nv_bfloat16* out = dst + (w0 + k) * stride + 16 * lane;
      st16(out, make_uint4(v[0], v[1], v[2], v[3]));
      st16(out + 8, make_uint4(v[4], v[5], v[6], v[7]));
    }
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k) {
      if (o.roff[k] < 0) continue;
      const int r = (lane >> 3) + 4 * k;
      st16(dst + (w0 + r) * stride + kNopeDim + 8 * (lane & 7), e4m3x8_to_bf16x8(rp[k]));
    }
  }
};

// fp8_ds_mla: per lane, NoPE bytes [16 lane, 16 lane + 16) with scale lane / 8,
// and 16-byte pieces of bf16 RoPE (copied).
struct Fp8Rows {
  static constexpr int kMinBlocks = KVQ_GATHER_FP8_MIN_BLOCKS;
  uint4 q[kRowsPerWarp];
  float s[kRowsPerWarp];
  uint4 rp[kRopeItems];

  __device__ __forceinline__ void load(const uint8_t* cache, const GroupOffsets& o, int lane) {
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (o.offs[k] >= 0) {
        q[k] = ld_stream16(cache + o.offs[k] + 16 * lane);
        s[k] = __uint_as_float(__ldg(reinterpret_cast<const unsigned int*>(
            cache + o.offs[k] + kF8ScaleOff + 4 * (lane >> 3))));
      }
    }
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k)
      if (o.roff[k] >= 0) rp[k] = ld_stream16(cache + o.roff[k] + kF8RopeOff + 16 * (lane & 7));
  }

  __device__ __forceinline__ void store(__nv_bfloat16* dst, int64_t stride, int64_t w0,
                                        const GroupOffsets& o, int lane) const {
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (o.offs[k] < 0) continue;
      const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
      uint32_t v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f0 = __half22float2(e4m3x2_to_half2(w[i]));
        const float2 f1 = __half22float2(e4m3x2_to_half2(w[i] >> 16));
        v[2 * i] = pack_bf16x2(__fmul_rn(f0.x, s[k]), __fmul_rn(f0.y, s[k]));
        v[2 * i + 1] = pack_bf16x2(__fmul_rn(f1.x, s[k]), __fmul_rn(f1.y, s[k]));
      }
      __nv_bfloat16* out = dst + (w0 + k) * stride + 16 * lane;
      st16(out, make_uint4(v[0], v[1], v[2], v[3]));
      st16(out + 8, make_uint4(v[4], v[5], v[6], v[7]));
    }
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k) {
      if (o.roff[k] < 0) continue;
      const int r = (lane >> 3) + 4 * k;
      st16(dst + (w0 + r) * stride + kNopeDim + 8 * (lane & 7), rp[k]);
    }
  }
};

template <class Rows>
__global__ void __launch_bounds__(kThreads, Rows::kMinBlocks) gather_kernel(const GatherArgs a) {
  __shared__ int32_t s_ws[kMaxSmemBatch];
  stage_starts(a, s_ws);
  const int lane = threadIdx.x & 31;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dst);
  const int64_t num_groups = (a.num_out + kRowsPerWarp - 1) / kRowsPerWarp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);

  // lane r < kRowsPerWarp holds the source offset of row r of group g
  auto resolve_group = [&](int64_t group) -> int64_t {
    const int64_t w = group * kRowsPerWarp + lane;
    return (group < num_groups && lane < kRowsPerWarp && w < a.num_out) ? resolve_row(w, a, s_ws) : -1;
  };
  int64_t mine = resolve_group(g);
  while (g < num_groups) {                       // warp-uniform
    GroupOffsets o;
    o.share(mine);
    Rows rows;
    rows.load(a.cache, o, lane);
    const int64_t next = g + stride;
    mine = resolve_group(next);                  // overlaps the loads in flight
    rows.store(dst, a.dst_stride, g * kRowsPerWarp, o, lane);
    g = next;
  }
}

cudaError_t launch_gather(const void* kernel_ptr, void (*kernel)(GatherArgs), const GatherArgs& a,
                          cudaStream_t stream) {
  const int64_t ctas_of_work = (a.num_out + kRowsPerBlock - 1) / kRowsPerBlock;
  const int grid = persistent_grid(kernel_ptr, kThreads, ctas_of_work);
  kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_nvfp4_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(reinterpret_cast<const void*>(gather_kernel<Nvfp4Rows>), gather_kernel<Nvfp4Rows>,
                       a, stream);
}

cudaError_t launch_gather_fp8_ds_mla(const GatherArgs& a, cudaStream_t stream) {
  return launch_gather(reinterpret_cast<const void*>(gather_kernel<Fp8Rows>), gather_kernel<Fp8Rows>,
                       a, stream);
}

}  // namespace kvq
