// kvq_write.cu -- MLA cache writes (concat_and_cache) for the 352-byte
// nvfp4_ds_mla entry and the 656-byte fp8_ds_mla entry.
//
// Design (GB300): one warp per token, kTokensPerWarp tokens per warp with all
// of their loads issued before any conversion, so each resident warp keeps
// kTokensPerWarp x 1152 bytes of HBM reads in flight.  Lane l owns the 16
// NoPE values of group l (32 contiguous bytes: one e4m3 scale, 8 output
// bytes), so the group amax needs no shuffle.  Stores are warp-contiguous:
// 256 B of packed NoPE, 64 B of RoPE and 32 B of scales per 352-byte entry,
// each a whole number of 32-byte sectors when the entry is 32-byte aligned,
// so L2 never has to read the line before writing it.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

// Launch shape (compile-time tuning knobs; the defaults are the measured best).
#ifndef KVQ_WRITE_WARPS_PER_BLOCK
#define KVQ_WRITE_WARPS_PER_BLOCK 4
#endif
#ifndef KVQ_WRITE_TOKENS_PER_WARP
#define KVQ_WRITE_TOKENS_PER_WARP 4
#endif
#ifndef KVQ_WRITE_SMALL_BATCH
#define KVQ_WRITE_SMALL_BATCH 65536   // below this many tokens: one token per warp
#endif
#ifndef KVQ_WRITE_MIN_BLOCKS
#define KVQ_WRITE_MIN_BLOCKS 8
#endif
constexpr int kWarpsPerBlock = KVQ_WRITE_WARPS_PER_BLOCK;
constexpr int kTokensPerWarp = KVQ_WRITE_TOKENS_PER_WARP;
constexpr int64_t kSmallBatch = KVQ_WRITE_SMALL_BATCH;
constexpr int kSmallMinBlocks = 16;       // one token per warp: a decode batch in one wave
constexpr int kMinBlocks = KVQ_WRITE_MIN_BLOCKS;

// The 8 packed bf16 pairs of one lane's 16 NoPE values, as fp32.
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&x)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
}

// amax over 16 bf16 values held as 8 packed words: exact, in bf16 pairs.
__device__ __forceinline__ float amax16(const uint4& a, const uint4& b) {
  __nv_bfloat162 m = __hmax2(__hmax2(abs_bf16x2(a.x), abs_bf16x2(a.y)),
                             __hmax2(abs_bf16x2(a.z), abs_bf16x2(a.w)));
  m = __hmax2(m, __hmax2(__hmax2(abs_bf16x2(b.x), abs_bf16x2(b.y)),
                         __hmax2(abs_bf16x2(b.z), abs_bf16x2(b.w))));
  return fmaxf(__low2float(m), __high2float(m));
}

// amax / 448 rounded to nearest even for a bf16 magnitude amax > 0, without a
// division: Markstein's correction of amax * RN(1/448) (see quotient2());
// equal to the IEEE quotient for every positive finite bf16 value, checked
// exhaustively in tests/c/fp8_quotient_check.c.
__device__ __forceinline__ float tile_scale(float amax) {
  constexpr float kInv448 = 1.0f / 448.0f;
  const float q0 = __fmul_rn(amax, kInv448);
  return __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), kInv448, q0);
}

// x / s rounded to nearest even, for |x| <= 448 s (a value of its own tile),
// from s2 = s * f and inv = RN(1 / s2), f a power of two that keeps s2 at or
// above 2^-64 (x * f is exact).  Markstein's theorem (P. Markstein, IBM J.
// Res. Dev. 34(1), 1990): q0 = RN(x * inv) is within an ulp of the quotient,
// the remainder x - q0 * s2 is exact in one fused multiply-add, and
// RN(q0 + remainder * inv) is the correctly rounded quotient (no overflow
// or harmful underflow here: s2 >= 2^-64 and |quotient| <= 448; quotients
// below 2^-11, where the remainder might not be exact, encode to an e4m3
// zero of the sign of x whichever neighbour is returned).  The sign is
// copied back so that -0 / s stays -0.  Two values per call (packed fp32
// pairs, each half rounded as the scalar operation).  An exhaustive
// comparison with IEEE division over every pair of bf16 values x, amax with
// |x| <= amax is in tests/c/fp8_quotient_check.c.
__device__ __forceinline__ float2 quotient2(float2 x, float f, float s2, float inv) {
  const float2 x2 = fmul2(x, make_float2(f, f));
  const float2 q0 = fmul2(x2, make_float2(inv, inv));
  const float2 rem = ffma2(q0, make_float2(-s2, -s2), x2);
  const float2 q = ffma2(rem, make_float2(inv, inv), q0);
  return make_float2(copysignf(q.x, x.x), copysignf(q.y, x.y));
}

// Slot -> entry pointer, or nullptr for padding / out-of-range slots.  Slots
// in range are below 2^32 (checked on the host), so 32-bit division applies.
__device__ __forceinline__ uint8_t* entry_of(int64_t slot, const WriteArgs& a) {
  if (slot < 0 || slot >= a.num_slots) return nullptr;
  const uint32_t s = static_cast<uint32_t>(slot);
  const uint32_t blk = a.block_div.div(s);
  const uint32_t off = s - blk * static_cast<uint32_t>(a.block_size);
  return a.cache + static_cast<int64_t>(blk) * a.block_stride + static_cast<int64_t>(off) * a.entry_stride;
}

// ---------------------------------------------------------------------------
// nvfp4_ds_mla: 352-byte entries
// ---------------------------------------------------------------------------
template <bool kWide, int kTokensPerWarp>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kTokensPerWarp == 1 ? kSmallMinBlocks : kMinBlocks)
write_nvfp4_ds_mla_kernel(const WriteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t0 =
      (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * kTokensPerWarp;
  if (t0 >= a.num_tokens) return;

  // One coalesced load of this warp's slots; lane j holds token t0 + j's.
  int64_t my_slot = -1;
  if (lane < kTokensPerWarp && t0 + lane < a.num_tokens) my_slot = __ldg(a.slot_mapping + t0 + lane);
  if (lane < kTokensPerWarp && my_slot >= a.num_slots) report(a.status, KVQ_STATUS_BAD_INDEX);

  const __nv_bfloat16* kv_c = static_cast<const __nv_bfloat16*>(a.kv_c);
  const __nv_bfloat16* k_pe = static_cast<const __nv_bfloat16*>(a.k_pe);

  // The rows are loaded without waiting for the slots (a padding token's row
  // is read but nothing is written for it), so the slot and row loads overlap.
  uint8_t* entry[kTokensPerWarp];
  uint4 na[kTokensPerWarp], nb[kTokensPerWarp];
  uint2 rp[kTokensPerWarp];
#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) {
    if (t0 + j < a.num_tokens) {
      load32<kWide>(kv_c + (t0 + j) * a.kv_c_stride + lane * kGroup, na[j], nb[j]);
      if (lane < 16) rp[j] = ld_stream8(k_pe + (t0 + j) * a.k_pe_stride + lane * 4);
    }
  }
#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) entry[j] = entry_of(__shfl_sync(kFull, my_slot, j), a);

#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) {
    if (entry[j] == nullptr) continue;
    // NoPE group `lane`: scale, inverse, 8 packed bytes at 8 * lane.
    const uint32_t sf = nvfp4_scale_code(amax16(na[j], nb[j]));
    float x[16];
    unpack16(na[j], nb[j], x);
    st8(entry[j] + 8 * lane, nvfp4_pack16(x, nvfp4_inverse_scale(sf)));
    // RoPE: lanes 0..15 convert 4 values each into bytes 256 + 4 * lane.
    if (lane < 16) {
      const uint32_t lo = cvt_e4m3x2(bf16_lo(rp[j].x), bf16_hi(rp[j].x));
      const uint32_t hi = cvt_e4m3x2(bf16_lo(rp[j].y), bf16_hi(rp[j].y));
      st4(entry[j] + kNvRopeOff + 4 * lane, lo | (hi << 16));
    }
    // Scale bytes: gather four per word; lanes 0, 4, ..., 28 store 32 bytes.
    uint32_t w = sf;
    w |= __shfl_down_sync(kFull, sf, 1) << 8;
    w |= __shfl_down_sync(kFull, sf, 2) << 16;
    w |= __shfl_down_sync(kFull, sf, 3) << 24;
    if ((lane & 3) == 0) st4(entry[j] + kNvSfOff + lane, w);
  }
}

// ---------------------------------------------------------------------------
// fp8_ds_mla: 656-byte entries
// ---------------------------------------------------------------------------
template <bool kWide, int kTokensPerWarp>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kTokensPerWarp == 1 ? kSmallMinBlocks : kMinBlocks)
write_fp8_ds_mla_kernel(const WriteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t0 =
      (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * kTokensPerWarp;
  if (t0 >= a.num_tokens) return;

  int64_t my_slot = -1;
  if (lane < kTokensPerWarp && t0 + lane < a.num_tokens) my_slot = __ldg(a.slot_mapping + t0 + lane);
  if (lane < kTokensPerWarp && my_slot >= a.num_slots) report(a.status, KVQ_STATUS_BAD_INDEX);

  const __nv_bfloat16* kv_c = static_cast<const __nv_bfloat16*>(a.kv_c);
  const __nv_bfloat16* k_pe = static_cast<const __nv_bfloat16*>(a.k_pe);

  uint8_t* entry[kTokensPerWarp];
  uint4 na[kTokensPerWarp], nb[kTokensPerWarp], rp[kTokensPerWarp];
#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) {
    if (t0 + j < a.num_tokens) {
      load32<kWide>(kv_c + (t0 + j) * a.kv_c_stride + lane * 16, na[j], nb[j]);
      if (lane < 8) rp[j] = ld_stream16(k_pe + (t0 + j) * a.k_pe_stride + lane * 8);
    }
  }
#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) entry[j] = entry_of(__shfl_sync(kFull, my_slot, j), a);

#pragma unroll
  for (int j = 0; j < kTokensPerWarp; ++j) {
    if (entry[j] == nullptr) continue;
    // Tile lane / 8 of 128 values: reduce the amax over its 8 lanes.
    float amax = amax16(na[j], nb[j]);
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
    const float s = amax == 0.0f ? 1.0f : tile_scale(amax);
    // x / s, correctly rounded, without a division per value: tile scales
    // below 2^-64 are first brought up by 2^96 together with the values
    // (exact, the quotient is unchanged), then Markstein's correction of a
    // product with the correctly rounded reciprocal applies (see quotient2()).
    const float f = s < 0x1p-64f ? 0x1p96f : 1.0f;
    const float s2 = __fmul_rn(s, f);
    const float inv = __frcp_rn(s2);
    float x[16];
    unpack16(na[j], nb[j], x);
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 lo = quotient2(make_float2(x[4 * k], x[4 * k + 1]), f, s2, inv);
      const float2 hi = quotient2(make_float2(x[4 * k + 2], x[4 * k + 3]), f, s2, inv);
      q[k] = cvt_e4m3x2(lo.x, lo.y) | (cvt_e4m3x2(hi.x, hi.y) << 16);
    }
    st16(entry[j] + 16 * lane, make_uint4(q[0], q[1], q[2], q[3]));
    if ((lane & 7) == 0) st4(entry[j] + kF8ScaleOff + 4 * (lane >> 3), __float_as_uint(s));
    if (lane < 8) st16(entry[j] + kF8RopeOff + 16 * lane, rp[j]);
  }
}

// kv_c rows that start on 32-byte boundaries are read with 32-byte accesses.
bool wide_rows(const WriteArgs& a) {
  return reinterpret_cast<uintptr_t>(a.kv_c) % 32 == 0 && (a.kv_c_stride * 2) % 32 == 0;
}

template <int kTpw>
cudaError_t launch_write(void (*kernel)(WriteArgs), const WriteArgs& a, cudaStream_t stream) {
  const int64_t tokens_per_block = int64_t{kWarpsPerBlock} * kTpw;
  const int64_t blocks = (a.num_tokens + tokens_per_block - 1) / tokens_per_block;
  kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

// Large batches: kTokensPerWarp tokens per warp (more bytes in flight per
// warp).  Small, latency-bound batches (decode steps): one token per warp,
// four times as many warps.
template <template <bool, int> class K>
cudaError_t dispatch_write(const WriteArgs& a, cudaStream_t stream) {
  const bool wide = wide_rows(a);
  if (a.num_tokens >= kSmallBatch)
    return launch_write<kTokensPerWarp>(wide ? K<true, kTokensPerWarp>::fn : K<false, kTokensPerWarp>::fn,
                                        a, stream);
  return launch_write<1>(wide ? K<true, 1>::fn : K<false, 1>::fn, a, stream);
}

template <bool W, int T>
struct Nvfp4Write {
  static constexpr void (*fn)(WriteArgs) = write_nvfp4_ds_mla_kernel<W, T>;
};
template <bool W, int T>
struct Fp8Write {
  static constexpr void (*fn)(WriteArgs) = write_fp8_ds_mla_kernel<W, T>;
};

}  // namespace

// The largest batch whose grid stays within 2^31 - 1 CTAs on either launch
// path (at least one token per warp).
int64_t write_max_tokens() { return int64_t{INT32_MAX} * kWarpsPerBlock; }

cudaError_t launch_write_nvfp4_ds_mla(const WriteArgs& a, cudaStream_t stream) {
  return dispatch_write<Nvfp4Write>(a, stream);
}

cudaError_t launch_write_fp8_ds_mla(const WriteArgs& a, cudaStream_t stream) {
  return dispatch_write<Fp8Write>(a, stream);
}

}  // namespace kvq
