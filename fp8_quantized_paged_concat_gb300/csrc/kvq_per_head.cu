// kvq_per_head.cu -- reshape_and_cache into (and read-back out of) the per-head NVFP4 K/V cache
// [num_pages, 2, block_size, H, full_dim] whose side regions hold
// [data [block_size][H][D/2] | scales [block_size][H][D/16]].
//
// Design (GB300): one thread per 16-value group of one (token, side, head):
// it loads its 32 contiguous input bytes, forms the group scale and writes 8
// data bytes and 1 scale byte.  Groups are numbered fastest within a head,
// then heads, then sides, so a warp covers whole heads of one token side and
// its stores are contiguous (8 x 32 = 256 data bytes and 32 scale bytes at
// H = 8, D = 128).
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

template <bool kWide>
__global__ void __launch_bounds__(kThreads) reshape_and_cache_nvfp4_kernel(const PerHeadArgs a) {
  // flat index = ((t * 2 + side) * H + h) * groups + g, below 2^32 (host check)
  const uint32_t idx = blockIdx.x * kThreads + threadIdx.x;
  const uint32_t t = a.unit_div.div(idx);
  if (t >= a.num_tokens) return;
  const uint32_t u = idx - t * a.unit_div.d;
  const uint32_t side = a.side_div.div(u);
  const uint32_t r = u - side * a.side_div.d;
  const uint32_t h = a.head_div.div(r);
  const uint32_t g = r - h * a.head_div.d;

  // The group is loaded without waiting for the slot (a padding token's
  // values are read but nothing is written for them).
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(side ? a.value : a.key) +
                             static_cast<int64_t>(t) * (side ? a.value_stride_t : a.key_stride_t) +
                             static_cast<int64_t>(h) * (side ? a.value_stride_h : a.key_stride_h) +
                             g * kGroup;
  uint4 lo, hi;
  load32<kWide>(src, lo, hi);
  const int64_t slot = __ldg(a.slot_mapping + t);
  const float scale_in = __ldg(side ? a.v_scale : a.k_scale);
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (side == 0 && h == 0 && g == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return;
  }
  const float inv_scale = 1.0f / scale_in;

  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  float y[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y[2 * i] = __fmul_rn(bf16_lo(w[i]), inv_scale);
    y[2 * i + 1] = __fmul_rn(bf16_hi(w[i]), inv_scale);
    amax = fmaxf(amax, fmaxf(fabsf(y[2 * i]), fabsf(y[2 * i + 1])));
  }
  const uint32_t sf = nvfp4_scale_code(amax);

  const uint32_t page = a.block_div.div(static_cast<uint32_t>(slot));
  const uint32_t off = static_cast<uint32_t>(slot) - page * static_cast<uint32_t>(a.block_size);
  const int64_t data_dim = a.head_size / 2;
  const int64_t scale_dim = a.head_size / kGroup;
  const int64_t region = static_cast<int64_t>(a.block_size) * a.num_heads * (data_dim + scale_dim);
  uint8_t* base = a.cache + (static_cast<int64_t>(page) * 2 + side) * region;
  const int64_t row = static_cast<int64_t>(off) * a.num_heads + h;
  st8(base + row * data_dim + 8 * g, nvfp4_pack16(y, nvfp4_inverse_scale(sf)));
  base[static_cast<int64_t>(a.block_size) * a.num_heads * data_dim + row * scale_dim + g] =
      static_cast<uint8_t>(sf);
}

// Read-back: the same thread-per-group decomposition; each thread reads its
// group's 8 data bytes and scale byte and writes 16 bf16 values
// bf16_rn((e2m1 * sf) * scale) -- the first product exact, one fp32 rounding
// for the per-tensor scale, one bf16 rounding.
template <bool kWide>
__global__ void __launch_bounds__(kThreads) dequant_nvfp4_per_head_kernel(const PerHeadArgs a) {
  const uint32_t idx = blockIdx.x * kThreads + threadIdx.x;
  const uint32_t t = a.unit_div.div(idx);
  if (t >= a.num_tokens) return;
  const uint32_t u = idx - t * a.unit_div.d;
  const uint32_t side = a.side_div.div(u);
  const uint32_t r = u - side * a.side_div.d;
  const uint32_t h = a.head_div.div(r);
  const uint32_t g = r - h * a.head_div.d;

  const int64_t slot = __ldg(a.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (side == 0 && h == 0 && g == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return;
  }
  const uint32_t page = a.block_div.div(static_cast<uint32_t>(slot));
  const uint32_t off = static_cast<uint32_t>(slot) - page * static_cast<uint32_t>(a.block_size);
  const int64_t data_dim = a.head_size / 2;
  const int64_t scale_dim = a.head_size / kGroup;
  const int64_t region = static_cast<int64_t>(a.block_size) * a.num_heads * (data_dim + scale_dim);
  const uint8_t* base = a.cache + (static_cast<int64_t>(page) * 2 + side) * region;
  const int64_t row = static_cast<int64_t>(off) * a.num_heads + h;
  const uint2 q = ld_stream8(base + row * data_dim + 8 * g);
  const float sf = e4m3_to_float(
      ld_byte(base + static_cast<int64_t>(a.block_size) * a.num_heads * data_dim + row * scale_dim + g));
  const float scale = __ldg(side ? a.v_scale : a.k_scale);

  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = (i < 4 ? q.x : q.y) >> (8 * (i & 3));
    const float2 v = __half22float2(e2m1x2_to_half2(byte));
    o[i] = pack_bf16x2(__fmul_rn(v.x * sf, scale), __fmul_rn(v.y * sf, scale));
  }
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(const_cast<void*>(side ? a.value : a.key)) +
                       static_cast<int64_t>(t) * (side ? a.value_stride_t : a.key_stride_t) +
                       static_cast<int64_t>(h) * (side ? a.value_stride_h : a.key_stride_h) + g * kGroup;
  store32<kWide>(dst, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
}

// key / value rows whose 16-value groups all start on 32-byte boundaries.
bool wide_rows(const PerHeadArgs& a) {
  return reinterpret_cast<uintptr_t>(a.key) % 32 == 0 && reinterpret_cast<uintptr_t>(a.value) % 32 == 0 &&
         (a.key_stride_t * 2) % 32 == 0 && (a.key_stride_h * 2) % 32 == 0 &&
         (a.value_stride_t * 2) % 32 == 0 && (a.value_stride_h * 2) % 32 == 0;
}

}  // namespace

cudaError_t launch_dequant_nvfp4_per_head(const PerHeadArgs& a, cudaStream_t stream) {
  const int64_t threads = a.num_tokens * 2 * a.num_heads * (a.head_size / kGroup);
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  (wide_rows(a) ? dequant_nvfp4_per_head_kernel<true> : dequant_nvfp4_per_head_kernel<false>)
      <<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_nvfp4(const PerHeadArgs& a, cudaStream_t stream) {
  const int64_t threads = a.num_tokens * 2 * a.num_heads * (a.head_size / kGroup);
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  (wide_rows(a) ? reshape_and_cache_nvfp4_kernel<true> : reshape_and_cache_nvfp4_kernel<false>)
      <<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
