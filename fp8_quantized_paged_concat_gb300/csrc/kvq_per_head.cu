// kvq_per_head.cu -- reshape_and_cache into the per-head NVFP4 K/V cache
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

  const int64_t slot = __ldg(a.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (side == 0 && h == 0 && g == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return;
  }

  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(side ? a.value : a.key) +
                             static_cast<int64_t>(t) * (side ? a.value_stride_t : a.key_stride_t) +
                             static_cast<int64_t>(h) * (side ? a.value_stride_h : a.key_stride_h) +
                             g * kGroup;
  const uint4 lo = ld_stream16(src);
  const uint4 hi = ld_stream16(src + 8);
  const float inv_scale = 1.0f / __ldg(side ? a.v_scale : a.k_scale);

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

}  // namespace

cudaError_t launch_reshape_and_cache_nvfp4(const PerHeadArgs& a, cudaStream_t stream) {
  const int64_t threads = a.num_tokens * 2 * a.num_heads * (a.head_size / kGroup);
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  reshape_and_cache_nvfp4_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
