// kvq_per_head.cu -- reshape_and_cache into (and read-back out of) the per-head NVFP4 K/V cache
// [num_pages, 2, block_size, H, full_dim] (NHD) or [num_pages, 2, H, block_size, full_dim] (HND)
// whose side regions hold [data rows of D/2 bytes | scale rows of D/16 bytes], rows in the
// layout's (offset, head) order.
//
// Design (GB300): one thread per 2 consecutive 16-value groups of one
// (token, side, head) (1 when a head's group count is odd; up to 4 with
// KVQ_PER_HEAD_MAX_GROUPS): it issues its 32-byte loads first, forms each
// group's scale and writes 8 data bytes per group and the groups' scale
// bytes in one store.  128-thread CTAs (measured best with 2 groups).
// Threads are numbered fastest within a head, then heads, then sides, so a
// warp covers whole heads of one token side and its stores are contiguous.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

#ifndef KVQ_PER_HEAD_THREADS
#define KVQ_PER_HEAD_THREADS 128
#endif
#ifndef KVQ_PER_HEAD_MAX_GROUPS
#define KVQ_PER_HEAD_MAX_GROUPS 2      // 16-value groups per thread, at most
#endif
constexpr int kThreads = KVQ_PER_HEAD_THREADS;
constexpr int kMaxGpt = KVQ_PER_HEAD_MAX_GROUPS;

// A thread owns kGpt consecutive 16-value groups of one (token, side, head):
// flat index = ((t * 2 + side) * H + h) * (groups / kGpt) + u, with
// unit_div / side_div / head_div set up by the launcher for that kGpt.
struct Unit {
  uint32_t t, side, h, g0;
};

template <int kGpt>
__device__ __forceinline__ bool unit_of(const PerHeadArgs& a, Unit& u) {
  const uint32_t idx = blockIdx.x * kThreads + threadIdx.x;     // < 2^32 - 256 (host check)
  u.t = a.unit_div.div(idx);
  if (u.t >= a.num_tokens) return false;
  const uint32_t r0 = idx - u.t * a.unit_div.d;
  u.side = a.side_div.div(r0);
  const uint32_t r1 = r0 - u.side * a.side_div.d;
  u.h = a.head_div.div(r1);
  u.g0 = (r1 - u.h * a.head_div.d) * kGpt;
  return true;
}

// Base of (page, side) and the row index of (offset, head) in it: offset * H
// + h for NHD (a token's heads together), h * block_size + offset for HND (a
// head's tokens together).
__device__ __forceinline__ int64_t side_base(const PerHeadArgs& a, int64_t slot, uint32_t side,
                                             uint32_t h, int64_t& row) {
  const uint32_t page = a.block_div.div(static_cast<uint32_t>(slot));
  const uint32_t off = static_cast<uint32_t>(slot) - page * static_cast<uint32_t>(a.block_size);
  const int64_t region = static_cast<int64_t>(a.block_size) * a.num_heads * (a.head_size / 2 + a.head_size / kGroup);
  row = a.layout == KVQ_LAYOUT_HND ? static_cast<int64_t>(h) * a.block_size + off
                                   : static_cast<int64_t>(off) * a.num_heads + h;
  return (static_cast<int64_t>(page) * 2 + side) * region;
}

template <bool kWide, int kGpt>
__global__ void __launch_bounds__(kThreads) reshape_and_cache_nvfp4_kernel(const PerHeadArgs a) {
  Unit u;
  if (!unit_of<kGpt>(a, u)) return;
  // The groups are loaded without waiting for the slot (a padding token's
  // values are read but nothing is written for them).
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(u.side ? a.value : a.key) +
                             static_cast<int64_t>(u.t) * (u.side ? a.value_stride_t : a.key_stride_t) +
                             static_cast<int64_t>(u.h) * (u.side ? a.value_stride_h : a.key_stride_h) +
                             u.g0 * kGroup;
  uint4 lo[kGpt], hi[kGpt];
#pragma unroll
  for (int j = 0; j < kGpt; ++j) load32<kWide>(src + j * kGroup, lo[j], hi[j]);
  const int64_t slot = __ldg(a.slot_mapping + u.t);
  const float scale_in = __ldg(u.side ? a.v_scale : a.k_scale);
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (u.side == 0 && u.h == 0 && u.g0 == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return;
  }
  const float inv_scale = 1.0f / scale_in;
  int64_t row;
  uint8_t* base = a.cache + side_base(a, slot, u.side, u.h, row);
  const int64_t data_dim = a.head_size / 2;
  const int64_t scale_dim = a.head_size / kGroup;
  uint8_t* data = base + row * data_dim + 8 * u.g0;
  uint8_t* scales = base + static_cast<int64_t>(a.block_size) * a.num_heads * data_dim + row * scale_dim + u.g0;
  // y = x * inv_scale.  amax(|y|) = RN(amax(|x|) * |inv_scale|) exactly, since
  // rounding is monotone, so the maximum is taken on the packed bf16 pairs;
  // when the per-tensor scale is 1 (warp-uniform), y = x needs no multiply.
  const bool unit_scale = inv_scale == 1.0f;
  uint32_t sf_word = 0;
  uint2 packed[kGpt];
#pragma unroll
  for (int j = 0; j < kGpt; ++j) {
    const uint32_t w[8] = {lo[j].x, lo[j].y, lo[j].z, lo[j].w, hi[j].x, hi[j].y, hi[j].z, hi[j].w};
    __nv_bfloat162 m = __hmax2(__hmax2(abs_bf16x2(w[0]), abs_bf16x2(w[1])), __hmax2(abs_bf16x2(w[2]), abs_bf16x2(w[3])));
    m = __hmax2(m, __hmax2(__hmax2(abs_bf16x2(w[4]), abs_bf16x2(w[5])), __hmax2(abs_bf16x2(w[6]), abs_bf16x2(w[7]))));
    float amax = fmaxf(__low2float(m), __high2float(m));
    float y[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[2 * i] = bf16_lo(w[i]);
      y[2 * i + 1] = bf16_hi(w[i]);
    }
    if (!unit_scale) {
      amax = __fmul_rn(amax, fabsf(inv_scale));
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 p = fmul2(make_float2(y[i], y[i + 1]), make_float2(inv_scale, inv_scale));
        y[i] = p.x;
        y[i + 1] = p.y;
      }
    }
    const uint32_t sf = nvfp4_scale_code(amax);
    packed[j] = nvfp4_pack16(y, nvfp4_inverse_scale(sf));
    sf_word |= sf << (8 * j);
  }
  // The groups' 8 * kGpt data bytes in 16-byte stores (the offset is a
  // multiple of 8 * kGpt), so one instruction covers whole sectors across the
  // threads of a head; then the kGpt scale bytes, contiguous.
  if constexpr (kGpt == 1) {
    st8(data, packed[0]);
  } else {
#pragma unroll
    for (int j = 0; j < kGpt; j += 2)
      st16(data + 8 * j, make_uint4(packed[j].x, packed[j].y, packed[j + 1].x, packed[j + 1].y));
  }
  if constexpr (kGpt == 4) {
    st4(scales, sf_word);
  } else if constexpr (kGpt == 2) {
    *reinterpret_cast<uint16_t*>(scales) = static_cast<uint16_t>(sf_word);
  } else {
    *scales = static_cast<uint8_t>(sf_word);
  }
}

// Read-back: the same thread-per-groups decomposition; each group's 8 data
// bytes and scale byte become 16 bf16 values bf16_rn((e2m1 * sf) * scale) --
// the first product exact, one fp32 rounding for the per-tensor scale, one
// bf16 rounding.
template <bool kWide, int kGpt>
__global__ void __launch_bounds__(kThreads) dequant_nvfp4_per_head_kernel(const PerHeadArgs a) {
  Unit u;
  if (!unit_of<kGpt>(a, u)) return;
  const int64_t slot = __ldg(a.slot_mapping + u.t);
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (u.side == 0 && u.h == 0 && u.g0 == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return;
  }
  int64_t row;
  const uint8_t* base = a.cache + side_base(a, slot, u.side, u.h, row);
  const int64_t data_dim = a.head_size / 2;
  const int64_t scale_dim = a.head_size / kGroup;
  const uint8_t* data = base + row * data_dim + 8 * u.g0;
  const uint8_t* scales = base + static_cast<int64_t>(a.block_size) * a.num_heads * data_dim + row * scale_dim + u.g0;
  uint2 q[kGpt];
  uint32_t sfb[kGpt];
  if constexpr (kGpt == 1) {
    q[0] = ld_stream8(data);
  } else {
#pragma unroll
    for (int j = 0; j < kGpt; j += 2) {           // 16-byte loads (offset a multiple of 16)
      const uint4 v = ld_stream16(data + 8 * j);
      q[j] = make_uint2(v.x, v.y);
      q[j + 1] = make_uint2(v.z, v.w);
    }
  }
#pragma unroll
  for (int j = 0; j < kGpt; ++j) sfb[j] = ld_byte(scales + j);
  const float scale = __ldg(u.side ? a.v_scale : a.k_scale);
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(const_cast<void*>(u.side ? a.value : a.key)) +
                       static_cast<int64_t>(u.t) * (u.side ? a.value_stride_t : a.key_stride_t) +
                       static_cast<int64_t>(u.h) * (u.side ? a.value_stride_h : a.key_stride_h) +
                       u.g0 * kGroup;
#pragma unroll
  for (int j = 0; j < kGpt; ++j) {
    const float sf = e4m3_to_float(sfb[j]);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = (i < 4 ? q[j].x : q[j].y) >> (8 * (i & 3));
      const float2 v = __half22float2(e2m1x2_to_half2(byte));
      const float2 y = fmul2(fmul2(v, make_float2(sf, sf)), make_float2(scale, scale));   // (v sf) scale, each RN
      o[i] = pack_bf16x2(y.x, y.y);
    }
    store32<kWide>(dst + j * kGroup, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
  }
}

// key / value rows whose 16-value groups all start on 32-byte boundaries.
bool wide_rows(const PerHeadArgs& a) {
  return reinterpret_cast<uintptr_t>(a.key) % 32 == 0 && reinterpret_cast<uintptr_t>(a.value) % 32 == 0 &&
         (a.key_stride_t * 2) % 32 == 0 && (a.key_stride_h * 2) % 32 == 0 &&
         (a.value_stride_t * 2) % 32 == 0 && (a.value_stride_h * 2) % 32 == 0;
}

// Groups per thread: the largest of kMaxGpt, 2, 1 that divides a head's group
// count.  Sets the index dividers for it.
template <template <bool, int> class K>
cudaError_t launch_per_head(PerHeadArgs a, cudaStream_t stream) {
  const int groups = a.head_size / kGroup;
  // Several groups per thread move their data bytes in 16-byte accesses; that
  // needs every (page, side) region, block_size * H * full_dim bytes, to start
  // on a 16-byte boundary (the host check guarantees only 8).
  const int64_t region = static_cast<int64_t>(a.block_size) * a.num_heads * (a.head_size / 2 + groups);
  const bool pairs_ok = region % 16 == 0;
  const int gpt = (pairs_ok && kMaxGpt >= 4 && groups % 4 == 0) ? 4
                  : ((pairs_ok && kMaxGpt >= 2 && groups % 2 == 0) ? 2 : 1);
  const uint32_t per_head = static_cast<uint32_t>(groups / gpt);
  a.head_div = FastDiv::make(per_head);
  a.side_div = FastDiv::make(per_head * static_cast<uint32_t>(a.num_heads));
  a.unit_div = FastDiv::make(2 * per_head * static_cast<uint32_t>(a.num_heads));
  const int64_t threads = a.num_tokens * a.unit_div.d;
  const unsigned blocks = static_cast<unsigned>((threads + kThreads - 1) / kThreads);
  const bool wide = wide_rows(a);
  void (*kernel)(PerHeadArgs) =
      gpt == 4 ? (wide ? K<true, 4>::fn : K<false, 4>::fn)
               : gpt == 2 ? (wide ? K<true, 2>::fn : K<false, 2>::fn) : (wide ? K<true, 1>::fn : K<false, 1>::fn);
  kernel<<<blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool W, int G>
struct WriteK {
  static constexpr void (*fn)(PerHeadArgs) = reshape_and_cache_nvfp4_kernel<W, G>;
};
template <bool W, int G>
struct ReadK {
  static constexpr void (*fn)(PerHeadArgs) = dequant_nvfp4_per_head_kernel<W, G>;
};

}  // namespace

cudaError_t launch_reshape_and_cache_nvfp4(const PerHeadArgs& a, cudaStream_t stream) {
  return launch_per_head<WriteK>(a, stream);
}

cudaError_t launch_dequant_nvfp4_per_head(const PerHeadArgs& a, cudaStream_t stream) {
  return launch_per_head<ReadK>(a, stream);
}

}  // namespace kvq
