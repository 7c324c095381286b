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
#ifndef KVQ_PER_HEAD_UNITS
#define KVQ_PER_HEAD_UNITS 1           // units (groups of one token side head) per thread
#endif
#ifndef KVQ_PER_HEAD_SCALE_FETCH
#define KVQ_PER_HEAD_SCALE_FETCH 0     // HND write: 0 none, 1 L2 prefetch, 2 8-byte load of the scale row
#endif
constexpr int kThreads = KVQ_PER_HEAD_THREADS;
constexpr int kMaxGpt = KVQ_PER_HEAD_MAX_GROUPS;
constexpr int kScaleFetch = KVQ_PER_HEAD_SCALE_FETCH;
constexpr int kUnitsPerThread = KVQ_PER_HEAD_UNITS;

// A thread owns kGpt consecutive 16-value groups of one (token, side, head)
// -- a unit -- and handles kUnits units kThreads apart: flat unit index =
// ((t * 2 + side) * H + h) * (groups / kGpt) + u, with unit_div / side_div /
// head_div set up by the launcher for that kGpt.
struct Unit {
  uint32_t t, side, h, g0;
};

template <int kGpt, int kUnits>
__device__ __forceinline__ bool unit_of(const PerHeadArgs& a, int j, Unit& u) {
  const uint64_t idx = (static_cast<uint64_t>(blockIdx.x) * kUnits + j) * kThreads + threadIdx.x;
  if (idx >= static_cast<uint64_t>(a.num_tokens) * a.unit_div.d) return false;   // < 2^32 (host check)
  const uint32_t i = static_cast<uint32_t>(idx);
  u.t = a.unit_div.div(i);
  const uint32_t r0 = i - u.t * a.unit_div.d;
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

// The data row and the scale row of a unit's groups in the cache, or false
// for a padding / out-of-range slot.
__device__ __forceinline__ bool unit_rows(const PerHeadArgs& a, const Unit& u, int64_t slot, uint8_t*& data,
                                          uint8_t*& scales) {
  if (slot < 0) return false;
  if (slot >= a.num_slots) {
    if (u.side == 0 && u.h == 0 && u.g0 == 0) report(a.status, KVQ_STATUS_BAD_INDEX);
    return false;
  }
  int64_t row;
  uint8_t* base = a.cache + side_base(a, slot, u.side, u.h, row);
  const int64_t data_dim = a.head_size / 2;
  data = base + row * data_dim + 8 * u.g0;
  scales = base + static_cast<int64_t>(a.block_size) * a.num_heads * data_dim + row * (a.head_size / kGroup) + u.g0;
  return true;
}

__device__ __forceinline__ const __nv_bfloat16* unit_src(const PerHeadArgs& a, const Unit& u) {
  return static_cast<const __nv_bfloat16*>(u.side ? a.value : a.key) +
         static_cast<int64_t>(u.t) * (u.side ? a.value_stride_t : a.key_stride_t) +
         static_cast<int64_t>(u.h) * (u.side ? a.value_stride_h : a.key_stride_h) + u.g0 * kGroup;
}

template <bool kWide, int kGpt, int kUnits>
__global__ void __launch_bounds__(kThreads) reshape_and_cache_nvfp4_kernel(const PerHeadArgs a) {
  // Every unit's groups are loaded first, without waiting for its slot (a
  // padding token's values are read but nothing is written for them).
  Unit u[kUnits];
  bool live[kUnits];
  uint4 lo[kUnits][kGpt], hi[kUnits][kGpt];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    live[j] = unit_of<kGpt, kUnits>(a, j, u[j]);
    if (live[j]) {
      const __nv_bfloat16* src = unit_src(a, u[j]);
#pragma unroll
      for (int g = 0; g < kGpt; ++g) load32<kWide>(src + g * kGroup, lo[j][g], hi[j][g]);
    }
  }
  int64_t slot[kUnits];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) slot[j] = live[j] ? __ldg(a.slot_mapping + u[j].t) : -1;
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    uint8_t *data, *scales;
    if (!live[j] || !unit_rows(a, u[j], slot[j], data, scales)) continue;
    if constexpr (kScaleFetch != 0) {
      if (a.layout == KVQ_LAYOUT_HND && u[j].g0 == 0) {
        if constexpr (kScaleFetch == 1) {
          asm volatile("prefetch.global.L2 [%0];" :: "l"(scales));
        } else {
          uint32_t d0, d1;
          asm volatile("ld.global.cg.v2.b32 {%0, %1}, [%2];" : "=r"(d0), "=r"(d1) : "l"(scales));
        }
      }
    }
    const float scale_in = __ldg(u[j].side ? a.v_scale : a.k_scale);
    const float inv_scale = 1.0f / scale_in;
    // y = x * inv_scale.  amax(|y|) = RN(amax(|x|) * |inv_scale|) exactly,
    // since rounding is monotone, so the maximum is taken on the packed bf16
    // pairs; when the per-tensor scale is 1 (warp-uniform), y = x needs no
    // multiply.
    const bool unit_scale = inv_scale == 1.0f;
    uint32_t sf_word = 0;
    uint2 packed[kGpt];
#pragma unroll
    for (int g = 0; g < kGpt; ++g) {
      const uint32_t w[8] = {lo[j][g].x, lo[j][g].y, lo[j][g].z, lo[j][g].w,
                             hi[j][g].x, hi[j][g].y, hi[j][g].z, hi[j][g].w};
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
      packed[g] = nvfp4_pack16(y, nvfp4_inverse_scale(sf));
      sf_word |= sf << (8 * g);
    }
    // The groups' 8 * kGpt data bytes in 16-byte stores (the offset is a
    // multiple of 8 * kGpt), so one instruction covers whole sectors across
    // the threads of a head; then the kGpt scale bytes, contiguous.
    if constexpr (kGpt == 1) {
      st8(data, packed[0]);
    } else {
#pragma unroll
      for (int g = 0; g < kGpt; g += 2)
        st16(data + 8 * g, make_uint4(packed[g].x, packed[g].y, packed[g + 1].x, packed[g + 1].y));
    }
    if constexpr (kGpt == 4) {
      st4(scales, sf_word);
    } else if constexpr (kGpt == 2) {
      *reinterpret_cast<uint16_t*>(scales) = static_cast<uint16_t>(sf_word);
    } else {
      *scales = static_cast<uint8_t>(sf_word);
    }
  }
}

// Loads of the read-back's cache rows with a 64-byte L2 fetch-size hint.  An
// L2 miss otherwise brings in the whole 128-byte line, and with scattered
// slots the rest of that line belongs to other slots: in HND a (token, side,
// head) has one 64-byte data row and one 8-byte scale row, each in a line of
// its own.  With the hint, 16,384 HND tokens read back in 20.3 instead of
// 22.7 us (NHD rows are contiguous per token side and do not change).
__device__ __forceinline__ uint4 ld_row16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.L2::64B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_row8(const void* p) {
  uint2 v;
  asm volatile("ld.global.cs.L2::64B.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_scale_byte(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L2::64B.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Read-back: the same thread-per-groups decomposition; each group's 8 data
// bytes and scale byte become 16 bf16 values bf16_rn((e2m1 * sf) * scale) --
// the first product exact, one fp32 rounding for the per-tensor scale, one
// bf16 rounding.  The slots of all of a thread's units are loaded first,
// then all of their cache rows.
template <bool kWide, int kGpt, int kUnits>
__global__ void __launch_bounds__(kThreads) dequant_nvfp4_per_head_kernel(const PerHeadArgs a) {
  Unit u[kUnits];
  int64_t slot[kUnits];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) slot[j] = unit_of<kGpt, kUnits>(a, j, u[j]) ? __ldg(a.slot_mapping + u[j].t) : -1;
  uint2 q[kUnits][kGpt];
  uint32_t sfb[kUnits][kGpt];
  bool live[kUnits];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    uint8_t *data, *scales;
    live[j] = unit_rows(a, u[j], slot[j], data, scales);
    if (!live[j]) continue;
    if constexpr (kGpt == 1) {
      q[j][0] = ld_row8(data);
    } else {
#pragma unroll
      for (int g = 0; g < kGpt; g += 2) {           // 16-byte loads (offset a multiple of 16)
        const uint4 v = ld_row16(data + 8 * g);
        q[j][g] = make_uint2(v.x, v.y);
        q[j][g + 1] = make_uint2(v.z, v.w);
      }
    }
#pragma unroll
    for (int g = 0; g < kGpt; ++g) sfb[j][g] = ld_scale_byte(scales + g);
  }
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    if (!live[j]) continue;
    const float scale = __ldg(u[j].side ? a.v_scale : a.k_scale);
    __nv_bfloat16* dst = const_cast<__nv_bfloat16*>(unit_src(a, u[j]));   // key / value are the outputs here
#pragma unroll
    for (int g = 0; g < kGpt; ++g) {
      const float sf = e4m3_to_float(sfb[j][g]);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = (i < 4 ? q[j][g].x : q[j][g].y) >> (8 * (i & 3));
        const float2 v = __half22float2(e2m1x2_to_half2(byte));
        const float2 y = fmul2(fmul2(v, make_float2(sf, sf)), make_float2(scale, scale));   // (v sf) scale, each RN
        o[i] = pack_bf16x2(y.x, y.y);
      }
      store32<kWide>(dst + g * kGroup, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
    }
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
  const int64_t units = a.num_tokens * a.unit_div.d;
  const int64_t per_block = int64_t{kThreads} * kUnitsPerThread;
  const unsigned blocks = static_cast<unsigned>((units + per_block - 1) / per_block);
  const bool wide = wide_rows(a);
  void (*kernel)(PerHeadArgs) =
      gpt == 4 ? (wide ? K<true, 4>::fn : K<false, 4>::fn)
               : gpt == 2 ? (wide ? K<true, 2>::fn : K<false, 2>::fn) : (wide ? K<true, 1>::fn : K<false, 1>::fn);
  kernel<<<blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool W, int G>
struct WriteK {
  static constexpr void (*fn)(PerHeadArgs) = reshape_and_cache_nvfp4_kernel<W, G, kUnitsPerThread>;
};
template <bool W, int G>
struct ReadK {
  static constexpr void (*fn)(PerHeadArgs) = dequant_nvfp4_per_head_kernel<W, G, kUnitsPerThread>;
};

}  // namespace

cudaError_t launch_reshape_and_cache_nvfp4(const PerHeadArgs& a, cudaStream_t stream) {
  return launch_per_head<WriteK>(a, stream);
}

cudaError_t launch_dequant_nvfp4_per_head(const PerHeadArgs& a, cudaStream_t stream) {
  return launch_per_head<ReadK>(a, stream);
}

}  // namespace kvq
