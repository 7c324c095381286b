// kvq_device.cuh -- device helpers shared by the sm_103a kernels: the
// number-format conversions (hand-written PTX from the public ISA) and the
// vector memory accesses.  Nothing here is visible outside the library.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq.h"

namespace kvq {

constexpr int kNopeDim = KVQ_MLA_NOPE_DIM;       // 512
constexpr int kRopeDim = KVQ_MLA_ROPE_DIM;       // 64
constexpr int kGroup = 16;                       // NVFP4 values per e4m3 scale
constexpr int kNvEntry = KVQ_NVFP4_DS_MLA_ENTRY_BYTES;  // 352
constexpr int kNvRopeOff = kNopeDim / 2;                 // 256
constexpr int kNvSfOff = kNvRopeOff + kRopeDim;          // 320
constexpr int kF8Entry = KVQ_FP8_DS_MLA_ENTRY_BYTES;     // 656
constexpr int kF8Tile = 128;                             // NoPE values per fp32 scale
constexpr int kF8ScaleOff = kNopeDim;                    // 512
constexpr int kF8RopeOff = kF8ScaleOff + 4 * (kNopeDim / kF8Tile);  // 528
constexpr int kWorkspaceDim = KVQ_WORKSPACE_DIM;         // 576
constexpr unsigned kFull = 0xffffffffu;

static_assert(kNvSfOff + kNopeDim / kGroup == kNvEntry, "352-byte entry");
static_assert(kF8RopeOff + 2 * kRopeDim == kF8Entry, "656-byte entry");

// ---------------------------------------------------------------------------
// division by a run-time invariant
// ---------------------------------------------------------------------------

// Unsigned 32-bit n / d for a divisor fixed at launch (1 <= d < 2^31), by a
// multiply-high and two shifts: the round-up method of Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication" (PLDI
// 1994), figure 4.1.  Exact for every 32-bit n.
struct FastDiv {
  uint32_t d = 1, m = 1, s1 = 0, s2 = 0;     // default: division by 1

  static FastDiv make(uint32_t divisor) {
    FastDiv f;
    f.d = divisor;
    uint32_t l = 0;
    while ((uint64_t{1} << l) < divisor) ++l;          // l = ceil(log2 d)
    f.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - divisor)) / divisor + 1);
    f.s1 = l < 1 ? l : 1;
    f.s2 = l > 0 ? l - 1 : 0;
    return f;
  }

  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> s1)) >> s2;
  }
};

// ---------------------------------------------------------------------------
// number formats
// ---------------------------------------------------------------------------

// Two fp32 -> two e2m1 codes, round to nearest even, satfinite
// (cvt.rn.satfinite.e2m1x2.f32, the conversion the NVFP4 DS-MLA page's write
// kernel names).  Returns lo's code in bits 3:0 and hi's in bits 7:4: the
// instruction packs its first source operand into the upper nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> two e4m3 codes, round to nearest even, satfinite.  lo's code in
// bits 7:0, hi's in bits 15:8.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes (bits 7:0 and 15:8) -> f16x2 holding the same two values
// (exact: every e4m3 value is an f16 normal or zero).
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return *reinterpret_cast<__half2*>(&r);
}

// Two e2m1 codes (bits 3:0 and 7:4 of the low byte) -> f16x2 (exact).
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(r) : "r"(byte));
  return *reinterpret_cast<__half2*>(&r);
}

__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  return __low2float(e4m3x2_to_half2(code & 0xffu));
}

// Two fp32 -> bf16x2 bits (round to nearest even; lo in bits 15:0).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The bf16 value held in bits 15:0 / 31:16 of a packed word, as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// max(|a|, |b|) over the bf16 pairs of a packed word, kept packed.
__device__ __forceinline__ __nv_bfloat162 abs_bf16x2(uint32_t w) {
  uint32_t a = w & 0x7fff7fffu;
  return *reinterpret_cast<__nv_bfloat162*>(&a);
}

// Two fp32 operations in one instruction (sm_100 and later; each half rounded
// to nearest even exactly as the scalar operation).
__device__ __forceinline__ float2 fmul2(float2 x, float2 y) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 x, float2 y) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y));
  return r;
}

__device__ __forceinline__ float2 ffma2(float2 x, float2 y, float2 z) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y), "f"(z.x), "f"(z.y));
  return r;
}

// NVFP4 group of 16 fp32 values (already scaled): sf = e4m3(amax / 6),
// inv = 1 / sf (0 when sf is 0), codes e2m1(x * inv) packed 2 per byte,
// value 2k in the low nibble of byte k.  Quotients are IEEE round-to-nearest
// (the library is built without fast-math), products single fp32 roundings.
//
// amax / 6 without a division: q0 = RN(amax * RN(1/6)) is within an ulp of
// the quotient, the remainder amax - 6 q0 is exact in one fused
// multiply-add, and RN(q0 + remainder * RN(1/6)) is the correctly rounded
// quotient (Markstein's theorem, P. Markstein, IBM J. Res. Dev. 34(1),
// 1990); +inf is passed through.  tests/c/nvfp4_scale_check.c compares it
// with IEEE division for every non-negative fp32 amax: equal wherever the
// e4m3 code can depend on it (quotients of 2^-11 and above).
__device__ __forceinline__ uint32_t nvfp4_scale_code(float amax) {
  constexpr float kInv6 = 1.0f / 6.0f;
  const float q0 = __fmul_rn(amax, kInv6);
  const float r = __fmaf_rn(-q0, 6.0f, amax);
  const float q = isinf(amax) ? amax : __fmaf_rn(r, kInv6, q0);
  return cvt_e4m3x2(q, 0.0f) & 0xffu;
}

__device__ __forceinline__ float nvfp4_inverse_scale(uint32_t sf_code) {
  const float sf = e4m3_to_float(sf_code);
  return sf == 0.0f ? 0.0f : 1.0f / sf;
}

__device__ __forceinline__ uint2 nvfp4_pack16(const float (&x)[16], float inv) {
  uint2 out;
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 a = fmul2(make_float2(x[2 * k], x[2 * k + 1]), make_float2(inv, inv));
    const float2 b = fmul2(make_float2(x[8 + 2 * k], x[8 + 2 * k + 1]), make_float2(inv, inv));
    w0 |= cvt_e2m1x2(a.x, a.y) << (8 * k);
    w1 |= cvt_e2m1x2(b.x, b.y) << (8 * k);
  }
  out.x = w0;
  out.y = w1;
  return out;
}

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------

// Read-once streaming loads (evict-first in L1 and L2).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint32_t ld_byte(const uint8_t* p) {
  return __ldg(p);
}

// 32 contiguous bytes in one access (256-bit vector load / store, sm_100 and
// later); the address must be 32-byte aligned.  A lane that moves 32 bytes as
// two 16-byte accesses leaves every 32-byte sector half-covered by each
// instruction; one 32-byte access covers whole sectors.
__device__ __forceinline__ void ld_stream32(const void* p, uint4& a, uint4& b) {
  asm("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z),
                  "r"(b.w)
               : "memory");
}

// 32 bytes at a 16-byte aligned address: one access when kWide (the caller
// has checked 32-byte alignment), else two.
template <bool kWide>
__device__ __forceinline__ void load32(const void* p, uint4& a, uint4& b) {
  if constexpr (kWide) {
    ld_stream32(p, a, b);
  } else {
    a = ld_stream16(p);
    b = ld_stream16(static_cast<const char*>(p) + 16);
  }
}
template <bool kWide>
__device__ __forceinline__ void store32(void* p, const uint4& a, const uint4& b) {
  if constexpr (kWide) {
    st32(p, a, b);
  } else {
    *reinterpret_cast<uint4*>(p) = a;
    *reinterpret_cast<uint4*>(static_cast<char*>(p) + 16) = b;
  }
}

__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st8(void* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }
__device__ __forceinline__ void st4(void* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

}  // namespace kvq
