// kvq_attention.cu -- sparse MLA attention read straight from the 352-byte
// nvfp4_ds_mla cache (the consumer the bf16 workspace would otherwise feed),
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
//
// vLLM PR #51724 ("Enable W4A16 DSA: NVFP4 DS-MLA KV cache format for the
// FlashMLA Sparse backend"), "Key source snippets" (flashmla_sparse.py): the
// sparse decode path serves the quantized DS-MLA formats and reads the cache
// itself.  vLLM PR #48642 ("[Bugfix] Sparse MLA: enable fp8_ds_mla dense
// prefill"), "Implementation breakdown" item 3: that decode runs as MQA over
// the latent cache.  For token t, head h and the token's top-k global slots j:
//   s_j = scale * (q[t,h] . k_j)        k_j = the entry's 576 decoded values
//   o[t,h] = sum_j softmax(s)_j * k_j[0:512],   lse[t,h] = log sum_j exp(s_j)
//
// Design (one CTA per (token, half of the 512 value dimensions)):
//   - the token's 128 query rows (heads, zero-padded) sit in shared memory
//     for the whole kernel as the A operand of S = Q K^T (K-major, 128-byte
//     swizzle, 9 blocks of 64 dimensions);
//   - per tile of 32 slots, all warps decode the 32 entries to bf16 (exact:
//     e2m1 x e4m3 products) into a swizzled shared tile that is both the B
//     operand of Q K^T (K-major) and, read MN-major, the V operand of P V;
//   - one thread issues the MMAs: S (128 x 32, fp32) into TMEM columns
//     [256, 288), the half of O (128 x 256, fp32) into TMEM columns [0, 256);
//   - warps 0-3 own TMEM lanes 0-127 (one query row per thread): they read S,
//     run the online softmax in the base-2 domain, round P to bf16 into
//     shared memory (the A operand of P V) and rescale their O row in TMEM
//     when the running maximum grows;
//   - the denominator sums the bf16-rounded P, the values the tensor cores
//     multiply, so the normalisation matches the weights used.
// Both halves compute the same S: the 128 x 512 fp32 O of a full token would
// fill all 512 TMEM columns and leave none for S.
//
// Every mbarrier wait is bounded; on expiry the CTA records
// KVQ_STATUS_TIMEOUT, stops issuing work, waits (bounded) for the MMAs it has
// in flight and frees its TMEM before it exits.
#include <cuda_bf16.h>

#include "kvq.h"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kDim = KVQ_MLA_NOPE_DIM + KVQ_MLA_ROPE_DIM;   // 576
constexpr int kNope = KVQ_MLA_NOPE_DIM;                      // 512
constexpr int kHalf = kNope / 2;                             // 256 value columns per CTA
constexpr int kRows = 128;                                   // query rows (heads) per CTA
constexpr int kTile = 32;                                    // slots per tile (N of Q K^T)
constexpr int kThreads = 256;
constexpr int kKBlocks = kDim / 64;                          // 9 swizzle blocks of 64 bf16
constexpr int kNvRopeOff = 256, kNvSfOff = 320;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr uint32_t kQBlock = kRows * 128;                    // 16 KB per 64-dim block
constexpr uint32_t kQBytes = kKBlocks * kQBlock;             // 144 KB
constexpr uint32_t kKBlock = kTile * 128;                    // 4 KB per 64-dim block
constexpr uint32_t kKOff = kQBytes;
constexpr uint32_t kKBytes = kKBlocks * kKBlock;             // 36 KB
constexpr uint32_t kPOff = kKOff + kKBytes;
constexpr uint32_t kPBytes = kRows * 128;                    // 16 KB (64 columns, 32 used)
constexpr uint32_t kMiscOff = kPOff + kPBytes;
constexpr uint32_t kSmemBytes = kMiscOff + 128 + 1024;       // + barriers, flags, alignment

// TMEM columns.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;
constexpr uint32_t kSCol = 256;

constexpr long long kWaitCycles = 4000000000LL;              // about 2 s at 2 GHz

// ---------------------------------------------------------------------------
// tcgen05 / mbarrier helpers (inline PTX, PTX ISA 8.7+ for sm_100a-family)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor: 128-byte swizzle, 1024-byte aligned atoms
// of 8 rows x 128 bytes.  lbo / sbo in bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (uint64_t{1} << 46) |                 // descriptor version of tcgen05
         (uint64_t{2} << 61);                  // 128-byte swizzle
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared stores made visible to the tensor cores' async proxy.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Waits for the phase with the given parity; false when the wait expired.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const long long start = clock64();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    if (done) return true;
    if (clock64() - start > kWaitCycles) return false;
    __nanosleep(20);
  }
}

// 32 consecutive fp32 TMEM columns of this warp's 32 lanes (one per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
         "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
         "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
         "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
         "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
         "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
         "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
         "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
         "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
         "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
         "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled block: chunks are permuted by XOR with row % 8.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ void st_shared16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 8 e4m3 codes -> 8 bf16 (exact).
__device__ __forceinline__ uint4 e4m3x8_bf16(uint2 c) {
  const float2 f0 = __half22float2(e4m3x2_to_half2(c.x));
  const float2 f1 = __half22float2(e4m3x2_to_half2(c.x >> 16));
  const float2 f2 = __half22float2(e4m3x2_to_half2(c.y));
  const float2 f3 = __half22float2(e4m3x2_to_half2(c.y >> 16));
  return make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y), pack_bf16x2(f2.x, f2.y),
                    pack_bf16x2(f3.x, f3.y));
}

// 4 bytes of e2m1 pairs times one scale -> 8 bf16 (exact products).
__device__ __forceinline__ uint4 e2m1x8_bf16(uint32_t four_bytes, float scale) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(e2m1x2_to_half2(four_bytes >> (8 * i)));
    o[i] = pack_bf16x2(v.x * scale, v.y * scale);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_attention_nvfp4_kernel(const AttentionArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(smem);
  const uint32_t q_base = base, k_base = base + kKOff, p_base = base + kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMiscOff);
  const uint32_t bar_s = smem_u32(&bars[0]), bar_o = smem_u32(&bars[1]), bar_d = smem_u32(&bars[2]);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMiscOff + 24);
  uint8_t* s_valid = smem + kMiscOff + 32;                  // [kTile]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t token = blockIdx.x >> 1;
  const int half = blockIdx.x & 1;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(s_tmem)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_d, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // Query rows -> swizzled K-major blocks (rows >= num_heads are zero).
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + token * a.q_stride_t;
  for (int i = threadIdx.x; i < kRows * (kDim / 8); i += kThreads) {
    const int row = i / (kDim / 8), c = i % (kDim / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < a.num_heads) v = __ldg(reinterpret_cast<const uint4*>(q + row * a.q_stride_h + 8 * c));
    st_shared16(q_base + (c >> 3) * kQBlock + sw128_offset(row, c & 7), v);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;

  const int32_t* idx = a.indices + token * a.indices_stride;
  const int n_tiles = (a.topk + kTile - 1) / kTile;
  constexpr uint32_t kIdescQK = idesc_bf16(kRows, kTile, false);
  constexpr uint32_t kIdescPV = idesc_bf16(kRows, kHalf, true);

  float m = -INFINITY, l = 0.0f;           // running max (base 2) and sum of row threadIdx.x
  const uint32_t row_lane = static_cast<uint32_t>(warp & 3) * 32u << 16;
  int mma_tiles = 0;                       // tiles whose S MMAs were issued (block-uniform)
  int pv_tiles = 0;                        // tiles whose P V MMAs were issued (block-uniform)
  bool bad_index = false, aborted = false;

  for (int tile = 0; tile < n_tiles; ++tile) {
    int expired = 0;
    // The previous P V must be done before its operands are overwritten.
    if (tile > 0 && !mbar_wait(bar_o, (tile - 1) & 1)) expired = 1;

    // Decode this tile's entries: warp w takes rows 4w .. 4w+3.
    {
      uint2 nib[4];
      uint32_t sf[4];
      uint2 rope[4];
      bool valid[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = warp * 4 + k, j = tile * kTile + r;
        const int32_t slot = j < a.topk ? __ldg(idx + j) : -1;
        valid[k] = slot >= 0 && slot < a.num_slots;
        if (slot >= a.num_slots) bad_index = true;
        if (valid[k]) {
          const uint32_t blk = a.block_div.div(static_cast<uint32_t>(slot));
          const uint32_t off = static_cast<uint32_t>(slot) - blk * static_cast<uint32_t>(a.block_size);
          const uint8_t* e = a.cache + static_cast<int64_t>(blk) * a.block_stride +
                             static_cast<int64_t>(off) * a.entry_stride;
          nib[k] = __ldg(reinterpret_cast<const uint2*>(e + 8 * lane));
          sf[k] = __ldg(e + kNvSfOff + lane);
          if (lane < 8) rope[k] = __ldg(reinterpret_cast<const uint2*>(e + kNvRopeOff + 8 * lane));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t r = warp * 4 + k;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo, rp = lo;
        if (valid[k]) {
          const float scale = e4m3_to_float(sf[k]);
          lo = e2m1x8_bf16(nib[k].x, scale);
          hi = e2m1x8_bf16(nib[k].y, scale);
          if (lane < 8) rp = e4m3x8_bf16(rope[k]);
        }
        // NoPE group `lane`: dims 16*lane .. 16*lane+15 = block lane/4, chunks 2*(lane%4) + {0,1}
        const uint32_t blk = k_base + (lane >> 2) * kKBlock;
        st_shared16(blk + sw128_offset(r, 2 * (lane & 3)), lo);
        st_shared16(blk + sw128_offset(r, 2 * (lane & 3) + 1), hi);
        if (lane < 8) st_shared16(k_base + 8 * kKBlock + sw128_offset(r, lane), rp);
        if (lane == 0) s_valid[r] = valid[k] ? 1 : 0;
      }
    }
    fence_async_smem();
    fence_before_sync();
    if (__syncthreads_or(expired)) { aborted = true; break; }
    mma_tiles = tile + 1;

    // S = Q K^T over 576 dims: 36 MMAs of K = 16.
    if (threadIdx.x == 0) {
      fence_after_sync();
#pragma unroll 4
      for (int k = 0; k < kDim / 16; ++k) {
        const uint32_t kb = k >> 2, kk = (k & 3) * 32;
        mma_bf16(tmem + kSCol, sw128_desc(q_base + kb * kQBlock + kk, 16, 1024),
                 sw128_desc(k_base + kb * kKBlock + kk, 16, 1024), kIdescQK, k > 0);
      }
      mma_commit(bar_s);
    }

    if (warp < 4) {
      if (!mbar_wait(bar_s, tile & 1)) expired = 1;
      fence_after_sync();
      float s[32];
      tmem_ld32(tmem + row_lane + kSCol, s);
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        s[j] = s_valid[j] ? s[j] * a.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, s[j]);
      }
      const float m_new = fmaxf(m, tmax);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      const float alpha = exp2f(m - m_use);             // 0 while m is -inf
      uint32_t pk[16];
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        pk[j] = pack_bf16x2(exp2f(s[2 * j] - m_use), exp2f(s[2 * j + 1] - m_use));
        psum += bf16_lo(pk[j]) + bf16_hi(pk[j]);
      }
      l = l * alpha + psum;
      m = m_new;
      // Rescale this row's O when the maximum grew (warp-wide TMEM access).
      if (tile > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + row_lane + kOCol + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + row_lane + kOCol + 32 * c, o);
        }
      }
      const uint32_t row = threadIdx.x;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared16(p_base + sw128_offset(row, c),
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      fence_async_smem();
      fence_before_sync();
    }
    if (__syncthreads_or(expired)) { aborted = true; break; }

    // O[:, half] += P V: 2 MMAs of K = 16 slots, N = 256 value columns.
    if (threadIdx.x == 0) {
      fence_after_sync();
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k)
        mma_bf16(tmem + kOCol, sw128_desc(p_base + 32 * k, 16, 1024),
                 sw128_desc(k_base + (4 * half) * kKBlock + 2048 * k, kKBlock, 1024), kIdescPV,
                 (tile > 0 || k > 0) ? 1u : 0u);
      mma_commit(bar_o);
    }
    pv_tiles = tile + 1;
  }

  // Drain every MMA still in flight: one more commit tracks all of them.
  if (mma_tiles > 0) {
    if (threadIdx.x == 0) mma_commit(bar_d);
    if (!mbar_wait(bar_d, 0)) aborted = true;
  }
  fence_after_sync();
  if (bad_index && a.status) atomicOr(a.status, KVQ_STATUS_BAD_INDEX);
  aborted = __syncthreads_or(aborted) != 0;
  if (aborted && threadIdx.x == 0 && a.status) atomicOr(a.status, KVQ_STATUS_TIMEOUT);

  if (warp < 4 && !aborted) {
    const int row = threadIdx.x;
    const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + token * a.out_stride_t +
                         static_cast<int64_t>(row) * a.out_stride_h + half * kHalf;
#pragma unroll 1
    for (int c = 0; c < kHalf / 32; ++c) {
      float o[32];
      if (pv_tiles > 0) tmem_ld32(tmem + row_lane + kOCol + 32 * c, o);
      if (row < a.num_heads) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (pv_tiles > 0)
            v = make_uint4(pack_bf16x2(o[8 * i] * inv_l, o[8 * i + 1] * inv_l),
                           pack_bf16x2(o[8 * i + 2] * inv_l, o[8 * i + 3] * inv_l),
                           pack_bf16x2(o[8 * i + 4] * inv_l, o[8 * i + 5] * inv_l),
                           pack_bf16x2(o[8 * i + 6] * inv_l, o[8 * i + 7] * inv_l));
          *reinterpret_cast<uint4*>(out + 32 * c + 8 * i) = v;
        }
      }
    }
    if (half == 0 && a.lse != nullptr && row < a.num_heads)
      a.lse[token * a.lse_stride_t + row] =
          l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

cudaError_t launch_sparse_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_attention_nvfp4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  sparse_mla_attention_nvfp4_kernel<<<static_cast<unsigned>(a.num_tokens * 2), kThreads, kSmemBytes,
                                      stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
