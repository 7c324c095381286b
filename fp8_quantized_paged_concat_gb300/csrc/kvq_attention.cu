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
// Design: a cluster of two CTAs per token, one per half of the 512 value
// dimensions.  CTA c (c = 0, 1) owns the query / key dimensions
// [256c, 256c + 256) of the NoPE part plus the RoPE part (64 dimensions, of
// which it multiplies the half [32c, 32c + 32)), so the 128 x 576 query block
// is split 80 KB / 80 KB and the 36 K-steps of Q K^T split 18 / 18:
//   - producers (8 warps) decode the CTA's share of each entry of a 64-slot
//     tile to bf16 (exact: e2m1 x e4m3 products) into a 3-stage ring of
//     swizzled tiles: the B operand of Q K^T (K-major) and, read MN-major,
//     the V operand of P V (the CTA's 256 value columns);
//   - one thread issues the MMAs: the partial S (128 x 64, fp32) into a TMEM
//     double buffer, O (128 x 256, fp32) into TMEM columns [0, 256);
//   - four exchange warps (one per TMEM lane quadrant) read each partial S
//     as soon as its MMAs complete, stage their 32 rows in shared memory and
//     hand them to the copy engine (cp.async.bulk into the peer CTA's shared
//     memory, completed on a transaction-counted mbarrier there), so the
//     transfer overlaps the softmax of the tile before; a forwarder thread
//     tells the peer when its copies have landed and when the receive
//     buffers have been read;
//   - the softmax warps (TMEM lanes 0-127, one query row per thread) add the
//     peer's partial to their own (a + b == b + a in IEEE arithmetic: both
//     CTAs hold bit-identical scores), run the online softmax in base 2 with
//     lazy rescaling (the reference maximum moves only when a tile exceeds
//     it by 2^8), round P to bf16 into TMEM (the A operand of P V) and
//     rescale their O row in TMEM when the reference moved;
//   - the denominator sums the bf16-rounded P, the weights the tensor cores
//     multiply.
//
// Every mbarrier wait is bounded; on expiry (or when another role of the CTA
// gave up) the CTA records KVQ_STATUS_TIMEOUT, stops issuing work, waits
// (bounded) for the MMAs in flight, frees its TMEM and meets its peer at the
// final cluster barrier, which every path reaches exactly once.
#include <cuda_bf16.h>

#include "kvq.h"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kHalf = KVQ_MLA_NOPE_DIM / 2;                  // 256 value columns per CTA
constexpr int kRows = 128;                                   // query rows (heads) per CTA
constexpr int kTile = 64;                                    // slots per tile (N of Q K^T)
// Warp roles: 0-3 softmax (columns 0-31), 4-7 producers, 8-11 softmax
// (columns 32-63), 12-15 producers, 16 MMA, 17-20 exchange, 21 forwarder
// (one thread).  A warp w that touches TMEM reads lanes 32 (w % 4) .. +31:
// softmax warps w and w + 8 share the query rows 32 (w % 4) .. +31, and the
// exchange warps cover all four quadrants (17 % 4 = 1, ..., 20 % 4 = 0).
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarps = 8;
constexpr int kExchangeWarps = 4;
constexpr int kRowsPerProducer = kTile / kProducerWarps;     // 8
constexpr int kThreads = (kSoftmaxWarps + kProducerWarps + 1 + kExchangeWarps + 1) * 32;   // 704
constexpr int kMmaThread = 16 * 32;
constexpr int kFirstExchangeWarp = 17;
constexpr int kForwardWarp = 21;
constexpr int kNvRopeOff = 256, kNvSfOff = 320;                  // nvfp4_ds_mla entry
constexpr int kF8ScaleOff = 512, kF8RopeOff = 528;                // fp8_ds_mla entry
constexpr float kRescaleLog2 = 8.0f;                         // lazy rescale threshold (base 2)

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kKStages = 3;                                  // K tiles in flight
// The CTA's 32 RoPE dimensions are 64 bytes per row: those blocks use the
// 64-byte swizzle (atoms of 8 rows x 64 bytes), the NoPE blocks (64
// dimensions, 128 bytes per row) the 128-byte swizzle.
constexpr uint32_t kQRope = kRows * 64;                      // the CTA's RoPE query dims: 8 KB
constexpr uint32_t kKBlock = kTile * 128;                    // 8 KB per 64-dim NoPE block
constexpr uint32_t kKRope = kTile * 64;                      // the tile's RoPE dims of the CTA: 4 KB
constexpr uint32_t kKBytes = 4 * kKBlock + kKRope;           // 36 KB per K stage
constexpr uint32_t kSBytes = kRows * kTile * 4;              // one partial S tile (fp32): 32 KB
constexpr uint32_t kKOff = kQRope;
constexpr uint32_t kRecvOff = kKOff + kKStages * kKBytes;    // 2 receive buffers (the peer's partial S)
constexpr uint32_t kSendOff = kRecvOff + 2 * kSBytes;        // this CTA's partial S, staged for the copy
constexpr uint32_t kPairOff = kSendOff + kSBytes;            // per-row maxima of the two column halves
constexpr uint32_t kMiscOff = kPairOff + 2 * 2 * kRows * 4;  // [tile parity][half][row]
constexpr uint32_t kSmemBytes = kMiscOff + 256 + 1024;       // + barriers, flags, alignment
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");
static_assert(kKOff % 1024 == 0 && kKBytes % 1024 == 0, "swizzle atoms must be 1024-byte aligned");
static_assert(kRecvOff % 16 == 0 && kSendOff % 16 == 0, "bulk copies move 16-byte aligned data");

// TMEM columns: O [0, 256), the CTA's 256 NoPE query dimensions as bf16
// pairs [256, 384) (the A operand of the NoPE K-steps), partial S double
// buffer [384, 512).  A tile's P (bf16 pairs, 32 columns) is written over
// the first half of its own S buffer, once its scores are in registers, and
// is the A operand of P V: the MMAs of one thread run in order, so the Q K^T
// two tiles later cannot overwrite it before P V has read it.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;
constexpr uint32_t kQCol = 256;
constexpr uint32_t kSCol = 384;

constexpr long long kWaitCycles = 4000000000LL;              // about 2 s at 2 GHz

// ---------------------------------------------------------------------------
// tcgen05 / mbarrier / cluster helpers (inline PTX, sm_100a family)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor: lbo / sbo in bytes; swizzle mode 2 =
// 128-byte (1024-byte atoms of 8 rows x 128 bytes), 4 = 64-byte (512-byte
// atoms of 8 rows x 64 bytes).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t mode) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (uint64_t{1} << 46) |                 // descriptor version of tcgen05
         (static_cast<uint64_t>(mode) << 61);
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(addr, lbo, sbo, 2);
}
__device__ __forceinline__ uint64_t sw64_desc(uint32_t addr) {
  return smem_desc(addr, 16, 512, 4);
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

// The same with A in TMEM: row i in lane i, element pairs (2c, 2c+1) of its
// 16 K-elements in columns a_tmem + c (the lower-indexed element in the low half).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

// Arrive on a barrier of the peer CTA (address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
               :: "r"(cluster_bar) : "memory");
}

// One bounded wait step: the thread sleeps in the barrier (up to about 1 ms,
// woken when the phase completes) instead of spinning on issue slots.
// Acquire at CTA scope for the barriers only this CTA arrives on, at
// cluster scope for those that order the peer's accesses.
template <bool kCluster>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  if constexpr (kCluster)
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
  return done != 0;
}

// Bounded wait that also gives up when another role of the CTA has aborted.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const long long start = clock64();
  while (!mbar_try_wait<kCluster>(bar, parity)) {
    if (*abort_flag || clock64() - start > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// `bytes` (a multiple of 16) from this CTA's shared memory into the peer's
// (address from mapa); the copy engine completes them on the peer's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t cluster_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst_cluster), "r"(src), "r"(bytes), "r"(cluster_bar) : "memory");
}

// 32 consecutive fp32 TMEM columns of this warp's 32 lanes (one per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
         "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
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

// The same for 64-byte rows (chunk 0..3) under the 64-byte swizzle: the
// chunk index is XORed with address bits 7-8, i.e. with (row / 2) % 4.
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

// A partial S tile (128 rows x 64 fp32 = 256 bytes per row) in a receive or
// send buffer: 16-byte chunk c of row r moves to chunk c ^ (r % 16), so that
// 32 threads reading the same chunk of 32 rows spread over all banks.
__device__ __forceinline__ uint32_t s_offset(uint32_t row, uint32_t chunk) {
  return row * 256u + ((chunk ^ (row & 15u)) << 4);
}

__device__ __forceinline__ void st_shared16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ float4 ld_shared16(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// 2^x for x <= 0 (0 for -inf): the hardware approximation, relative error
// below 2^-22, flushed to zero below 2^-126 (weights that small vanish next
// to the largest weight, which is at least 2^-8).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
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

// One NVFP4 group as bf16 without conversion instructions.  The eight
// products m * sf (m = 0, 0.5, 1, 1.5, 2, 3, 4, 6) are exact in bf16 (at most
// 6 significant bits, inside e4m3's range), so they are formed once per group
// with four bf16x2 multiplies; each code then selects its product's low and
// high byte with byte permutes (the code's magnitude is the byte index) and
// its sign bit is copied to bit 15.
struct GroupTable {
  uint32_t lo_a, lo_b, hi_a, hi_b;       // low / high bytes of products 0-3 and 4-7
};

__device__ __forceinline__ GroupTable group_table(uint32_t sf_code) {
  const uint32_t sf = __float_as_uint(e4m3_to_float(sf_code)) >> 16;   // exact bf16
  const uint32_t sf2 = sf | (sf << 16);
  const uint32_t t0 = bf16x2_mul(0x3F000000u, sf2);   // (0, 0.5) * sf
  const uint32_t t1 = bf16x2_mul(0x3FC03F80u, sf2);   // (1, 1.5) * sf
  const uint32_t t2 = bf16x2_mul(0x40404000u, sf2);   // (2, 3) * sf
  const uint32_t t3 = bf16x2_mul(0x40C04080u, sf2);   // (4, 6) * sf
  return {prmt(t0, t1, 0x6420), prmt(t2, t3, 0x6420), prmt(t0, t1, 0x7531), prmt(t2, t3, 0x7531)};
}

// 4 bytes of codes (8 values, value 2k in the low nibble of byte k) -> 8 bf16.
__device__ __forceinline__ uint4 e2m1x8_lut(uint32_t x, const GroupTable& t) {
  const uint32_t mag_even = x & 0x07070707u, mag_odd = (x >> 4) & 0x07070707u;
  const uint32_t sign = x & 0x88888888u;
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // selector: magnitude of value 2k in nibble 0, of value 2k+1 in nibble 2
    const uint32_t sel = prmt(mag_even, mag_odd, static_cast<uint32_t>(k | ((4 + k) << 4)));
    const uint32_t lo = prmt(t.lo_a, t.lo_b, sel);          // bytes 0, 2: low bytes
    const uint32_t hi = prmt(t.hi_a, t.hi_b, sel << 4);     // bytes 1, 3: high bytes
    // byte k of the sign bits into bytes 1 and 3 (zeros elsewhere): bit 11
    // (value 2k) moves to bit 15, bit 31 (value 2k+1) stays; XOR, so that a
    // negative scale byte gives the product's sign
    const uint32_t sg = prmt(sign, 0, static_cast<uint32_t>(0x0404 | (k << 4) | (k << 12)));
    o[k] = ((lo & 0x00FF00FFu) | (hi & 0xFF00FF00u)) ^ (((sg << 4) & 0x00008000u) | (sg & 0x80000000u));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// producers: the CTA's share of a 64-slot tile
// ---------------------------------------------------------------------------

// The two entry formats the producers decode (the rest of the kernel is the
// same): 352-byte nvfp4_ds_mla and 656-byte fp8_ds_mla.
enum class Entry { kNvfp4, kFp8 };

// Producer p handles rows 8p .. 8p+7 of the tile; the lanes split them by
// format (each mapping measured fastest for its format):
//  - nvfp4: lane `lane` takes row 8p + lane / 4 and, with k = lane % 4, the
//    CTA's NoPE values 64k .. 64k+63 (four 16-value groups, one 64-dim block
//    of the tile: 32 contiguous code bytes and 4 scale bytes), one entry
//    address per lane;
//  - fp8: lane `lane` takes the 16-value piece g = lane % 16 (local values
//    16g .. 16g+15) of rows 8p + lane / 16 + 2i (i < 4): every 16-byte load
//    covers 256 contiguous bytes of two rows;
//  - both: RoPE piece k = lane % 4 (values 32 half + 8k .. +7) of row
//    8p + lane / 4.
template <Entry F> struct TileRegs;
template <> struct TileRegs<Entry::kNvfp4> {
  uint4 nib[2];                          // 64 e2m1 codes (groups 4k .. 4k+3)
  uint32_t sf;                           // their four e4m3 scales, byte j = group 4k + j
  uint2 rope;                            // 8 e4m3 RoPE values
  uint32_t valid;
};
template <> struct TileRegs<Entry::kFp8> {
  uint4 code[4];                         // 16 e4m3 codes of row i
  float sc[4];                           // their 128-value tile's fp32 scale
  uint4 rope;                            // 8 bf16 RoPE values
  uint32_t valid;                        // bits 0-3: NoPE rows, bit 4: RoPE row
};

__device__ __forceinline__ const uint8_t* entry_of(const AttentionArgs& a, int32_t slot) {
  const uint32_t blk = a.block_div.div(static_cast<uint32_t>(slot));
  const uint32_t off = static_cast<uint32_t>(slot) - blk * static_cast<uint32_t>(a.block_size);
  return a.cache + static_cast<int64_t>(blk) * a.block_stride + static_cast<int64_t>(off) * a.entry_stride;
}

// The slot this lane reads for its mapping: row row0 + lane / 4 (nvfp4) or
// row0 + lane % 8 (fp8, passed on by shuffles) of a tile; -1 past top-k.
template <Entry F>
__device__ __forceinline__ int32_t tile_slot(const AttentionArgs& a, const int32_t* idx, int tile, int row0,
                                             int lane) {
  const int j = tile * kTile + row0 + (F == Entry::kNvfp4 ? lane >> 2 : lane & 7);
  return j < a.topk ? __ldg(idx + j) : -1;
}

// Issues the tile's entry loads; `mine` = tile_slot(...) of this lane, read
// a tile earlier so that the loads need not wait for it.
template <Entry F>
__device__ __forceinline__ void load_tile(const AttentionArgs& a, int32_t mine, int lane, uint32_t half,
                                          TileRegs<F>& e, bool& bad_index) {
  if (mine >= a.num_slots) bad_index = true;
  const int k = lane & 3;
  if constexpr (F == Entry::kNvfp4) {
    e.valid = mine >= 0 && mine < a.num_slots;
    if (!e.valid) return;
    const uint8_t* p = entry_of(a, mine);
    const uint4* c = reinterpret_cast<const uint4*>(p + 128 * half + 32 * k);
    e.nib[0] = __ldg(c);
    e.nib[1] = __ldg(c + 1);
    e.sf = __ldg(reinterpret_cast<const uint32_t*>(p + kNvSfOff + 16 * half + 4 * k));
    e.rope = __ldg(reinterpret_cast<const uint2*>(p + kNvRopeOff + 32 * half + 8 * k));
  } else {
    e.valid = 0;
    const int g = lane & 15;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int32_t slot = __shfl_sync(0xffffffffu, mine, (lane >> 4) + 2 * i);
      if (slot >= 0 && slot < a.num_slots) {
        const uint8_t* p = entry_of(a, slot);
        e.valid |= 1u << i;
        e.code[i] = __ldg(reinterpret_cast<const uint4*>(p + kHalf * half + 16 * g));
        e.sc[i] = __ldg(reinterpret_cast<const float*>(p + kF8ScaleOff) + 2 * half + (g >> 3));
      }
    }
    const int32_t slot = __shfl_sync(0xffffffffu, mine, lane >> 2);
    if (slot >= 0 && slot < a.num_slots) {
      e.valid |= 16u;
      e.rope = __ldg(reinterpret_cast<const uint4*>(entry_of(a, slot) + kF8RopeOff + 64 * half + 16 * k));
    }
  }
}

// 16 e4m3 codes times their tile's fp32 scale -> 16 bf16, as the fp8 gather
// upconverts them: one fp32 product rounding, one bf16 rounding.
__device__ __forceinline__ void e4m3x16_scaled(const uint4& c, float s, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 v = fmul2(__half22float2(e4m3x2_to_half2(w[i >> 1] >> (16 * (i & 1)))), make_float2(s, s));
    o[i] = pack_bf16x2(v.x, v.y);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <Entry F>
__device__ __forceinline__ void store_tile(uint32_t kbuf, int row0, int lane, const TileRegs<F>& e) {
  const int k = lane & 3;
  const uint32_t rr = row0 + (lane >> 2);              // the RoPE row (and the nvfp4 row)
  uint4 v = make_uint4(0, 0, 0, 0);
  if constexpr (F == Entry::kNvfp4) {
    const uint32_t blk = kbuf + k * kKBlock;           // this lane's 64 dims: a whole block row
#pragma unroll
    for (int j = 0; j < 4; ++j) {                      // group 4k + j -> chunks 2j, 2j + 1
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (e.valid) {
        const GroupTable t = group_table((e.sf >> (8 * j)) & 0xffu);
        const uint4& c = e.nib[j >> 1];
        lo = e2m1x8_lut((j & 1) ? c.z : c.x, t);
        hi = e2m1x8_lut((j & 1) ? c.w : c.y, t);
      }
      st_shared16(blk + sw128_offset(rr, 2 * j), lo);
      st_shared16(blk + sw128_offset(rr, 2 * j + 1), hi);
    }
    if (e.valid) v = e4m3x8_bf16(e.rope);
  } else {
    const int g = lane & 15;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t r = row0 + (lane >> 4) + 2 * i;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (e.valid & (1u << i)) e4m3x16_scaled(e.code[i], e.sc[i], lo, hi);
      // piece g: local dims 16g .. 16g+15 = block g/4, chunks 2(g%4) + {0, 1}
      const uint32_t blk = kbuf + (g >> 2) * kKBlock;
      st_shared16(blk + sw128_offset(r, 2 * (g & 3)), lo);
      st_shared16(blk + sw128_offset(r, 2 * (g & 3) + 1), hi);
    }
    if (e.valid & 16u) v = e.rope;       // bf16 as stored
  }
  st_shared16(kbuf + 4 * kKBlock + sw64_offset(rr, k), v);
}

template <Entry F>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
sparse_mla_attention_kernel(const AttentionArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(smem);
  const uint32_t qr_base = base, recv_base = base + kRecvOff;
  float* s_pair = reinterpret_cast<float*>(smem + kPairOff);        // [2][2][kRows]
  const uint32_t bar0 = base + kMiscOff;
  // k_full[3], k_empty[3], s_full[2], p_full, o_done, drain, x_full[2], x_empty[2], s_read[2],
  // recv_done[2], send_free
  const uint32_t k_full0 = bar0, k_empty0 = bar0 + 24;
  const uint32_t s_full[2] = {bar0 + 48, bar0 + 56};
  const uint32_t p_full = bar0 + 64, o_done = bar0 + 72, drain = bar0 + 80;
  const uint32_t x_full0 = bar0 + 88;    // [b]: the peer's partial S has landed in receive buffer b
  const uint32_t x_empty0 = bar0 + 104;  // [b]: the peer has read what was sent to its buffer b
  const uint32_t s_read0 = bar0 + 120;   // [b]: the exchange warps have read partial S buffer b
  const uint32_t recv_done0 = bar0 + 136;  // [b]: the softmax warps have read receive buffer b
  const uint32_t send_free = bar0 + 152;   // the last copy out of the send buffer has landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMiscOff + 168);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 172);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t token = blockIdx.x >> 1;
  const uint32_t half = cluster_rank();
  const uint32_t peer = half ^ 1u;
  const bool is_softmax = warp < 4 || (warp >= 8 && warp < 12);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(s_tmem)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(k_full0 + 8 * b, kProducerWarps);
      mbar_init(k_empty0 + 8 * b, 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(s_full[b], 1);
    mbar_init(p_full, kSoftmaxWarps);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(x_full0 + 8 * b, 1);
      mbar_init(x_empty0 + 8 * b, 1);
      mbar_init(s_read0 + 8 * b, kExchangeWarps);
      mbar_init(recv_done0 + 8 * b, kSoftmaxWarps);
    }
    mbar_init(send_free, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // Receive buffers 0 and 1 expect tiles 0 and 1 (32 KB each) before the
    // cluster barrier below, i.e. before the peer can send anything.
    const int n = (a.topk + kTile - 1) / kTile;
    for (int b = 0; b < 2 && b < n; ++b) mbar_arrive_expect_tx(x_full0 + 8 * b, kSBytes);
  }

  // The CTA's 32 RoPE query dimensions -> a 64-byte-swizzled K-major block
  // (rows >= num_heads are zero).
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + token * a.q_stride_t;
  for (int i = threadIdx.x; i < kRows * 4; i += kThreads) {
    const int row = i >> 2, c = i & 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < a.num_heads)
      v = __ldg(reinterpret_cast<const uint4*>(q + row * a.q_stride_h + KVQ_MLA_NOPE_DIM + 32 * half + 8 * c));
    st_shared16(qr_base + sw64_offset(row, c), v);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;
  // The CTA's 256 NoPE query dimensions -> TMEM (softmax warps: lane = row,
  // warp w < 4 dims 0-127, warp w + 8 dims 128-255 of the half).
  if (is_softmax) {
    const uint32_t quad = warp & 3, ch = warp >> 3;
    const int row = quad * 32 + lane;
    const uint4* src = reinterpret_cast<const uint4*>(q + row * a.q_stride_h + kHalf * half + 128 * ch);
#pragma unroll
    for (int part = 0; part < 2; ++part) {            // 64 dims = 32 columns per part
      float w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = row < a.num_heads ? __ldg(src + 8 * part + i) : make_uint4(0, 0, 0, 0);
        w[4 * i] = __uint_as_float(v.x);
        w[4 * i + 1] = __uint_as_float(v.y);
        w[4 * i + 2] = __uint_as_float(v.z);
        w[4 * i + 3] = __uint_as_float(v.w);
      }
      tmem_st32(tmem + (quad * 32u << 16) + kQCol + 64 * ch + 32 * part, w);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  cluster_sync();                        // the peer's barriers are initialised from here on

  const int32_t* idx = a.indices + token * a.indices_stride;
  const int n_tiles = (a.topk + kTile - 1) / kTile;
  bool bad_index = false;
  int mma_issued = 0;                    // MMA thread: any MMA issued
  float m = -INFINITY, l = 0.0f;         // softmax: reference max (base 2), partial sum of the row

  if (is_softmax) {
    // ---- softmax: thread = (query row, column half) ------------------------
    const uint32_t quad = warp & 3, ch = warp >> 3;         // column half: 0 = cols 0-31
    const uint32_t row_lane = quad * 32u << 16;
    const uint32_t row = quad * 32 + lane;
    const uint32_t pair_bar = 1 + quad;                      // named barrier of warps quad, quad + 8
    // Receive buffer b holds the peer's partial scores of the tiles t with
    // t % 2 == b; it is re-armed for tile t + 2 once tile t is read and
    // before the forwarder tells the peer (x_empty) that it may send there
    // again.
    // validity of this thread's 32 slots of the next tile (one per lane)
    int32_t next_slot = lane + 32 * ch < a.topk ? __ldg(idx + lane + 32 * ch) : -1;
    for (int t = 0; t < n_tiles && !*s_abort; ++t) {
      const uint32_t vm = __ballot_sync(0xffffffffu, next_slot >= 0 && next_slot < a.num_slots);
      const uint32_t cb = t & 1, par = (t >> 1) & 1;
      // tile t: this CTA's partial scores, then the peer's
      float s[32];
      if (!wait_or_abort(s_full[cb], par, s_abort)) break;
      fence_after_sync();
      tmem_ld32(tmem + row_lane + kSCol + kTile * cb + 32 * ch, s);
      if (!wait_or_abort<true>(x_full0 + 8 * cb, par, s_abort)) break;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 v = ld_shared16(recv_base + cb * kSBytes + s_offset(row, 8 * ch + c));
        const float2 a = fadd2(make_float2(s[4 * c], s[4 * c + 1]), make_float2(v.x, v.y));
        const float2 b = fadd2(make_float2(s[4 * c + 2], s[4 * c + 3]), make_float2(v.z, v.w));
        s[4 * c] = a.x;
        s[4 * c + 1] = a.y;
        s[4 * c + 2] = b.x;
        s[4 * c + 3] = b.y;
      }
      if (threadIdx.x == 0 && t + 2 < n_tiles) mbar_arrive_expect_tx(x_full0 + 8 * cb, kSBytes);
      __syncwarp();
      if (lane == 0) mbar_arrive(recv_done0 + 8 * cb);
      float hmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 y = fmul2(make_float2(s[i], s[i + 1]), make_float2(a.scale_log2, a.scale_log2));
        s[i] = (vm >> i) & 1u ? y.x : -INFINITY;
        s[i + 1] = (vm >> (i + 1)) & 1u ? y.y : -INFINITY;
        hmax = fmaxf(hmax, fmaxf(s[i], s[i + 1]));
      }
      // row max over both column halves (the barrier also orders both
      // warps' reads of the scores before either writes P over them)
      s_pair[((t & 1) * 2 + ch) * kRows + row] = hmax;
      asm volatile("bar.sync %0, 64;" :: "r"(pair_bar) : "memory");
      const float tmax = fmaxf(hmax, s_pair[((t & 1) * 2 + (ch ^ 1)) * kRows + row]);
      // Lazy rescaling: the reference max moves only when the tile's max
      // exceeds it by more than 2^8 (weights stay below 256 otherwise).
      const bool grow = tmax > m + kRescaleLog2;
      const float alpha = grow ? ex2(m - tmax) : 1.0f;          // 0 while m is -inf
      if (grow) m = tmax;
      const float m_use = m == -INFINITY ? 0.0f : m;
      uint32_t pk[16];
      float2 psum2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 d = fadd2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(-m_use, -m_use));
        pk[i] = pack_bf16x2(ex2(d.x), ex2(d.y));
        psum2 = fadd2(psum2, make_float2(bf16_lo(pk[i]), bf16_hi(pk[i])));
      }
      const float psum = psum2.x + psum2.y;
      l = l * alpha + psum;
      // The exchange warps must have read tile t's partial scores before P
      // overwrites them (normally long done), and P V of the previous tile
      // must be done before O is rescaled (the wait also keeps the
      // barrier's phases in step).
      if (!wait_or_abort(s_read0 + 8 * cb, par, s_abort)) break;
      if (t > 0 && !wait_or_abort(o_done, (t - 1) & 1, s_abort)) break;
      if (t > 0 && __any_sync(0xffffffffu, grow)) {
        fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kHalf / 64; ++c) {          // this half's 128 O columns
          float o[32];
          const uint32_t col = kOCol + 128 * ch + 32 * c;
          tmem_ld32(tmem + row_lane + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + row_lane + col, o);
        }
      }
      // P (32 values = 16 bf16 pairs of this column half) over tile t's S.
      tmem_st16(tmem + row_lane + kSCol + kTile * cb + 16 * ch, pk);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // the next slots' indices, after the arrive (a release waits for
      // accesses in flight)
      {
        const int j = (t + 1) * kTile + 32 * ch + lane;
        next_slot = j < a.topk ? __ldg(idx + j) : -1;
      }
    }
    if (n_tiles > 0) wait_or_abort(o_done, (n_tiles - 1) & 1, s_abort);
  } else if (warp < 16) {
    // ---- producers: decode tiles into the K ring ----------------------------
    const int row0 = (warp < 8 ? warp - 4 : warp - 8) * kRowsPerProducer;
    // A tile's loads are issued right after the tile before it is handed
    // over, and their latency hides behind the wait for the next free
    // stage.  (Loads go after the arrive: a release waits for every access
    // of the thread in flight.  Loading two tiles ahead, in a second
    // register set, measured slower: the producers are short of registers.)
    uint32_t stage = 0, phase = 0;                               // ring position of the next tile
    int32_t slot_next = tile_slot<F>(a, idx, 1, row0, lane);        // slots of the next tile to load
    auto produce = [&](int t, TileRegs<F>& r) -> bool {
      // stage reuse: P V of tile t - kKStages must be done
      if (t >= kKStages && !wait_or_abort(k_empty0 + 8 * stage, phase ^ 1, s_abort)) return false;
      store_tile<F>(base + kKOff + stage * kKBytes, row0, lane, r);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(k_full0 + 8 * stage);
      if (++stage == kKStages) { stage = 0; phase ^= 1; }
      if (t + 1 < n_tiles) {
        load_tile<F>(a, slot_next, lane, half, r, bad_index);
        slot_next = tile_slot<F>(a, idx, t + 2, row0, lane);
      }
      return true;
    };
    TileRegs<F> regs;
    if (n_tiles > 0) load_tile<F>(a, tile_slot<F>(a, idx, 0, row0, lane), lane, half, regs, bad_index);
    for (int t = 0; t < n_tiles; ++t)
      if (!produce(t, regs)) break;
  } else if (warp == kMmaThread / 32 && lane == 0) {
    // ---- MMA issue (one thread) -------------------------------------------
    constexpr uint32_t kIdescQK = idesc_bf16(kRows, kTile, false);
    constexpr uint32_t kIdescPV = idesc_bf16(kRows, kHalf, true);
    uint32_t qk_stage = 0, qk_phase = 0, pv_stage = 0;           // ring positions of u and t
    for (int t = 0; t < n_tiles; ++t) {
      for (int u = (t == 0 ? 0 : t + 1); u <= t + 1 && u < n_tiles; ++u) {
        // partial S[u & 1] = Q_c K_c(u)^T: 16 NoPE K-steps (A in TMEM) + 2 RoPE K-steps
        if (!wait_or_abort(k_full0 + 8 * qk_stage, qk_phase, s_abort)) goto mma_done;
        fence_after_sync();
        const uint32_t d = tmem + kSCol + kTile * (u & 1);
        // descriptors built once; a K-step adds its byte offset / 16 to the
        // start-address field (addresses stay below 256 KB: no carry out)
        const uint64_t kdesc = sw128_desc(base + kKOff + qk_stage * kKBytes, 16, 1024);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          mma_bf16_ta(d, tmem + kQCol + 8 * k, kdesc + (((k >> 2) * kKBlock + (k & 3) * 32) >> 4), kIdescQK,
                      k > 0);
        const uint64_t qrdesc = sw64_desc(qr_base);
        const uint64_t krdesc = sw64_desc(base + kKOff + qk_stage * kKBytes + 4 * kKBlock);
#pragma unroll
        for (int k = 0; k < 2; ++k) mma_bf16(d, qrdesc + 2 * k, krdesc + 2 * k, kIdescQK, 1u);
        mma_commit(s_full[u & 1]);
        mma_issued = 1;
        if (++qk_stage == kKStages) { qk_stage = 0; qk_phase ^= 1; }
      }
      // O += P(t) V(t): 4 MMAs of K = 16 slots, N = 256 value columns
      if (!wait_or_abort(p_full, t & 1, s_abort)) break;
      fence_after_sync();
      const uint64_t vdesc = sw128_desc(base + kKOff + pv_stage * kKBytes, kKBlock, 1024);
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k)
        mma_bf16_ta(tmem + kOCol, tmem + kSCol + kTile * (t & 1) + 8 * k, vdesc + 128 * k, kIdescPV,
                    (t > 0 || k > 0) ? 1u : 0u);
      mma_commit(k_empty0 + 8 * pv_stage);
      mma_commit(o_done);
      if (++pv_stage == kKStages) pv_stage = 0;
    }
  mma_done:;
  } else if (warp >= kFirstExchangeWarp && warp < kFirstExchangeWarp + kExchangeWarps) {
    // ---- exchange: each partial S to the peer as soon as it is complete ----
    // Each warp stages its 32 rows (8 KB, contiguous) in the send buffer and
    // hands them to the copy engine, which moves them into the peer's
    // receive buffer without holding up this SM's load / store pipeline; the
    // four copies of a tile complete its 32 KB on the peer's x_full.
    // Every decision to stop is taken by the whole warp (the TMEM loads are
    // warp-collective), and the warps meet only on bounded mbarrier waits.
    const uint32_t quad = warp & 3;
    const uint32_t row_lane = quad * 32u << 16;
    const uint32_t row = quad * 32 + lane;
    const uint32_t send = base + kSendOff;
    const uint32_t peer_recv0 = map_to_rank(recv_base, peer);
    const uint32_t peer_x_full0 = map_to_rank(x_full0, peer);
    for (int u = 0; u < n_tiles; ++u) {
      const uint32_t b = u & 1, par = (u >> 1) & 1;
      if (!__all_sync(0xffffffffu, wait_or_abort(s_full[b], par, s_abort))) break;
      fence_after_sync();
      float v[64];
      tmem_ld32(tmem + row_lane + kSCol + kTile * b, v);
      tmem_ld32(tmem + row_lane + kSCol + kTile * b + 32, v + 32);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_read0 + 8 * b);
      // the copy of tile u - 1 has landed in the peer: the send buffer is free
      if (u >= 1 && !__all_sync(0xffffffffu, wait_or_abort<true>(send_free, (u - 1) & 1, s_abort))) break;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_shared16(send + s_offset(row, c), make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                                       __float_as_uint(v[4 * c + 2]),
                                                       __float_as_uint(v[4 * c + 3])));
      fence_async_smem();                // the stores, visible to the copy engine
      __syncwarp();
      bool ok = true;
      if (lane == 0) {
        // the peer has read (and re-armed) its buffer b, which held tile u - 2
        ok = u < 2 || wait_or_abort<true>(x_empty0 + 8 * b, par ^ 1u, s_abort);
        const uint32_t part = quad * 32 * 256;   // this warp's rows
        if (ok) bulk_copy_to_peer(peer_recv0 + b * kSBytes + part, send + part, kSBytes / 4, peer_x_full0 + 8 * b);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else if (warp == kForwardWarp && lane == 0) {
    // ---- forwarder: the peer's copies and this CTA's reads, to the peer -----
    // For tile t: once the peer's copy has landed here, the peer's send
    // buffer is free again (send_free); once the softmax warps have read
    // receive buffer t % 2, the peer may copy tile t + 2 into it (x_empty).
    // Off the softmax warps' path: a cluster-scope release stalls the thread
    // that issues it.  The softmax warps' local release, this thread's
    // acquire and its cluster-scope release order their reads of the buffer
    // before the peer's next writes into it.
    const uint32_t peer_x_empty0 = map_to_rank(x_empty0, peer);
    const uint32_t peer_send_free = map_to_rank(send_free, peer);
    for (int t = 0; t + 1 < n_tiles; ++t) {
      if (!wait_or_abort<true>(x_full0 + 8 * (t & 1), (t >> 1) & 1, s_abort)) break;
      mbar_arrive_remote(peer_send_free);
      if (t + 2 < n_tiles) {
        if (!wait_or_abort(recv_done0 + 8 * (t & 1), (t >> 1) & 1, s_abort)) break;
        mbar_arrive_remote(peer_x_empty0 + 8 * (t & 1));
      }
    }
  }

  // Drain every MMA still in flight: one more commit tracks all of them.
  fence_before_sync();
  const bool any_mma = __syncthreads_or(mma_issued) != 0;
  fence_after_sync();
  bool aborted = *s_abort != 0;
  if (any_mma) {
    if (threadIdx.x == kMmaThread) mma_commit(drain);
    const long long start = clock64();
    while (!mbar_try_wait<false>(drain, 0)) {     // bounded, ignores the abort flag
      if (clock64() - start > kWaitCycles) { aborted = true; break; }
    }
  }
  fence_after_sync();
  if (bad_index && a.status) atomicOr(a.status, KVQ_STATUS_BAD_INDEX);
  // the row sums of the two column halves
  if (is_softmax) s_pair[(warp >> 3) * kRows + (warp & 3) * 32 + lane] = l;
  aborted = __syncthreads_or(aborted) != 0;
  if (aborted && threadIdx.x == 0 && a.status) atomicOr(a.status, KVQ_STATUS_TIMEOUT);

  if (is_softmax && !aborted) {
    const uint32_t quad = warp & 3, ch = warp >> 3;
    const uint32_t row_lane = quad * 32u << 16;
    const int row = quad * 32 + lane;
    const float l_row = s_pair[row] + s_pair[kRows + row];
    const float inv_l = l_row > 0.0f ? 1.0f / l_row : 0.0f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + token * a.out_stride_t +
                         static_cast<int64_t>(row) * a.out_stride_h + kHalf * half + 128 * ch;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float o[32];
      if (n_tiles > 0) tmem_ld32(tmem + row_lane + kOCol + 128 * ch + 32 * c, o);
      if (row < a.num_heads) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (n_tiles > 0)
            v = make_uint4(pack_bf16x2(o[8 * i] * inv_l, o[8 * i + 1] * inv_l),
                           pack_bf16x2(o[8 * i + 2] * inv_l, o[8 * i + 3] * inv_l),
                           pack_bf16x2(o[8 * i + 4] * inv_l, o[8 * i + 5] * inv_l),
                           pack_bf16x2(o[8 * i + 6] * inv_l, o[8 * i + 7] * inv_l));
          *reinterpret_cast<uint4*>(out + 32 * c + 8 * i) = v;
        }
      }
    }
    if (half == 0 && ch == 0 && a.lse != nullptr && row < a.num_heads)
      a.lse[token * a.lse_stride_t + row] =
          l_row > 0.0f ? (m + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
  // Neither CTA leaves while the peer may still write into its shared memory
  // or arrive on its barriers.
  cluster_sync();
}

}  // namespace

template <Entry F>
cudaError_t launch_attention(const AttentionArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_attention_kernel<F>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  sparse_mla_attention_kernel<F><<<static_cast<unsigned>(a.num_tokens * 2), kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sparse_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kNvfp4>(a, stream);
}

cudaError_t launch_sparse_mla_attention_fp8(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kFp8>(a, stream);
}

}  // namespace kvq
