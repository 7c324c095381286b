// kvq_attention.cu -- MLA attention read straight from the quantized paged
// caches (352-byte nvfp4_ds_mla and 656-byte fp8_ds_mla entries), on the
// fifth-generation tensor cores (tcgen05, accumulators in TMEM).  It is the
// consumer that makes the bf16 workspace unnecessary, in two forms (and, as
// a third key mode, the same dense prefill over a workspace that a gather
// filled, its keys landed by the copy engine):
//   - sparse decode: each token attends to its own top-k list of global slots
//     (vLLM PR #51724, "Enable W4A16 DSA: NVFP4 DS-MLA KV cache format for the
//     FlashMLA Sparse backend", "Key source snippets" (flashmla_sparse.py):
//     the sparse decode path serves the quantized DS-MLA formats and reads the
//     cache itself; vLLM PR #48642, "[Bugfix] Sparse MLA: enable fp8_ds_mla
//     dense prefill", "Implementation breakdown" item 3: MQA over the latent
//     cache);
//   - dense prefill: the query tokens of a request attend to every position of
//     its context, read through the block table (vLLM PR #48642, "Function
//     and motivation" and "Key source snippets", _compute_prefill_context,
//     which otherwise gathers that context into the bf16 workspace first).
// For a query row (token t, head h) and its keys j:
//   s_j = scale * (q[t,h] . k_j)        k_j = the entry's 576 decoded values
//   o[t,h] = sum_j softmax(s)_j * k_j[0:512],   lse[t,h] = log sum_j exp(s_j)
//
// Design: one CTA per (block of 128 query rows, half c of the 512 value
// dimensions), one CTA per SM, no cluster.  A row block is the heads of one
// decode token, or, for prefill, 128 consecutive (token, head) rows of one
// request, so that every decoded key tile feeds the rows of several query
// tokens when a token has fewer than 128 heads.  The 128 x 512 fp32 output of
// a row block would fill all of an SM's TMEM, so each CTA keeps O for its 256
// value columns and computes the whole score tile Q K^T itself (the two CTAs
// of a row block duplicate that product; in exchange no partial scores travel
// between SMs and nothing on a tile's critical path waits for another SM).
// Per CTA (13 warps):
//   - TMEM: O [0, 256), the CTA's own 256 NoPE query dimensions as bf16 pairs
//     [256, 384) (the A operand of their K-steps), the score tile S (128 x 64
//     fp32) double buffered in [384, 512); P (bf16) is written over the first
//     half of its own S buffer as the A operand of P V;
//   - shared memory: the other 256 NoPE query dimensions and the 64 RoPE
//     dimensions (80 KB); key tile group A, the 320 dimensions no value column
//     of this CTA uses (2 stages, free again once their K-steps are done);
//     key tile group B, this CTA's own 256 dimensions, which are also the V
//     operand of P V (2 stages, free once P V is done);
//   - eight producer warps decode group A of each 64-key tile, then group B,
//     8 rows each (e2m1 x e4m3 products formed exactly by byte-permute table
//     lookups; fp8 codes times their tile scale as the fp8 gather does);
//     group B of tile t is decoded as soon as P V of tile t - 2 is done,
//     while the 20 group-A K-steps of tile t run;
//   - one thread issues the MMAs: S(u) = the 20 group-A K-steps and the 16
//     group-B K-steps of Q K^T, then O += P(t) V(t) (4 K-steps, N = 256), in
//     the order S(0), S(1), PV(0), S(2), PV(1), ...: the 36 K-steps of the
//     next tile's scores run while the softmax of this tile is computed;
//   - four softmax warps (TMEM lanes 0-127, one query row of 64 scores per
//     thread) run the online softmax in base 2 with lazy rescaling (the
//     reference maximum moves only when a tile exceeds it by 2^8), write P as
//     bf16 into TMEM and rescale their O row when the reference moved; the
//     denominator sums the bf16-rounded P.
// Start-up: the query rows arrive by nine tensor-map copies (the own
// dimensions through the idle key stages into TMEM); the epilogue writes each
// output row by one bulk copy.  Split over the keys (small batches): a CTA
// pair per (row block, key range) writes a normalised fp32 partial row and
// its base-2 log-sum-exp, and combine_splits_kernel weighs the ranges.
//
// Every wait is bounded; on expiry (or when another role of the CTA gave up)
// the CTA records KVQ_STATUS_TIMEOUT, stops issuing work, waits (with its own
// long limit) for the MMAs in flight, frees its TMEM, leaves its outputs
// unwritten and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>

#include "kvq.h"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kHalf = KVQ_MLA_NOPE_DIM / 2;                  // 256 value columns per CTA
constexpr int kRows = 128;                                   // query rows per CTA
constexpr int kTile = 64;                                    // keys per tile (N of Q K^T)
// Warp roles: 0-3 softmax (warp w: TMEM lanes 32 w .. +31), 4-11 producers,
// 12 MMA (one thread).  13 warps put at most 4 on an SM sub-partition: 128
// registers per thread.
constexpr int kSoftmaxWarps = 4;
constexpr int kFirstProducerWarp = 4;
constexpr int kProducerWarps = 8;
constexpr int kMmaWarp = 12;
constexpr int kThreads = 13 * 32;                            // 416
constexpr int kNvRopeOff = 256, kNvSfOff = 320;              // nvfp4_ds_mla entry
constexpr int kF8ScaleOff = 512, kF8RopeOff = 528;           // fp8_ds_mla entry
constexpr float kRescaleLog2 = 8.0f;                         // lazy rescale threshold (base 2)

// Shared memory (offsets from a 1024-byte aligned base).  Every block is 64
// dimensions wide (128-byte rows, 128-byte swizzle, K-major).
#ifndef KVQ_ATTN_A_STAGES
#define KVQ_ATTN_A_STAGES 2
#endif
#ifndef KVQ_ATTN_B_STAGES
#define KVQ_ATTN_B_STAGES 2
#endif
constexpr int kAStages = KVQ_ATTN_A_STAGES;
constexpr int kBStages = KVQ_ATTN_B_STAGES;
constexpr uint32_t kQBlock = kRows * 128;                    // 16 KB: 64 query dims of 128 rows
constexpr uint32_t kKBlock = kTile * 128;                    // 8 KB: 64 key dims of 64 keys
constexpr uint32_t kQOff = 0;                                // 4 other-NoPE blocks + RoPE: 80 KB
constexpr uint32_t kAOff = kQOff + 5 * kQBlock;              // group A: 4 other-NoPE blocks + RoPE per stage
constexpr uint32_t kAStage = 5 * kKBlock;
constexpr uint32_t kBOff = kAOff + kAStages * kAStage;       // group B: 4 own-NoPE blocks per stage
constexpr uint32_t kBStage = 4 * kKBlock;
constexpr uint32_t kMiscOff = kBOff + kBStages * kBStage;
constexpr uint32_t kBiasOff = kMiscOff + 256;                // per softmax warp: 64 fp32 score biases
constexpr uint32_t kLastOff = kBiasOff + kSoftmaxWarps * 256;  // per warp: the last valid key (list search)
constexpr uint32_t kSmemBytes = kLastOff + 64 + 1024;          // + alignment
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103a CTA");
// The key stages (group A then group B, contiguous) are idle before the
// first tile and after the last: they stage the own query dimensions on their
// way to TMEM and the output rows on their way out.
constexpr uint32_t kStagingOff = kAOff;
constexpr uint32_t kStageRowBytes = 528;                     // an output row (512 bytes) + 16
constexpr uint32_t kPartRowBytes = 1040;                     // a partial fp32 row (1 KB) + 16
static_assert(kMiscOff - kStagingOff >= kRows * kPartRowBytes && kMiscOff - kStagingOff >= 4 * kQBlock,
              "the staging fits the key stages");
static_assert(kAOff % 1024 == 0 && kBOff % 1024 == 0 && kAStage % 1024 == 0 && kBStage % 1024 == 0,
              "1024-byte swizzle atoms");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;
constexpr uint32_t kQCol = 256;
constexpr uint32_t kSCol = 384;

// Limit of every wait of a role on another role, in SM clock cycles (the
// default is about 2 s at 2 GHz).  The final wait for the CTA's own MMAs has
// its own, separate limit, so that a shortened role limit never cuts it short.
#ifndef KVQ_ATTN_WAIT_CYCLES
#define KVQ_ATTN_WAIT_CYCLES 4000000000LL
#endif
constexpr long long kWaitCycles = KVQ_ATTN_WAIT_CYCLES;
constexpr long long kDrainCycles = 4000000000LL;

// ---------------------------------------------------------------------------
// tcgen05 / mbarrier helpers (inline PTX, sm_100a family)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor with the 128-byte swizzle (1024-byte atoms
// of 8 rows x 128 bytes); lbo / sbo in bytes.
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
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

// Tensor-map tile loads into shared memory, completing on an mbarrier
// (coordinates innermost first; the innermost one times 2 bytes is a multiple
// of 16 here).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}

// One bounded wait step: the thread sleeps in the barrier (up to about 1 ms,
// woken when the phase completes) instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
  return done != 0;
}

// Bounded wait that also gives up when another role of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag || clock64() - start > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// The same taken by a whole warp: every lane waits, and the warp goes on
// only if every lane saw the phase complete, so that the warp-collective
// instructions after it (TMEM loads and stores, shuffles) are reached by all
// of its lanes or by none.
__device__ __forceinline__ bool warp_wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
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

// 64 consecutive fp32 TMEM columns of this warp's 32 lanes in one load.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
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

// No memory clobber: the decode arithmetic around these stores may be
// scheduled across them (the fence that publishes the stores to the tensor
// cores is a volatile asm with a memory clobber, which stays after them).
__device__ __forceinline__ void st_shared16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// 16 bytes global -> shared without passing through registers; with
// src_bytes = 0 nothing is read and the 16 bytes are zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from shared to global memory by the copy engine, tracked by the thread's
// bulk group; the thread waits only until its source has been read.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(src), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// L2 prefetch hints: `bytes` (a multiple of 16, 16-byte aligned) from addr,
// or the 128-byte line holding addr.
__device__ __forceinline__ void prefetch_l2_bulk(const void* addr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(addr), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_line(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(addr) : "memory");
}

// 2^x for x <= 0 (0 for -inf): the hardware approximation, relative error
// below 2^-22, flushed to zero below 2^-126 (weights that small vanish next
// to the largest weight, which is at least 2^-8).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input max, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// lo_acc += the bf16 in bits 15:0 of p, hi_acc += the one in bits 31:16, each
// an fp32 addition of the exactly widened bf16 (mixed-precision add, one
// instruction each: no shift or mask to widen the halves first).
__device__ __forceinline__ void add_bf16x2(float& lo_acc, float& hi_acc, uint32_t p) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
      : "+f"(lo_acc), "+f"(hi_acc) : "r"(p));
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
// with four bf16x2 multiplies and kept as two 8-byte tables, one of their low
// and one of their high bytes.
struct GroupTable {
  uint32_t lo_a, lo_b, hi_a, hi_b;       // low / high bytes of products 0-3 and 4-7
};

__device__ __forceinline__ GroupTable group_table(float sf_f32) {
  const uint32_t sf2 = prmt(__float_as_uint(sf_f32), 0u, 0x3232);       // its bf16 (exact) in both halves
  const uint32_t t0 = bf16x2_mul(0x3F000000u, sf2);   // (0, 0.5) * sf
  const uint32_t t1 = bf16x2_mul(0x3FC03F80u, sf2);   // (1, 1.5) * sf
  const uint32_t t2 = bf16x2_mul(0x40404000u, sf2);   // (2, 3) * sf
  const uint32_t t3 = bf16x2_mul(0x40C04080u, sf2);   // (4, 6) * sf
  return {prmt(t0, t1, 0x6420), prmt(t2, t3, 0x6420), prmt(t0, t1, 0x7531), prmt(t2, t3, 0x7531)};
}

// 4 bytes of codes (8 values, value 2k in the low nibble of byte k) -> 8 bf16.
// With the sign bits cleared, the eight code nibbles are byte selectors into
// the group's tables: one byte permute gathers the low (or high) bytes of
// four values' products, two more interleave them into bf16 pairs.  A code's
// sign bit is the top bit of a byte of x (odd values) or of x << 4 (even
// values); one byte permute in sign-replicate mode spreads the signs of four
// values over four bytes, in the order of their high bytes, and the sign bits
// are XORed into those high bytes before the interleave (so a negative scale
// byte still gives the product's sign): 15 operations per 8 values.  An
// exhaustive CPU emulation of the byte logic against the exact products over
// every code and scale byte was run, and of this sign placement against the
// earlier one (sign XORed into each bf16 pair after the interleave).
__device__ __forceinline__ uint4 e2m1x8_bf16(uint32_t x, const GroupTable& t) {
  const uint32_t mag = x & 0x77777777u, mag_hi = mag >> 16, x4 = x << 4;
  const uint32_t s0 = prmt(x, x4, 0x9D8C), s1 = prmt(x, x4, 0xBFAE);   // values 0-3, 4-7
  const uint32_t l0 = prmt(t.lo_a, t.lo_b, mag), h0 = prmt(t.hi_a, t.hi_b, mag) ^ (s0 & 0x80808080u);
  const uint32_t l1 = prmt(t.lo_a, t.lo_b, mag_hi), h1 = prmt(t.hi_a, t.hi_b, mag_hi) ^ (s1 & 0x80808080u);
  return make_uint4(prmt(l0, h0, 0x5140), prmt(l0, h0, 0x7362), prmt(l1, h1, 0x5140), prmt(l1, h1, 0x7362));
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

// ---------------------------------------------------------------------------
// rows and keys
// ---------------------------------------------------------------------------

enum class Entry { kNvfp4, kFp8 };          // 352-byte nvfp4_ds_mla, 656-byte fp8_ds_mla
// per-token slot lists; a request's whole context through its block table;
// the same context as rows of a gathered bf16 workspace
enum class Keys { kSparse, kDense, kWorkspace };

// What one CTA works on: its query rows and its list of keys.
struct Block {
  bool live;                  // false: the CTA has no rows (prefill grid padding)
  int64_t token0;             // sparse: the token; dense: the request's first query token
  int32_t row0;               // dense: first packed (token, head) row of the block
  int32_t rows;               // rows of the block (query rows past it are zero)
  int32_t request;            // dense: the request
  int32_t n_keys;             // keys of the block: topk or the context, or the block's range of them
  int32_t split;              // split over the keys: the block's range
  int32_t key0;               // dense: the context position of the block's key 0
  int64_t ws_row0;            // workspace: the row of context position 0
  const int32_t* idx;         // sparse: the block's part of the token's slot list
};

// The block of CTA (bx, by); `report`: record a skipped request in the
// status word (only the CTA's own block does).
template <Keys K>
__device__ __forceinline__ Block block_of(const AttentionArgs& a, uint32_t bx, uint32_t by, bool report) {
  Block b{};
  if constexpr (K == Keys::kSparse) {
    b.live = true;
    b.row0 = 0;
    b.rows = a.num_heads;
    if (a.num_splits > 1) {
      // CTA pair (token, split): keys [split * split_keys, +split_keys) of the list
      const uint32_t unit = bx >> 1, splits = static_cast<uint32_t>(a.num_splits);
      b.token0 = unit / splits;
      b.split = static_cast<int32_t>(unit - static_cast<uint32_t>(b.token0) * splits);
      const int32_t key0 = b.split * a.split_keys;
      b.n_keys = max(0, min(a.topk - key0, a.split_keys));
      b.idx = a.indices + b.token0 * a.indices_stride + key0;
    } else {
      b.token0 = bx >> 1;
      b.n_keys = a.topk;
      b.idx = a.indices + b.token0 * a.indices_stride;
    }
  } else {
    b.request = static_cast<int32_t>(by);
    const int32_t q0 = __ldg(a.query_start + b.request), q1 = __ldg(a.query_start + b.request + 1);
    if (q0 < 0 || q1 < q0 || q1 > a.num_tokens || q1 - q0 > a.max_query_len) {
      // a request whose query tokens are not inside [0, num_tokens) or longer
      // than max_query_len: skipped
      if (report && bx == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, KVQ_STATUS_BAD_BATCH);
      b.live = false;
      return b;
    }
    const int64_t total = static_cast<int64_t>(q1 - q0) * a.num_heads;
    const int32_t ctx = max(0, __ldg(a.context_lens + b.request));
    if constexpr (K == Keys::kWorkspace) {
      b.ws_row0 = __ldg(a.ws_starts + b.request);
      if (b.ws_row0 < 0 || b.ws_row0 + ctx > a.ws_rows) {
        // a context that does not lie inside the workspace: skipped
        if (report && bx == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, KVQ_STATUS_BAD_BATCH);
        b.live = false;
        return b;
      }
    }
    uint32_t unit = bx >> 1;
    if (a.num_splits > 1) {
      // CTA pair (row block, split): context positions [split * split_keys,
      // +split_keys), the last range also every position past the others
      const uint32_t splits = static_cast<uint32_t>(a.num_splits);
      const uint32_t rb = unit / splits;
      b.split = static_cast<int32_t>(unit - rb * splits);
      unit = rb;
      b.key0 = b.split * a.split_keys;
      b.n_keys = b.split == a.num_splits - 1 ? max(0, ctx - b.key0) : max(0, min(ctx - b.key0, a.split_keys));
    } else {
      b.n_keys = ctx;
    }
    b.row0 = static_cast<int32_t>(unit) * kRows;
    b.live = q1 > q0 && b.row0 < total;
    b.token0 = q0;
    b.rows = static_cast<int32_t>(min(static_cast<int64_t>(kRows), total - b.row0));
  }
  return b;
}

// Token and head of query row `row` (< b.rows) of the block.
template <Keys K>
__device__ __forceinline__ void row_of(const AttentionArgs& a, const Block& b, int row, int64_t& token,
                                       int32_t& head) {
  if constexpr (K == Keys::kSparse) {
    token = b.token0;
    head = row;
  } else {
    const uint32_t g = static_cast<uint32_t>(b.row0 + row);
    const uint32_t tk = a.head_div.div(g);
    token = b.token0 + tk;
    head = static_cast<int32_t>(g - tk * a.head_div.d);
  }
}

// The CTAs of a launch run in waves of `a.wave` (one per SM, in launch
// order), every CTA of this kernel taking about as long as the others, so the
// CTA that follows this one onto some SM is about `a.wave` places later in
// launch order.  Halfway through its keys a CTA asks L2 for that CTA's query
// rows (an even CTA) or its slot list (an odd one), so that the next wave's
// start-up reads come from L2 and not all at once from HBM.  Only a hint: a
// wrong guess costs an L2 fill and nothing else.
template <Keys K>
__device__ __forceinline__ void prefetch_next_wave(const AttentionArgs& a, uint32_t row) {
  const uint64_t grid = static_cast<uint64_t>(gridDim.x) * gridDim.y;
  const uint64_t id = static_cast<uint64_t>(blockIdx.y) * gridDim.x + blockIdx.x + static_cast<uint32_t>(a.wave);
  if (a.wave <= 0 || id >= grid) return;
  const Block nb = block_of<K>(a, static_cast<uint32_t>(id % gridDim.x), static_cast<uint32_t>(id / gridDim.x), false);
  if (!nb.live) return;
  if ((id & 1) == 0) {
    if (row < static_cast<uint32_t>(nb.rows)) {
      int64_t token;
      int32_t head;
      row_of<K>(a, nb, static_cast<int>(row), token, head);
      prefetch_l2_bulk(static_cast<const __nv_bfloat16*>(a.q) + token * a.q_stride_t + head * a.q_stride_h,
                       KVQ_WORKSPACE_DIM * 2);
    }
  } else if constexpr (K == Keys::kSparse) {
    for (int j = static_cast<int>(row) * 32; j < nb.n_keys; j += kRows * 32) prefetch_l2_line(nb.idx + j);
  }
}

// The raw index of key j, loaded ahead of its use: sparse, the slot (< 0
// unused; -1 also past the list); dense, the block id of position j's
// block-table column (-1 past the context; INT32_MAX for a column past the
// table or a negative id, which makes the position out of range).
template <Keys K>
__device__ __forceinline__ int32_t key_raw(const AttentionArgs& a, const Block& b, int j) {
  if (j >= b.n_keys) return -1;
  if constexpr (K == Keys::kSparse) {
    return __ldg(b.idx + j);
  } else if constexpr (K == Keys::kWorkspace) {
    return 0;                                 // every position inside the context is a key
  } else {
    const uint32_t col = a.block_div.div(static_cast<uint32_t>(b.key0 + j));
    if (col >= static_cast<uint32_t>(a.block_table_width)) return INT32_MAX;
    const int32_t id = __ldg(a.block_table + b.request * a.block_table_stride + col);
    return id < 0 ? INT32_MAX : id;
  }
}

// Whether a key with this raw index takes part.
template <Keys K>
__device__ __forceinline__ bool raw_valid(const AttentionArgs& a, int32_t raw) {
  if constexpr (K == Keys::kWorkspace) return raw >= 0;
  return raw >= 0 && (K == Keys::kSparse ? raw < a.num_slots : raw < a.num_blocks);
}

// Entry of key j from its raw index, or nullptr when the key is unused or out
// of range (bad_index set for the latter).
template <Keys K>
__device__ __forceinline__ const uint8_t* key_entry(const AttentionArgs& a, const Block& b, int32_t raw, int j,
                                                    bool& bad_index) {
  if (raw < 0) return nullptr;
  if (!raw_valid<K>(a, raw)) {
    bad_index = true;
    return nullptr;
  }
  uint32_t blk, off;
  if constexpr (K == Keys::kSparse) {
    blk = a.block_div.div(static_cast<uint32_t>(raw));
    off = static_cast<uint32_t>(raw) - blk * static_cast<uint32_t>(a.block_size);
  } else {
    const uint32_t p = static_cast<uint32_t>(b.key0 + j);
    blk = static_cast<uint32_t>(raw);
    off = p - a.block_div.div(p) * static_cast<uint32_t>(a.block_size);
  }
  return a.cache + static_cast<int64_t>(blk) * a.block_stride + static_cast<int64_t>(off) * a.entry_stride;
}

// ---------------------------------------------------------------------------
// producers: both groups of every key tile, 8 rows per warp
// ---------------------------------------------------------------------------
//
// Producer thread (w, lane) takes tile row r = 8 w + lane % 8 and k = lane /
// 8: of group A the other half's NoPE block k (dimensions 256 (1 - c) + 64 k
// .. +64) and the RoPE dimensions 16 k .. +16, of group B the own NoPE block
// k (256 c + 64 k .. +64).  All eight warps decode group A of a tile, then
// group B, so a group's decode is spread over all of them.  The 8 lanes of a
// quarter warp write 8 consecutive rows of one block, whose 128-byte swizzle
// puts a given 16-byte chunk in 8 different bank groups.

template <Entry F, bool kRope> struct PartRegs;
template <bool kRope> struct PartRegs<Entry::kNvfp4, kRope> {
  uint4 code[2];                         // 64 e2m1 codes (4 groups)
  uint32_t sf;                           // their 4 e4m3 scales
  uint4 rope;                            // group A: 16 e4m3 RoPE values
};
template <bool kRope> struct PartRegs<Entry::kFp8, kRope> {
  uint4 code[4];                         // 64 e4m3 codes
  float sc;                              // the scale of their 128-value tile
  uint4 rope[2];                         // group A: 16 bf16 RoPE values
};

// Issues the loads of this thread's share of one key's entry: NoPE
// dimensions nope0 .. nope0 + 63 and, with kRope, the RoPE dimensions
// 16 k .. 16 k + 15.  For p = nullptr (an unused key) the registers are
// zeroed instead: zero codes and a zero scale decode to zeros, so the decode
// needs no per-value select.
template <Entry F, bool kRope>
__device__ __forceinline__ void load_part(const uint8_t* p, int nope0, int k, PartRegs<F, kRope>& e) {
  if (p == nullptr) {
    e = PartRegs<F, kRope>{};
    return;
  }
  if constexpr (F == Entry::kNvfp4) {
    const uint4* c = reinterpret_cast<const uint4*>(p + nope0 / 2);
    e.code[0] = __ldg(c);
    e.code[1] = __ldg(c + 1);
    e.sf = __ldg(reinterpret_cast<const uint32_t*>(p + kNvSfOff + nope0 / 16));
    if constexpr (kRope) e.rope = __ldg(reinterpret_cast<const uint4*>(p + kNvRopeOff + 16 * k));
  } else {
    const uint4* c = reinterpret_cast<const uint4*>(p + nope0);
#pragma unroll
    for (int i = 0; i < 4; ++i) e.code[i] = __ldg(c + i);
    e.sc = __ldg(reinterpret_cast<const float*>(p + kF8ScaleOff) + nope0 / 128);
    if constexpr (kRope) {
      const uint4* r = reinterpret_cast<const uint4*>(p + kF8RopeOff + 32 * k);
      e.rope[0] = __ldg(r);
      e.rope[1] = __ldg(r + 1);
    }
  }
}

// Decodes this thread's share of a key row into registers: chunks 2g, 2g + 1
// hold NoPE group g and, with kRope, v[8], v[9] the RoPE values (an unused
// key's zeroed registers decode to zeros).
template <Entry F, bool kRope>
__device__ __forceinline__ void decode_part(const PartRegs<F, kRope>& e, uint4 (&v)[kRope ? 10 : 8]) {
  float2 sf01, sf23;                     // nvfp4: the 4 group scales, exact
  if constexpr (F == Entry::kNvfp4) {
    sf01 = __half22float2(e4m3x2_to_half2(e.sf));
    sf23 = __half22float2(e4m3x2_to_half2(e.sf >> 16));
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if constexpr (F == Entry::kNvfp4) {
      const GroupTable t = group_table(g == 0 ? sf01.x : g == 1 ? sf01.y : g == 2 ? sf23.x : sf23.y);
      const uint4& c = e.code[g >> 1];
      v[2 * g] = e2m1x8_bf16((g & 1) ? c.z : c.x, t);
      v[2 * g + 1] = e2m1x8_bf16((g & 1) ? c.w : c.y, t);
    } else {
      e4m3x16_scaled(e.code[g], e.sc, v[2 * g], v[2 * g + 1]);
    }
  }
  if constexpr (kRope) {
    if constexpr (F == Entry::kNvfp4) {
      v[8] = e4m3x8_bf16(make_uint2(e.rope.x, e.rope.y));
      v[9] = e4m3x8_bf16(make_uint2(e.rope.z, e.rope.w));
    } else {
      v[8] = e.rope[0];                                  // bf16 as stored
      v[9] = e.rope[1];
    }
  }
}

// Stores a decoded share into tile row r: NoPE block `blk` (chunks 0-7) and,
// with kRope, RoPE chunks 2k, 2k + 1 of the block at `rope_blk`.
template <bool kRope>
__device__ __forceinline__ void write_part(uint32_t blk, uint32_t rope_blk, uint32_t r, int k,
                                           const uint4 (&v)[kRope ? 10 : 8]) {
  // blocks are 1024-byte aligned: row r's chunk c is at (blk + 128 r + 16 (r % 8)) XOR 16 c
  const uint32_t row = r * 128u + ((r & 7u) << 4);
  const uint32_t b = blk + row;
#pragma unroll
  for (int c = 0; c < 8; ++c) st_shared16(b ^ (static_cast<uint32_t>(c) << 4), v[c]);
  if constexpr (kRope) {
    const uint32_t rb = rope_blk + row;
    st_shared16(rb ^ (static_cast<uint32_t>(2 * k) << 4), v[8]);
    st_shared16(rb ^ (static_cast<uint32_t>(2 * k + 1) << 4), v[9]);
  }
}

template <Entry F, Keys K>
__global__ void __launch_bounds__(kThreads, 1) mla_attention_kernel(const AttentionArgs a,
                                                                    const __grid_constant__ CUtensorMap qmap,
                                                                    const __grid_constant__ CUtensorMap kmap) {
  const Block blk = block_of<K>(a, blockIdx.x, blockIdx.y, true);
  if (!blk.live) return;                 // uniform over the CTA, before any barrier or allocation
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_u32(smem);
  const uint32_t bar0 = base + kMiscOff;
  const uint32_t a_full0 = bar0, a_empty0 = bar0 + 8 * kAStages;
  const uint32_t b_full0 = bar0 + 16 * kAStages, b_empty0 = b_full0 + 8 * kBStages;
  const uint32_t s_full0 = b_full0 + 16 * kBStages;                 // [2]
  const uint32_t p_full = s_full0 + 16, o_done = s_full0 + 24, drain = s_full0 + 32;
  static_assert(16 * kAStages + 16 * kBStages + 40 <= 160, "barriers fit below the flags");
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMiscOff + 160);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 164);
  const uint32_t q_full = bar0 + 168;    // the query rows' tensor-map loads
  int* s_last = reinterpret_cast<int*>(smem + kMiscOff + 176);   // [13]: per warp, the last valid key
  static_assert(176 + 4 * (kThreads / 32) <= 256, "the per-warp key bounds fit the flags area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t half = blockIdx.x & 1;  // value columns [256 half, +256)
  const int other = kHalf * (1 - static_cast<int>(half)), own = kHalf * static_cast<int>(half);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(s_tmem)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    // a stage is full when the producer warps have stored it, or (workspace
    // keys) when the copy engine has landed it after its issuer's arrival
    constexpr uint32_t kFullCount = K == Keys::kWorkspace ? 1 : kProducerWarps;
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(a_full0 + 8 * s, kFullCount);
      mbar_init(a_empty0 + 8 * s, 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(b_full0 + 8 * s, kFullCount);
      mbar_init(b_empty0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(s_full0 + 8 * s, 1);
    mbar_init(p_full, kSoftmaxWarps);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_full, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.q_tma) {
      // Query rows -> shared memory, nine 16 KB tiles by the copy engine: the
      // other half's 256 NoPE dimensions and the 64 RoPE dimensions as five
      // 128-byte-swizzled K-major blocks (the A operand of the group-A
      // K-steps), and the CTA's own 256 NoPE dimensions staged in the same
      // layout in the key stages on their way to TMEM.  Rows past the tensor
      // are zero-filled; rows past the block's rows (dense form) hold other
      // query rows, whose results are never written.
      mbar_arrive_expect_tx(q_full, 9 * kQBlock);
#pragma unroll 1
      for (int j = 0; j < 9; ++j) {
        const int dim = j < 4 ? other + 64 * j : j == 4 ? KVQ_MLA_NOPE_DIM : own + 64 * (j - 5);
        const uint32_t dst = j < 5 ? base + kQOff + j * kQBlock : base + kStagingOff + (j - 5) * kQBlock;
        if constexpr (K == Keys::kSparse)
          tma_load_3d(dst, &qmap, dim, 0, static_cast<int32_t>(blk.token0), q_full);
        else
          tma_load_2d(dst, &qmap, dim, static_cast<int32_t>(blk.token0 * a.num_heads + blk.row0), q_full);
      }
    }
  }

  // Without a tensor map: the same nine blocks by asynchronous 16-byte copies,
  // all in flight at once (rows past the block's rows zero-filled).
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  for (int i = a.q_tma ? kRows * 72 : threadIdx.x; i < kRows * 9 * 8; i += kThreads) {
    const int row = i / 72, rem = i % 72, j = rem >> 3, c = rem & 7;   // block j: 0-3 other, 4 RoPE, 5-8 own
    const __nv_bfloat16* src = q;
    uint32_t bytes = 0;
    if (row < blk.rows) {
      int64_t token;
      int32_t head;
      row_of<K>(a, blk, row, token, head);
      const int dim = j < 4 ? other + 64 * j : j == 4 ? KVQ_MLA_NOPE_DIM : own + 64 * (j - 5);
      src = q + token * a.q_stride_t + head * a.q_stride_h + dim + 8 * c;
      bytes = 16;
    }
    const uint32_t blk_base = j < 5 ? base + kQOff + j * kQBlock : base + kStagingOff + (j - 5) * kQBlock;
    cp_async16(blk_base + sw128_offset(row, c), src, bytes);
  }

  // Sparse lists often end in unused entries (a context shorter than the
  // list): the tiles past the last valid key are skipped (they would add
  // nothing; an out-of-range entry among them is still reported).  Each
  // thread checks one of the last kThreads entries here; only a list whose
  // last kThreads entries are all unused is searched further (below).  The
  // first tile's loads go by the whole list.
  bool bad_index = false;
  if constexpr (K == Keys::kSparse) {
    const int j = blk.n_keys - 1 - static_cast<int>(threadIdx.x);
    int last = -1;
    if (j >= 0) {
      const int32_t raw = __ldg(blk.idx + j);
      if (raw_valid<K>(a, raw)) last = j;
      else if (raw >= 0) bad_index = true;
    }
    last = __reduce_max_sync(0xffffffffu, last);
    if (lane == 0) s_last[warp] = last;
  }
  const int n_tiles0 = (blk.n_keys + kTile - 1) / kTile;
  const bool is_softmax = warp < kSoftmaxWarps;
  const bool is_producer = warp >= kFirstProducerWarp && warp < kMmaWarp;
  // Producer row r of a tile, dimension block k of its parts (see below).
  const uint32_t r = 8 * (warp - kFirstProducerWarp) + (lane & 7);
  const int k = lane >> 3;
  const int a_nope0 = other + 64 * k, b_nope0 = own + 64 * k;
  // Row r's raw index is loaded two tiles ahead and becomes an entry address
  // one tile ahead, when the entry's loads are issued; the first tile's are
  // issued here, while the query copies land.
  PartRegs<F, true> ra;
  PartRegs<F, false> rb;
  const uint8_t* cur = nullptr;
  int32_t raw_next = 0, raw_next2 = 0;
  if (K != Keys::kWorkspace && is_producer) {
    cur = key_entry<K>(a, blk, key_raw<K>(a, blk, r), r, bad_index);
    raw_next = key_raw<K>(a, blk, kTile + r);
    raw_next2 = key_raw<K>(a, blk, 2 * kTile + r);
    if (n_tiles0 > 0) {
      load_part<F, true>(cur, a_nope0, k, ra);
      load_part<F, false>(cur, b_nope0, k, rb);
    }
  }
  if (!a.q_tma) {
    cp_async_wait_all();
    fence_async_smem();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;
  int n_tiles = n_tiles0;
  int last_key = -1;
  if constexpr (K == Keys::kSparse) {
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) last_key = max(last_key, s_last[w]);
    if (last_key < 0 && blk.n_keys > kThreads) {
      // the last kThreads entries are all unused: search the rest of the list
      int last = -1;
      for (int j = threadIdx.x; j < blk.n_keys - kThreads; j += kThreads) {
        const int32_t raw = __ldg(blk.idx + j);
        if (raw_valid<K>(a, raw)) last = j;
        else if (raw >= 0) bad_index = true;
      }
      last = __reduce_max_sync(0xffffffffu, last);
      if (lane == 0) reinterpret_cast<volatile int*>(smem + kLastOff)[warp] = last;
    }
  }
  // The CTA's own 256 NoPE query dimensions: staging -> TMEM (softmax warp w:
  // lane = row 32 w + lane), once the tensor-map loads have landed.
  if (is_softmax && (!a.q_tma || warp_wait_or_abort(q_full, 0, s_abort))) {
    const uint32_t row = warp * 32 + lane;
#pragma unroll 1
    for (int part = 0; part < 4; ++part) {            // 64 dims = 32 columns per part
      float w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = ld_shared16(base + kStagingOff + part * kQBlock + sw128_offset(row, i));
        w[4 * i] = __uint_as_float(v.x);
        w[4 * i + 1] = __uint_as_float(v.y);
        w[4 * i + 2] = __uint_as_float(v.z);
        w[4 * i + 3] = __uint_as_float(v.w);
      }
      tmem_st32(tmem + (warp * 32u << 16) + kQCol + 32 * part, w);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if constexpr (K == Keys::kSparse) {
    if (last_key < 0 && blk.n_keys > kThreads) {
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w)
        last_key = max(last_key, reinterpret_cast<volatile int*>(smem + kLastOff)[w]);
    }
    n_tiles = (last_key + kTile) / kTile;            // tiles up to the last valid key
  }

  int mma_issued = 0;                    // MMA thread: any MMA issued
  float m = -INFINITY, l = 0.0f;         // softmax: reference max (base 2), partial sum of the row

  if (is_softmax) {
    // ---- softmax: thread = query row ----------------------------------------
    const uint32_t row_lane = warp * 32u << 16;
    // raw indices of this lane's keys (lane and 32 + lane) of the next two
    // tiles: loaded a tile before their validity is needed
    int32_t raw1_lo = key_raw<K>(a, blk, lane), raw1_hi = key_raw<K>(a, blk, 32 + lane);
    int32_t raw2_lo = key_raw<K>(a, blk, kTile + lane), raw2_hi = key_raw<K>(a, blk, kTile + 32 + lane);
    // Every wait is bounded and taken by the whole warp; a warp that gives up
    // leaves its loop and meets no other warp before the end.
    // The tile's key validity is the same for every row: each lane writes the
    // score bias (0, or -inf for an unused or bad key) of keys lane and 32 +
    // lane to the warp's bias row, and every lane reads the 64 back as
    // broadcasts, so that masking costs one fused multiply-add per score pair.
    const uint32_t bias_row = base + kBiasOff + warp * 256;
    for (int t = 0; t < n_tiles; ++t) {
      __syncwarp();                                             // the last tile's bias reads are done
      st_shared_f32(bias_row + 4 * lane, raw_valid<K>(a, raw1_lo) ? 0.0f : -INFINITY);
      st_shared_f32(bias_row + 128 + 4 * lane, raw_valid<K>(a, raw1_hi) ? 0.0f : -INFINITY);
      __syncwarp();
      const uint32_t sb = t & 1;
      if (!warp_wait_or_abort(s_full0 + 8 * sb, (t >> 1) & 1, s_abort)) break;
      fence_after_sync();
      float s[64];
      tmem_ld32(tmem + row_lane + kSCol + kTile * sb, s);
      tmem_ld32(tmem + row_lane + kSCol + kTile * sb + 32, s + 32);
      float mx[8];                                              // 8 independent running maxima
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const uint4 b = ld_shared16(bias_row + 4 * i);
        const float2 y0 = ffma2(make_float2(s[i], s[i + 1]), make_float2(a.scale_log2, a.scale_log2),
                                make_float2(__uint_as_float(b.x), __uint_as_float(b.y)));
        const float2 y1 = ffma2(make_float2(s[i + 2], s[i + 3]), make_float2(a.scale_log2, a.scale_log2),
                                make_float2(__uint_as_float(b.z), __uint_as_float(b.w)));
        s[i] = y0.x;
        s[i + 1] = y0.y;
        s[i + 2] = y1.x;
        s[i + 3] = y1.y;
        mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], y0.x, y0.y);
        mx[((i >> 1) + 1) & 7] = fmax3(mx[((i >> 1) + 1) & 7], y1.x, y1.y);
      }
      const float tmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
      // Lazy rescaling: the reference max moves only when the tile's max
      // exceeds it by more than 2^8 (weights stay below 256 otherwise).
      const bool grow = tmax > m + kRescaleLog2;
      const float alpha = grow ? ex2(m - tmax) : 1.0f;          // 0 while m is -inf
      if (grow) m = tmax;
      const float m_use = m == -INFINITY ? 0.0f : m;
      uint32_t pk[32];
      float2 ps[4];                                             // 4 independent running sums
#pragma unroll
      for (int i = 0; i < 4; ++i) ps[i] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 d = fadd2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(-m_use, -m_use));
        pk[i] = pack_bf16x2(ex2(d.x), ex2(d.y));
        add_bf16x2(ps[i & 3].x, ps[i & 3].y, pk[i]);
      }
      const float2 p01 = fadd2(ps[0], ps[1]), p23 = fadd2(ps[2], ps[3]);
      const float2 psum2 = fadd2(p01, p23);
      l = l * alpha + (psum2.x + psum2.y);
      // P V of the previous tile must be done before O is rescaled (the wait
      // also keeps the barrier's phases in step).
      if (t > 0 && !warp_wait_or_abort(o_done, (t - 1) & 1, s_abort)) break;
      if (t > 0 && __any_sync(0xffffffffu, grow)) {
        fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {          // the row's 256 O columns
          float o[32];
          const uint32_t col = kOCol + 32 * c;
          tmem_ld32(tmem + row_lane + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + row_lane + col, o);
        }
      }
      // P (64 values = 32 bf16 pairs) over the first half of tile t's S.
      tmem_st16(tmem + row_lane + kSCol + kTile * sb, pk);
      tmem_st16(tmem + row_lane + kSCol + kTile * sb + 16, pk + 16);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // the keys two tiles ahead, after the arrive (a release waits for
      // accesses in flight)
      raw1_lo = raw2_lo;
      raw1_hi = raw2_hi;
      raw2_lo = key_raw<K>(a, blk, (t + 2) * kTile + lane);
      raw2_hi = key_raw<K>(a, blk, (t + 2) * kTile + 32 + lane);
      if (t == n_tiles / 2) prefetch_next_wave<K>(a, warp * 32 + lane);
    }
  } else if (warp < kMmaWarp) {
    if constexpr (K == Keys::kWorkspace) {
      // ---- workspace keys: one thread has the copy engine land every tile --
      // (the nine 8 KB blocks of a tile as tensor-map loads of 64 rows x 64
      // dimensions, 128-byte swizzled: group A then group B, each completing
      // its stage's full barrier).  Rows of a tile past the context (or past
      // the workspace, zero-filled) are masked by the softmax.
      if (warp == kFirstProducerWarp && lane == 0) {
        int last_a[kAStages], last_b[kBStages];     // last tile issued into each stage
        for (int s2 = 0; s2 < kAStages; ++s2) last_a[s2] = -1;
        for (int s2 = 0; s2 < kBStages; ++s2) last_b[s2] = -1;
        for (int t = 0; t < n_tiles; ++t) {
          const int32_t row = static_cast<int32_t>(blk.ws_row0 + blk.key0 + static_cast<int64_t>(t) * kTile);
          const int sa = t % kAStages;
          if (t >= kAStages && !wait_or_abort(a_empty0 + 8 * sa, (t / kAStages - 1) & 1, s_abort)) break;
          const uint32_t astage = base + kAOff + sa * kAStage;
          mbar_arrive_expect_tx(a_full0 + 8 * sa, 5 * kKBlock);
#pragma unroll
          for (int j = 0; j < 4; ++j) tma_load_2d(astage + j * kKBlock, &kmap, other + 64 * j, row, a_full0 + 8 * sa);
          tma_load_2d(astage + 4 * kKBlock, &kmap, KVQ_MLA_NOPE_DIM, row, a_full0 + 8 * sa);
          last_a[sa] = t;
          const int sb = t % kBStages;
          if (t >= kBStages && !wait_or_abort(b_empty0 + 8 * sb, (t / kBStages - 1) & 1, s_abort)) break;
          const uint32_t bstage = base + kBOff + sb * kBStage;
          mbar_arrive_expect_tx(b_full0 + 8 * sb, 4 * kKBlock);
#pragma unroll
          for (int j = 0; j < 4; ++j) tma_load_2d(bstage + j * kKBlock, &kmap, own + 64 * j, row, b_full0 + 8 * sb);
          last_b[sb] = t;
        }
        // Before the CTA may leave, the copies of the last tile issued into
        // each stage have landed (normally long since consumed).
        for (int s2 = 0; s2 < kAStages + kBStages; ++s2) {
          const int t = s2 < kAStages ? last_a[s2] : last_b[s2 - kAStages];
          if (t < 0) continue;
          const uint32_t bar = s2 < kAStages ? a_full0 + 8 * s2 : b_full0 + 8 * (s2 - kAStages);
          const int stages = s2 < kAStages ? kAStages : kBStages;
          const long long start = clock64();
          while (!mbar_try_wait(bar, (t / stages) & 1)) {
            if (clock64() - start > kDrainCycles) { *s_abort = 1; break; }
          }
        }
      }
    } else {
      // ---- producers: group A, then group B, of every tile ----------------------
      // A group's loads for the next tile are issued right after this tile's
      // group is handed over (a release waits for every access of the thread in
      // flight, so loads go after an arrive), so that their latency hides
      // behind the other group's decode and the waits for free stages.
      for (int t = 0; t < n_tiles; ++t) {
        // group A: decoded into registers, then stored once stage t % kAStages
        // is free (the group-A K-steps of tile t - kAStages are done)
        uint4 va[10];
        decode_part<F, true>(ra, va);
        const int sa = t % kAStages;
        if (t >= kAStages && !warp_wait_or_abort(a_empty0 + 8 * sa, (t / kAStages - 1) & 1, s_abort)) break;
        const uint32_t astage = base + kAOff + sa * kAStage;
        write_part<true>(astage + k * kKBlock, astage + 4 * kKBlock, r, k, va);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full0 + 8 * sa);
        // the next tile's group-A loads now: they are consumed a whole group-B
        // decode and one wait later
        const uint8_t* next =
            t + 1 < n_tiles ? key_entry<K>(a, blk, raw_next, (t + 1) * kTile + r, bad_index) : nullptr;
        if (t + 1 < n_tiles) load_part<F, true>(next, a_nope0, k, ra);
        // group B: stage t % kBStages is free once P V of tile t - kBStages is done
        uint4 vb[8];
        decode_part<F, false>(rb, vb);
        const int sb = t % kBStages;
        if (t >= kBStages && !warp_wait_or_abort(b_empty0 + 8 * sb, (t / kBStages - 1) & 1, s_abort)) break;
        write_part<false>(base + kBOff + sb * kBStage + k * kKBlock, 0, r, k, vb);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_full0 + 8 * sb);
        if (t + 1 < n_tiles) load_part<F, false>(next, b_nope0, k, rb);
        cur = next;
        raw_next = raw_next2;
        raw_next2 = key_raw<K>(a, blk, (t + 3) * kTile + r);
        if constexpr (F == Entry::kFp8 && K == Keys::kSparse) {
          // Scattered 656-byte entries: the lines of the entry two tiles ahead
          // are asked into L2 now (the four lanes of a row take one line
          // each, then the rest), so that next tile's register loads of it
          // find them there.  The nvfp4 entries' loads, and a dense prefill's
          // consecutive entries of one block, are already covered; there the
          // prefetch only costs issue slots.
          if (t + 2 < n_tiles && raw_valid<K>(a, raw_next)) {
            bool unused = false;
            const uint8_t* p2 = key_entry<K>(a, blk, raw_next, (t + 2) * kTile + r, unused);
            constexpr int kBytes = KVQ_FP8_DS_MLA_ENTRY_BYTES;
#pragma unroll
            for (int o = 0; o < kBytes + 127; o += 512) {
              const int off = o + 128 * k;
              if (off < kBytes + 127) prefetch_l2_line(p2 + (off < kBytes ? off : kBytes - 1));
            }
          }
        }
      }
    }
  } else if (lane == 0) {
    // ---- MMA issue (one thread) -------------------------------------------
    constexpr uint32_t kIdescQK = idesc_bf16(kRows, kTile, false);
    constexpr uint32_t kIdescPV = idesc_bf16(kRows, kHalf, true);
    // descriptors built once; a K-step adds its byte offset / 16 to the
    // start-address field (addresses stay below 256 KB: no carry out)
    const uint64_t qdesc = sw128_desc(base + kQOff, 16, 1024);
    const uint64_t adesc = sw128_desc(base + kAOff, 16, 1024);
    const uint64_t bdesc = sw128_desc(base + kBOff, 16, 1024);
    auto scores = [&](int u) -> bool {
      // S(u) = Q K(u)^T: 20 group-A K-steps (A from shared memory), then 16
      // group-B K-steps (A = the own query dimensions in TMEM)
      const int sa = u % kAStages;
      if (!wait_or_abort(a_full0 + 8 * sa, (u / kAStages) & 1, s_abort)) return false;
      fence_after_sync();
      const uint32_t d = tmem + kSCol + kTile * (u & 1);
#pragma unroll
      for (int j = 0; j < 5; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(d, qdesc + ((j * kQBlock + 32 * k) >> 4),
                   adesc + ((sa * kAStage + j * kKBlock + 32 * k) >> 4), kIdescQK, (j | k) != 0);
      mma_commit(a_empty0 + 8 * sa);
      mma_issued = 1;
      const int st = u % kBStages;
      if (!wait_or_abort(b_full0 + 8 * st, (u / kBStages) & 1, s_abort)) return false;
      fence_after_sync();
#pragma unroll
      for (int k = 0; k < 16; ++k)
        mma_bf16_ta(d, tmem + kQCol + 8 * k, bdesc + ((st * kBStage + (k >> 2) * kKBlock + 32 * (k & 3)) >> 4),
                    kIdescQK, 1u);
      mma_commit(s_full0 + 8 * (u & 1));
      return true;
    };
    if (n_tiles > 0 && (!a.q_tma || wait_or_abort(q_full, 0, s_abort)) && scores(0)) {
      for (int t = 0; t < n_tiles; ++t) {
#ifdef KVQ_ATTN_STALL_TILE
        // Failure-detection build only: from this tile on no MMA is issued, as
        // if the tensor work never completed; the thread idles until another
        // role's bounded wait runs out, and every role then takes the abort path.
        if (t == KVQ_ATTN_STALL_TILE) {
          wait_or_abort(drain, 0, s_abort);
          break;
        }
#endif
        if (t + 1 < n_tiles && !scores(t + 1)) break;
        // O += P(t) V(t): 4 MMAs of K = 16 keys, N = 256 value columns
        if (!wait_or_abort(p_full, t & 1, s_abort)) break;
        fence_after_sync();
        const int st = t % kBStages;
        const uint64_t vdesc = sw128_desc(base + kBOff + st * kBStage, kKBlock, 1024);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_bf16_ta(tmem + kOCol, tmem + kSCol + kTile * (t & 1) + 8 * k, vdesc + 128 * k, kIdescPV,
                      (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(b_empty0 + 8 * st);
        mma_commit(o_done);
      }
    }
  }

  // Every role has left its loop.  Drain every MMA still in flight: one more
  // commit tracks all of them.
  fence_before_sync();
  const bool any_mma = __syncthreads_or(mma_issued) != 0;
  fence_after_sync();
  bool aborted = *s_abort != 0;
  if (any_mma) {
    if (threadIdx.x == kMmaWarp * 32) mma_commit(drain);
    const long long start = clock64();
    while (!mbar_try_wait(drain, 0)) {            // bounded, ignores the abort flag
      if (clock64() - start > kDrainCycles) { aborted = true; break; }
    }
  }
  if (a.q_tma) {
    // the query tiles have landed before the CTA may leave (normally long ago)
    const long long start = clock64();
    while (!mbar_try_wait(q_full, 0)) {
      if (clock64() - start > kDrainCycles) { aborted = true; break; }
    }
  }
  fence_after_sync();
  if (bad_index && a.status) atomicOr(a.status, KVQ_STATUS_BAD_INDEX);
  aborted = __syncthreads_or(aborted) != 0;
  if (aborted && threadIdx.x == 0 && a.status) atomicOr(a.status, KVQ_STATUS_TIMEOUT);

  if (is_softmax && !aborted) {
    const uint32_t row_lane = warp * 32u << 16;
    const uint32_t row = warp * 32 + lane;
    const float l_row = l;
    const float inv_l = l_row > 0.0f ? 1.0f / l_row : 0.0f;
    int64_t token = 0;
    int32_t head = 0;
    const bool live = row < static_cast<uint32_t>(blk.rows);
    if (live) row_of<K>(a, blk, row, token, head);
    if (a.part_o != nullptr) {
      // A key range of a split decode: the normalised fp32 partial row (1 KB,
      // staged 1040 bytes apart) and the range's base-2 log-sum-exp, for the
      // combine launch.
      const uint32_t part_row = base + kStagingOff + row * kPartRowBytes;
#pragma unroll 1
      for (int c = 0; c < kHalf; c += 64) {
        uint32_t o[64];
        if (n_tiles > 0) {
          tmem_ld64(tmem + row_lane + kOCol + c, o);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = 0;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          st_shared16(part_row + 4 * c + 16 * i,
                      make_uint4(__float_as_uint(__uint_as_float(o[4 * i]) * inv_l),
                                 __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv_l),
                                 __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv_l),
                                 __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv_l)));
      }
      fence_async_smem();
      const int64_t prow = (token * a.num_heads + head) * a.num_splits + blk.split;
      if (live) {
        bulk_store(a.part_o + prow * KVQ_MLA_NOPE_DIM + own, part_row, kHalf * 4);
        bulk_wait_read();
        // both CTAs of the pair compute the same m and l; each records them,
        // so that a range one of them did not write is seen by the combine
        a.part_lse[prow * 2 + half] = l_row > 0.0f ? m + log2f(l_row) : -INFINITY;
      }
    } else {
      // Each thread scales its row's 256 O columns into bf16 and writes them
      // as one 512-byte row of a staging area in the (now idle) key stages
      // (rows 528 bytes apart, so that a warp's 16-byte stores spread over all
      // banks), then hands the row to the copy engine as one bulk copy to its
      // output row.
      const uint32_t stage_row = base + kStagingOff + row * kStageRowBytes;
#pragma unroll 1
      for (int c = 0; c < kHalf; c += 64) {
        uint32_t o[64];
        if (n_tiles > 0) {
          tmem_ld64(tmem + row_lane + kOCol + c, o);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = make_uint4(
              pack_bf16x2(__uint_as_float(o[8 * i]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l));
          st_shared16(stage_row + 2 * c + 16 * i, v);
        }
      }
      fence_async_smem();                 // the staged row -> visible to the copy engine
      if (live) {
        bulk_store(static_cast<__nv_bfloat16*>(a.out) + token * a.out_stride_t +
                       static_cast<int64_t>(head) * a.out_stride_h + own,
                   stage_row, kHalf * 2);
        bulk_wait_read();                 // the staging area is read before the CTA leaves
      }
      if (half == 0 && a.lse != nullptr && live)
        a.lse[token * a.lse_stride_t + head] =
            l_row > 0.0f ? (m + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// split decode: the key ranges' partial results combined
// ---------------------------------------------------------------------------
//
// One warp per (token, head) row; lane s holds range s's base-2 log-sum-exp
// L_s (at most 32 ranges; both CTAs of a range record it).  With M = max L_s
// and w_s = 2^(L_s - M):
//   out = sum_s w_s o_s / sum_s w_s,   lse = (M + log2 sum_s w_s) ln 2,
// o_s being range s's normalised partial output (an empty range: L_s = -inf,
// weight 0; no valid key at all: out = 0, lse = -inf, as unsplit).  Every L_s
// is set to NaN before the partial launch: a row with a range that no CTA
// wrote (a query token of no request, a skipped request, a CTA that timed
// out) keeps its outputs untouched, as unsplit.
constexpr int kCombineWarps = 8;

__global__ void fill_nan_kernel(float* p, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[i] = __int_as_float(0x7fc00000);
}

__global__ void __launch_bounds__(kCombineWarps * 32) combine_splits_kernel(const AttentionArgs a) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.num_tokens * a.num_heads) return;          // whole warps
  const int splits = a.num_splits;
  const float ls = lane < splits ? a.part_lse[(row * splits + lane) * 2] : -INFINITY;
  const float ls1 = lane < splits ? a.part_lse[(row * splits + lane) * 2 + 1] : -INFINITY;
  if (__any_sync(0xffffffffu, ls != ls || ls1 != ls1)) return;   // a range half not written
  float mx = ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float w = ls == -INFINITY ? 0.0f : ex2(ls - mx);
  float den = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  const float* po = a.part_o + row * splits * KVQ_MLA_NOPE_DIM + 16 * lane;
  for (int sp = 0; sp < splits; ++sp) {
    const float ws = __shfl_sync(0xffffffffu, w, sp);
    if (ws == 0.0f) continue;                               // uniform over the warp
    const float4* src = reinterpret_cast<const float4*>(po + sp * KVQ_MLA_NOPE_DIM);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(src + i);
      acc[4 * i] += ws * v.x;
      acc[4 * i + 1] += ws * v.y;
      acc[4 * i + 2] += ws * v.z;
      acc[4 * i + 3] += ws * v.w;
    }
  }
  const float inv = den > 0.0f ? 1.0f / den : 0.0f;
  const int64_t token = row / a.num_heads;
  const int64_t head = row - token * a.num_heads;
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + token * a.out_stride_t +
                                        head * a.out_stride_h + 16 * lane);
#pragma unroll
  for (int h = 0; h < 2; ++h)
    dst[h] = make_uint4(pack_bf16x2(acc[8 * h] * inv, acc[8 * h + 1] * inv),
                        pack_bf16x2(acc[8 * h + 2] * inv, acc[8 * h + 3] * inv),
                        pack_bf16x2(acc[8 * h + 4] * inv, acc[8 * h + 5] * inv),
                        pack_bf16x2(acc[8 * h + 6] * inv, acc[8 * h + 7] * inv));
  if (lane == 0 && a.lse != nullptr)
    a.lse[token * a.lse_stride_t + head] = den > 0.0f ? (mx + log2f(den)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace

// The driver's tensor-map encoder, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult found{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &found) !=
            cudaSuccess ||
        found != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map of the query rows, tiles of 64 dimensions x 128 rows with the
// 128-byte swizzle: sparse form [tokens][heads][576] (a tile is 128 heads of
// one token, heads past num_heads zero-filled); dense form [token x head
// rows][576], which needs the tokens' rows packed (q_stride_t = num_heads x
// q_stride_h).  false: no map (the kernel copies the rows itself).
template <Keys K>
bool query_tensor_map(const AttentionArgs& a, CUtensorMap* map) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr || a.num_tokens < 1) return false;
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r;
  if constexpr (K == Keys::kSparse) {
    const cuuint64_t dims[3] = {KVQ_WORKSPACE_DIM, static_cast<cuuint64_t>(a.num_heads),
                                static_cast<cuuint64_t>(a.num_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.q_stride_h) * 2, static_cast<cuuint64_t>(a.q_stride_t) * 2};
    const cuuint32_t box[3] = {64, kRows, 1};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const int64_t rows = a.num_tokens * a.num_heads;
    if (a.q_stride_t != a.num_heads * a.q_stride_h || rows >= (int64_t{1} << 31)) return false;
    const cuuint64_t dims[2] = {KVQ_WORKSPACE_DIM, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.q_stride_h) * 2};
    const cuuint32_t box[2] = {64, kRows};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

// Tensor map of a gathered bf16 workspace [ws_rows, 576] (row stride
// ws_stride elements): tiles of 64 dimensions x 64 rows, 128-byte swizzled,
// the layout of one key block of a stage; rows past ws_rows read as zeros
// (with no rows at all, one row of q stands in: no tile is then loaded).
bool workspace_tensor_map(const AttentionArgs& a, CUtensorMap* map) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {KVQ_WORKSPACE_DIM, static_cast<cuuint64_t>(a.ws_rows > 0 ? a.ws_rows : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.ws_stride) * 2};
  const cuuint32_t box[2] = {64, kTile};
  const cuuint32_t elem_strides[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.ws), dims, strides, box, elem_strides,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <Entry F, Keys K>
cudaError_t launch_attention(const AttentionArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(mla_attention_kernel<F, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  int device = 0, sms = 0;
  if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) return e;
  AttentionArgs args = a;
  args.wave = sms;                      // one CTA per SM
  CUtensorMap qmap, kmap;
  std::memset(&qmap, 0, sizeof(qmap));
  std::memset(&kmap, 0, sizeof(kmap));
  args.q_tma = query_tensor_map<K>(a, &qmap) ? 1 : 0;
  if (K == Keys::kWorkspace && !workspace_tensor_map(a, &kmap)) return cudaErrorInvalidValue;
  dim3 grid;
  if constexpr (K == Keys::kSparse) {
    grid = dim3(static_cast<unsigned>(a.num_tokens * 2 * (a.num_splits > 1 ? a.num_splits : 1)));
  } else {
    const int64_t blocks = (static_cast<int64_t>(a.max_query_len) * a.num_heads + kRows - 1) / kRows;
    grid = dim3(static_cast<unsigned>(blocks * 2 * (a.num_splits > 1 ? a.num_splits : 1)),
                static_cast<unsigned>(a.batch_size));
  }
  mla_attention_kernel<F, K><<<grid, kThreads, kSmemBytes, stream>>>(args, qmap, kmap);
  return cudaGetLastError();
}

cudaError_t launch_sparse_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kNvfp4, Keys::kSparse>(a, stream);
}
cudaError_t launch_sparse_mla_attention_fp8(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kFp8, Keys::kSparse>(a, stream);
}
template <Entry F, Keys K>
cudaError_t launch_split(const AttentionArgs& a, cudaStream_t stream) {
  const int64_t rows = a.num_tokens * a.num_heads;
  const int64_t n = rows * a.num_splits * 2;
  fill_nan_kernel<<<static_cast<unsigned>(min(int64_t{1024}, (n + 255) / 256)), 256, 0, stream>>>(a.part_lse, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_attention<F, K>(a, stream);
  if (e != cudaSuccess) return e;
  combine_splits_kernel<<<static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps), kCombineWarps * 32, 0,
                          stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sparse_mla_attention_split_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  return launch_split<Entry::kNvfp4, Keys::kSparse>(a, stream);
}
cudaError_t launch_sparse_mla_attention_split_fp8(const AttentionArgs& a, cudaStream_t stream) {
  return launch_split<Entry::kFp8, Keys::kSparse>(a, stream);
}
cudaError_t launch_prefill_mla_attention_split_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  return launch_split<Entry::kNvfp4, Keys::kDense>(a, stream);
}
cudaError_t launch_prefill_mla_attention_split_fp8(const AttentionArgs& a, cudaStream_t stream) {
  return launch_split<Entry::kFp8, Keys::kDense>(a, stream);
}
cudaError_t launch_prefill_mla_attention_workspace(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kNvfp4, Keys::kWorkspace>(a, stream);   // keys are bf16: no entry format
}
cudaError_t launch_prefill_mla_attention_nvfp4(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kNvfp4, Keys::kDense>(a, stream);
}
cudaError_t launch_prefill_mla_attention_fp8(const AttentionArgs& a, cudaStream_t stream) {
  return launch_attention<Entry::kFp8, Keys::kDense>(a, stream);
}

}  // namespace kvq
