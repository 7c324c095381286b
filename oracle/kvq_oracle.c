/*
 * kvq_oracle.c -- CPU oracle for the quantized paged KV-cache write and
 * gather-upconvert path.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg, never by the product path.  It shares
 * no code with the CUDA library.  Build: gcc -O2 -std=c11 -ffp-contract=off
 * (no fused multiply-add, no fast math), so every float expression below is
 * one IEEE-754 binary32 operation rounded to nearest-even.
 *
 * Sources are cited by page title and section; see kvq_oracle.h for the list
 * ([P1] [P2] [P3] [OFP8] [MX]).
 *
 * Parity unpinned against the pages: the per-head NVFP4 region order inside a
 * page, the 656-byte fp8_ds_mla entry order and the sparse-decode index
 * formula (fixed by the format spec only).  Every other step is pinned by the
 * oracle's own tests.
 */
#include "kvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ========================================================================== */
/* Number formats                                                             */
/* ========================================================================== */

/* [OFP8] E4M3: sign bit 7, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 holds subnormals m * 2^-6 / 8; S.1111.111 is NaN; there
 * is no infinity.  Largest finite magnitude: 1.75 * 2^8 = 448. */
double kvqo_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* [MX] FP4 E2M1: sign bit 3, 2 exponent bits (bias 1), 1 mantissa bit;
 * exponent field 0 holds the subnormal 0.5 * m; no NaN, no infinity.
 * Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double kvqo_e2m1_value(uint8_t nibble) {
    int sign = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int m = nibble & 0x1;
    double mag;
    if (e == 0)
        mag = ldexp((double)m / 2.0, 1 - 1);
    else
        mag = ldexp(1.0 + (double)m / 2.0, e - 1);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32 bit pattern. */
float kvqo_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest, ties to the even code, onto a sorted table of the
 * non-negative magnitudes of codes 0..n_codes-1 (magnitude increases with the
 * code), saturating at the last code.  Works on exact doubles: every
 * comparison below is exact, because the midpoint of two adjacent table
 * values needs one more bit than they do and binary32 inputs convert to
 * double exactly. */
static int nearest_code(double a, const double* mag, int n_codes) {
    int lo = 0, hi = n_codes - 1;
    if (a >= mag[hi]) return hi;             /* satfinite                  */
    /* bisection for the last code whose magnitude is <= a */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (mag[mid] <= a) lo = mid; else hi = mid;
    }
    /* now mag[lo] <= a < mag[hi], hi == lo + 1 */
    if (a == mag[lo]) return lo;
    {
        double midpoint = (mag[lo] + mag[hi]) / 2.0;
        if (a < midpoint) return lo;
        if (a > midpoint) return hi;
        return (lo % 2 == 0) ? lo : hi;      /* tie: the even code         */
    }
}

static double e4m3_mag[127];  /* codes 0x00..0x7E */
static double e2m1_mag[8];    /* codes 0x0..0x7   */

/* Filled once when the library is loaded, before any thread calls in. */
__attribute__((constructor)) static void build_tables(void) {
    int c;
    for (c = 0; c < 127; ++c) e4m3_mag[c] = kvqo_e4m3_value((uint8_t)c);
    for (c = 0; c < 8; ++c) e2m1_mag[c] = kvqo_e2m1_value((uint8_t)c);
}

/* e4m3 encoding with cvt.rn.satfinite semantics (the conversion the
 * [P1] "Key source snippets" kernel names): round to nearest even, finite
 * values beyond 448 and infinities clamp to +-448, NaN stays NaN (0x7F with
 * the input's sign), the sign of zero is kept. */
uint8_t kvqo_e4m3_rn_sat(float f) {
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    if (isnan(f)) return (uint8_t)(sign | 0x7F);
    return (uint8_t)(sign | nearest_code(fabs((double)f), e4m3_mag, 127));
}

/* e2m1 encoding with cvt.rn.satfinite.e2m1x2.f32 semantics ([P1] "Key source
 * snippets"): nearest of +-{0,0.5,1,1.5,2,3,4,6}, ties to the even code,
 * |f| > 6 clamps to 6; a negative input that rounds to zero gives code 0x8.
 * NaN inputs are outside the contract (this returns +-6). */
uint8_t kvqo_e2m1_rn_sat(float f) {
    uint8_t sign = signbit(f) ? 0x8 : 0x0;
    if (isnan(f)) return (uint8_t)(sign | 0x7);
    return (uint8_t)(sign | nearest_code(fabs((double)f), e2m1_mag, 8));
}

/* binary32 -> bfloat16, round to nearest even: the two bfloat16 neighbours of
 * f are its truncation toward zero and the next value away from zero; pick the
 * nearer, the one with an even last bit on a tie. */
uint16_t kvqo_bf16_rn(float f) {
    uint32_t u, t_bits, n_bits;
    float t, n;
    double a, dt, dn;
    if (isnan(f)) {
        memcpy(&u, &f, sizeof u);
        return (uint16_t)((u >> 16) | 0x0040);   /* quiet NaN, outside contract */
    }
    memcpy(&u, &f, sizeof u);
    t_bits = u & 0xFFFF0000u;            /* truncation toward zero            */
    n_bits = t_bits + 0x00010000u;       /* next magnitude up (may be inf)    */
    if ((u & 0xFFFFu) == 0) return (uint16_t)(u >> 16);
    memcpy(&t, &t_bits, sizeof t);
    memcpy(&n, &n_bits, sizeof n);
    a = fabs((double)f);
    dt = a - fabs((double)t);
    if (isinf(n)) {
        /* the step above the largest finite bfloat16 is 2^128; use it */
        dn = ldexp(1.0, 128) - a;
    } else {
        dn = fabs((double)n) - a;
    }
    if (dt < dn) return (uint16_t)(t_bits >> 16);
    if (dn < dt) return (uint16_t)(n_bits >> 16);
    return ((t_bits >> 16) & 1) ? (uint16_t)(n_bits >> 16) : (uint16_t)(t_bits >> 16);
}

static float bits_to_float(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void kvqo_encode_bits_range(uint32_t first_bits, int64_t count,
                            uint8_t* e4m3_out, uint8_t* e2m1_out) {
    int64_t i;
    for (i = 0; i < count; ++i) {
        float f = bits_to_float(first_bits + (uint32_t)i);
        if (e4m3_out) e4m3_out[i] = kvqo_e4m3_rn_sat(f);
        if (e2m1_out) e2m1_out[i] = kvqo_e2m1_rn_sat(f);
    }
}

void kvqo_bf16_rn_bits_range(uint32_t first_bits, int64_t count, uint16_t* out) {
    int64_t i;
    for (i = 0; i < count; ++i) out[i] = kvqo_bf16_rn(bits_to_float(first_bits + (uint32_t)i));
}

void kvqo_e4m3_rn_sat_array(const float* in, int64_t n, uint8_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = kvqo_e4m3_rn_sat(in[i]);
}

void kvqo_e2m1_rn_sat_array(const float* in, int64_t n, uint8_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = kvqo_e2m1_rn_sat(in[i]);
}

void kvqo_bf16_rn_array(const float* in, int64_t n, uint16_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = kvqo_bf16_rn(in[i]);
}

/* ========================================================================== */
/* Format constants                                                           */
/* ========================================================================== */

/* [P1] "Implementation breakdown" item 3: 256 B e2m1 NoPE + 64 B e4m3 RoPE +
 * 32 B e4m3 NoPE scale factors; item 2: 352 bytes per token. */
#define NV_NOPE_DIM      512
#define NV_ROPE_DIM      64
#define NV_GROUP         16
#define NV_NOPE_BYTES    (NV_NOPE_DIM / 2)                 /* 256 */
#define NV_ROPE_OFF      NV_NOPE_BYTES                     /* 256 */
#define NV_SF_OFF        (NV_ROPE_OFF + NV_ROPE_DIM)       /* 320 */
#define NV_ENTRY         (NV_SF_OFF + NV_NOPE_DIM / NV_GROUP) /* 352 */

/* [P1] "Implementation breakdown" item 2: 656 bytes per token for
 * fp8_ds_mla.  Composition and order are the format spec's reading: 512 e4m3
 * NoPE, then 4 little-endian fp32 scales (one per 128 NoPE values), then 64
 * bf16 RoPE. */
#define F8_TILE          128
#define F8_SCALE_OFF     NV_NOPE_DIM                       /* 512 */
#define F8_ROPE_OFF      (F8_SCALE_OFF + 4 * (NV_NOPE_DIM / F8_TILE)) /* 528 */
#define F8_ENTRY         (F8_ROPE_OFF + 2 * NV_ROPE_DIM)   /* 656 */

int32_t kvqo_nvfp4_ds_mla_entry_bytes(void) { return NV_ENTRY; }
int32_t kvqo_fp8_ds_mla_entry_bytes(void) { return F8_ENTRY; }

/* [P2] "Key source snippets" (flashinfer.py get_kv_cache_shape):
 * full_dim = head_size // 2 + head_size // 16. */
int32_t kvqo_nvfp4_full_dim(int32_t head_size) { return head_size / 2 + head_size / 16; }

/* [P2] "Key source snippets" (torch_utils.py nvfp4_kv_cache_split_views):
 * data_dim = full_dim * 8 // 9, scale_dim = full_dim - data_dim. */
int32_t kvqo_nvfp4_data_dim(int32_t full_dim) { return full_dim * 8 / 9; }
int32_t kvqo_nvfp4_scale_dim(int32_t full_dim) { return full_dim - kvqo_nvfp4_data_dim(full_dim); }

/* ========================================================================== */
/* Shared arithmetic steps of the NVFP4 recipe                                */
/* ========================================================================== */

/* One 16-value NVFP4 group ([P1] "Key source snippets", write kernel warp 0,
 * and the test's _ref_nvfp4_sf_bytes(x, 6.0)): amax over |x| in fp32,
 * sf = e4m3_rn_sat(amax / 6), inverse scale 1/sf (0 when sf is zero), codes
 * e2m1_rn_sat(x * inv).  Value 2k of the group goes to the low nibble of byte
 * k, value 2k+1 to the high nibble. */
static uint8_t nvfp4_group(const float* x, uint8_t* packed8) {
    float amax = 0.0f, sf_value, inv;
    uint8_t sf;
    int i;
    for (i = 0; i < NV_GROUP; ++i) amax = fmaxf(amax, fabsf(x[i]));
    sf = kvqo_e4m3_rn_sat(amax / 6.0f);
    sf_value = (float)kvqo_e4m3_value(sf);
    inv = (sf_value == 0.0f) ? 0.0f : 1.0f / sf_value;
    for (i = 0; i < NV_GROUP / 2; ++i) {
        uint8_t lo = kvqo_e2m1_rn_sat(x[2 * i] * inv);
        uint8_t hi = kvqo_e2m1_rn_sat(x[2 * i + 1] * inv);
        packed8[i] = (uint8_t)(lo | (hi << 4));
    }
    return sf;
}

/* Slot -> (block, offset) as in the [P1] write kernel: block = slot /
 * block_size, offset = slot % block_size. */
static uint8_t* slot_entry(uint8_t* cache, int64_t slot, int32_t block_size,
                           int64_t block_stride, int64_t entry_stride) {
    return cache + (slot / block_size) * block_stride + (slot % block_size) * entry_stride;
}

/* ========================================================================== */
/* Write: concat_and_cache_nvfp4_ds_mla                                       */
/* ========================================================================== */

/* [P1] "Key source snippets", concat_and_cache_nvfp4_ds_mla_kernel: for each
 * token, slot = slot_mapping[t]; a negative slot is a padding token and is
 * skipped; otherwise the 352-byte entry at (slot / block_size, slot %
 * block_size) receives the 512 NoPE values as 32 NVFP4 groups (bytes
 * 8g..8g+7 for group g), the 64 RoPE values as unscaled e4m3 (bytes
 * 256..319) and the 32 group scales (bytes 320..351, scale g at 320 + g: the
 * identity element order of the format spec). */
int64_t kvqo_write_nvfp4_ds_mla(
    const uint16_t* kv_c, int64_t kv_c_stride,
    const uint16_t* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride) {
    int64_t t, skipped = 0;
    for (t = t_begin; t < t_end; ++t) {
        int64_t slot = slot_mapping[t];
        uint8_t* entry;
        float x[NV_NOPE_DIM];
        int g, j;
        if (slot < 0) continue;                               /* padding   */
        if (slot >= num_blocks * (int64_t)block_size) { ++skipped; continue; }
        entry = slot_entry(cache, slot, block_size, block_stride, entry_stride);
        for (j = 0; j < NV_NOPE_DIM; ++j) x[j] = kvqo_bf16_value(kv_c[t * kv_c_stride + j]);
        for (g = 0; g < NV_NOPE_DIM / NV_GROUP; ++g)
            entry[NV_SF_OFF + g] = nvfp4_group(&x[g * NV_GROUP], &entry[g * (NV_GROUP / 2)]);
        for (j = 0; j < NV_ROPE_DIM; ++j)
            entry[NV_ROPE_OFF + j] = kvqo_e4m3_rn_sat(kvqo_bf16_value(k_pe[t * k_pe_stride + j]));
    }
    return skipped;
}

/* ========================================================================== */
/* Write: 656-byte fp8_ds_mla entry (format-spec filler)                      */
/* ========================================================================== */

/* [P1] "Implementation breakdown" item 2 (656 bytes per token) and [P3]
 * "Function and motivation" (packed 656-byte FP8 cache).  The recipe is the
 * format spec's: per 128-value tile j, s_j = amax_j / 448 (1 when amax_j is
 * zero), NoPE byte k = e4m3_rn_sat(x_k / s_j), scales stored as fp32, RoPE
 * stored as its bf16 bits. */
int64_t kvqo_write_fp8_ds_mla(
    const uint16_t* kv_c, int64_t kv_c_stride,
    const uint16_t* k_pe, int64_t k_pe_stride,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride) {
    int64_t t, skipped = 0;
    for (t = t_begin; t < t_end; ++t) {
        int64_t slot = slot_mapping[t];
        uint8_t* entry;
        int j, k;
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) { ++skipped; continue; }
        entry = slot_entry(cache, slot, block_size, block_stride, entry_stride);
        for (j = 0; j < NV_NOPE_DIM / F8_TILE; ++j) {
            float amax = 0.0f, s;
            for (k = 0; k < F8_TILE; ++k)
                amax = fmaxf(amax, fabsf(kvqo_bf16_value(kv_c[t * kv_c_stride + j * F8_TILE + k])));
            s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
            for (k = 0; k < F8_TILE; ++k) {
                float x = kvqo_bf16_value(kv_c[t * kv_c_stride + j * F8_TILE + k]);
                entry[j * F8_TILE + k] = kvqo_e4m3_rn_sat(x / s);
            }
            memcpy(&entry[F8_SCALE_OFF + 4 * j], &s, 4);   /* little-endian host */
        }
        for (j = 0; j < NV_ROPE_DIM; ++j) {
            uint16_t r = k_pe[t * k_pe_stride + j];
            entry[F8_ROPE_OFF + 2 * j] = (uint8_t)(r & 0xFF);
            entry[F8_ROPE_OFF + 2 * j + 1] = (uint8_t)(r >> 8);
        }
    }
    return skipped;
}

/* ========================================================================== */
/* Gather index walk                                                          */
/* ========================================================================== */

/* [P1] "Key source snippets", cp_gather_and_upconvert_nvfp4_kv_cache_kernel,
 * and [P3] "Implementation breakdown" item 2 / "Key source snippets"
 * (cp_gather_and_upconvert_fp8_kv_cache with workspace_starts = cu_seq_lens
 * and seq_starts, seq_lens removed): workspace row w belongs to the request b
 * with the largest workspace_starts[b] <= w; it is position
 * seq_starts[b] + (w - workspace_starts[b]) of that request, found through
 * block_table[b][position / block_size] at offset position % block_size.
 * Returns the entry, or NULL when some index is out of range. */
static const uint8_t* gather_source(
    int64_t w, const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts, int32_t batch_size) {
    int32_t b, found = -1;
    int64_t position, column, block;
    for (b = 0; b < batch_size; ++b)
        if ((int64_t)workspace_starts[b] <= w) found = b;
    if (found < 0) return NULL;
    position = (int64_t)seq_starts[found] + (w - (int64_t)workspace_starts[found]);
    if (position < 0) return NULL;
    column = position / block_size;
    if (column >= block_table_width) return NULL;
    block = block_table[(int64_t)found * block_table_stride + column];
    if (block < 0 || block >= num_blocks) return NULL;
    return cache + block * block_stride + (position % block_size) * entry_stride;
}

/* ========================================================================== */
/* Gather-upconvert: nvfp4_ds_mla -> bf16 [T, 576]                            */
/* ========================================================================== */

/* [P1] "Key source snippets": unpack the e2m1 NoPE and apply the scale
 * factors to get bf16, convert the e4m3 RoPE straight to bf16, write the
 * contiguous bf16 [total_tokens, 576] workspace (NoPE 0..511, RoPE 512..575).
 * Each product e2m1 * e4m3 is exact in bf16. */
void kvqo_decode_nvfp4_ds_mla_entry(const uint8_t* entry, double* out576) {
    int k;
    for (k = 0; k < NV_NOPE_DIM; ++k) {
        uint8_t byte = entry[k / 2];
        uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        out576[k] = kvqo_e2m1_value(nib) * kvqo_e4m3_value(entry[NV_SF_OFF + k / NV_GROUP]);
    }
    for (k = 0; k < NV_ROPE_DIM; ++k)
        out576[NV_NOPE_DIM + k] = kvqo_e4m3_value(entry[NV_ROPE_OFF + k]);
}

int64_t kvqo_gather_nvfp4_ds_mla(
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    uint16_t* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts,
    int32_t batch_size, const int64_t* rows, int64_t n_rows) {
    int64_t i, skipped = 0;
    for (i = 0; i < n_rows; ++i) {
        int64_t w = rows ? rows[i] : i;
        const uint8_t* entry;
        double v[NV_NOPE_DIM + NV_ROPE_DIM];
        int k;
        if (w < 0 || w >= num_out_tokens) { ++skipped; continue; }
        entry = gather_source(w, cache, num_blocks, block_size, block_stride, entry_stride,
                              block_table, block_table_stride, block_table_width,
                              workspace_starts, seq_starts, batch_size);
        if (!entry) { ++skipped; continue; }
        kvqo_decode_nvfp4_ds_mla_entry(entry, v);
        for (k = 0; k < NV_NOPE_DIM + NV_ROPE_DIM; ++k)
            dst[i * dst_stride + k] = kvqo_bf16_rn((float)v[k]);   /* exact */
    }
    return skipped;
}

/* ========================================================================== */
/* Gather-upconvert: fp8_ds_mla -> bf16 [T, 576]                              */
/* ========================================================================== */

/* [P3] "Implementation breakdown" items 2 and 4: gather the packed 656-byte
 * FP8 entries into a bf16 workspace.  NoPE value k = bf16_rn(e4m3(n_k) *
 * s_{k/128}) with the product rounded once in fp32; RoPE bf16 bits copied. */
int64_t kvqo_gather_fp8_ds_mla(
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride,
    uint16_t* dst, int64_t dst_stride, int64_t num_out_tokens,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width,
    const int32_t* workspace_starts, const int32_t* seq_starts,
    int32_t batch_size, const int64_t* rows, int64_t n_rows) {
    int64_t i, skipped = 0;
    for (i = 0; i < n_rows; ++i) {
        int64_t w = rows ? rows[i] : i;
        const uint8_t* entry;
        int k;
        if (w < 0 || w >= num_out_tokens) { ++skipped; continue; }
        entry = gather_source(w, cache, num_blocks, block_size, block_stride, entry_stride,
                              block_table, block_table_stride, block_table_width,
                              workspace_starts, seq_starts, batch_size);
        if (!entry) { ++skipped; continue; }
        for (k = 0; k < NV_NOPE_DIM; ++k) {
            float s, product;
            memcpy(&s, &entry[F8_SCALE_OFF + 4 * (k / F8_TILE)], 4);
            product = (float)kvqo_e4m3_value(entry[k]) * s;
            dst[i * dst_stride + k] = kvqo_bf16_rn(product);
        }
        for (k = 0; k < NV_ROPE_DIM; ++k)
            dst[i * dst_stride + NV_NOPE_DIM + k] =
                (uint16_t)(entry[F8_ROPE_OFF + 2 * k] | (entry[F8_ROPE_OFF + 2 * k + 1] << 8));
    }
    return skipped;
}

/* ========================================================================== */
/* Per-head NVFP4 K/V cache: reshape_and_cache                                */
/* ========================================================================== */

/* Byte offsets inside the per-head cache.  [P2] "Key source snippets"
 * (flashinfer.py): shape (num_pages, 2, block_size, num_kv_heads, full_dim);
 * [P2] "Function and motivation" / "Implementation breakdown" item 4: layout
 * [K_data | K_scale | V_data | V_scale], each contiguous.  Format-spec
 * reading: inside page p and side s (K = 0, V = 1) the block_size * H *
 * full_dim bytes hold first the data (one data_dim row per (offset, head)),
 * then the scales (one scale_dim row each), rows in the cache's layout order,
 * with data_dim and scale_dim from the split-view formula. */
static int64_t perhead_side_base(int64_t page, int side, int32_t block_size,
                                 int32_t num_heads, int32_t head_size) {
    int64_t region = (int64_t)block_size * num_heads * kvqo_nvfp4_full_dim(head_size);
    return page * 2 * region + side * region;
}

/* Row of (offset, head) inside a side region: NHD keeps a token's heads
 * together (row = offset * H + h, the shape's (block_size, num_kv_heads)
 * order); HND keeps a head's tokens together (row = h * block_size + offset).
 * [P2] "Key source snippets" (torch_utils.py _nvfp4_split_data_scale): the
 * split views keep the cache's own layout, NHD or HND. */
static int64_t perhead_row(int32_t off, int32_t h, int32_t block_size, int32_t num_heads, int32_t layout) {
    return layout == 1 ? (int64_t)h * block_size + off : (int64_t)off * num_heads + h;
}

static int64_t perhead_data_off(int64_t row, int32_t head_size) {
    int32_t data_dim = kvqo_nvfp4_data_dim(kvqo_nvfp4_full_dim(head_size));
    return row * data_dim;
}

static int64_t perhead_scale_off(int64_t row, int32_t block_size, int32_t num_heads, int32_t head_size) {
    int32_t full_dim = kvqo_nvfp4_full_dim(head_size);
    int32_t data_dim = kvqo_nvfp4_data_dim(full_dim);
    int32_t scale_dim = kvqo_nvfp4_scale_dim(full_dim);
    return (int64_t)block_size * num_heads * data_dim + row * scale_dim;
}

/* [P2] "Implementation breakdown" item 4: reshape_and_cache_nvfp4_kernel
 * quantises bf16 K and V to FP4 data plus e4m3 block scales with a
 * per-tensor scale.  Format-spec reading of the per-tensor scale: y = x *
 * (1 / scale) in fp32, then the 16-value NVFP4 group recipe on y. */
int64_t kvqo_reshape_and_cache_nvfp4(
    const uint16_t* key, const uint16_t* value,
    int64_t key_stride_t, int64_t key_stride_h,
    int64_t value_stride_t, int64_t value_stride_h,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    int32_t num_heads, int32_t head_size,
    uint8_t* cache, int64_t num_pages, int32_t block_size,
    float k_scale, float v_scale, int32_t layout) {
    int64_t t, skipped = 0;
    for (t = t_begin; t < t_end; ++t) {
        int64_t slot = slot_mapping[t], page;
        int32_t off, h, side;
        if (slot < 0) continue;
        if (slot >= num_pages * (int64_t)block_size) { ++skipped; continue; }
        page = slot / block_size;
        off = (int32_t)(slot % block_size);
        for (side = 0; side < 2; ++side) {
            const uint16_t* src = side ? value : key;
            int64_t st = side ? value_stride_t : key_stride_t;
            int64_t sh = side ? value_stride_h : key_stride_h;
            float inv_scale = 1.0f / (side ? v_scale : k_scale);
            uint8_t* base = cache + perhead_side_base(page, side, block_size, num_heads, head_size);
            for (h = 0; h < num_heads; ++h) {
                int32_t g;
                int64_t row = perhead_row(off, h, block_size, num_heads, layout);
                uint8_t* data = base + perhead_data_off(row, head_size);
                uint8_t* scales = base + perhead_scale_off(row, block_size, num_heads, head_size);
                for (g = 0; g < head_size / NV_GROUP; ++g) {
                    float y[NV_GROUP];
                    int i;
                    for (i = 0; i < NV_GROUP; ++i)
                        y[i] = kvqo_bf16_value(src[t * st + h * sh + g * NV_GROUP + i]) * inv_scale;
                    scales[g] = nvfp4_group(y, &data[g * (NV_GROUP / 2)]);
                }
            }
        }
    }
    return skipped;
}

/* Read-back of the per-head cache ([P2] "Implementation breakdown" item 5,
 * dequant_nvfp4_kv_cache): value = bf16_rn((e2m1 * sf) * scale), where the
 * e2m1 * sf product is exact and the multiply by the per-tensor scale rounds
 * once in fp32. */
int64_t kvqo_dequant_nvfp4_per_head(
    const uint8_t* cache, int64_t num_pages, int32_t block_size,
    int32_t num_heads, int32_t head_size,
    const int64_t* slot_mapping, int64_t t_begin, int64_t t_end,
    float k_scale, float v_scale, int32_t layout, uint16_t* key_out, uint16_t* value_out) {
    int64_t t, skipped = 0;
    for (t = t_begin; t < t_end; ++t) {
        int64_t slot = slot_mapping[t], page;
        int32_t off, h, side, d;
        if (slot < 0) continue;
        if (slot >= num_pages * (int64_t)block_size) { ++skipped; continue; }
        page = slot / block_size;
        off = (int32_t)(slot % block_size);
        for (side = 0; side < 2; ++side) {
            uint16_t* out = side ? value_out : key_out;
            float scale = side ? v_scale : k_scale;
            const uint8_t* base = cache + perhead_side_base(page, side, block_size, num_heads, head_size);
            for (h = 0; h < num_heads; ++h) {
                int64_t row = perhead_row(off, h, block_size, num_heads, layout);
                const uint8_t* data = base + perhead_data_off(row, head_size);
                const uint8_t* scales = base + perhead_scale_off(row, block_size, num_heads, head_size);
                for (d = 0; d < head_size; ++d) {
                    uint8_t byte = data[d / 2];
                    uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
                    float q = (float)(kvqo_e2m1_value(nib) * kvqo_e4m3_value(scales[d / NV_GROUP]));
                    out[(t * num_heads + h) * (int64_t)head_size + d] = kvqo_bf16_rn(q * scale);
                }
            }
        }
    }
    return skipped;
}

/* ========================================================================== */
/* Sparse-decode index conversion                                             */
/* ========================================================================== */

/* [P3] "Implementation breakdown" item 1 (triton_convert_req_index_to_global
 * _index with its length check).  Format-spec reading of the conversion: for
 * token i of request r = req_id[i] and each of its topk positions p =
 * token_indices[i][k], the global slot is block_table[r][p / block_size] *
 * block_size + p % block_size; p < 0 (an unused top-k entry) gives -1, and so
 * does any index outside the table, which is also counted. */
int64_t kvqo_req_index_to_global_slot(
    const int32_t* req_id, const int32_t* token_indices, int64_t num_tokens,
    int32_t topk, const int32_t* block_table, int64_t block_table_stride,
    int32_t block_table_width, int32_t num_requests, int32_t block_size,
    int64_t num_blocks, int32_t* out) {
    int64_t i, skipped = 0;
    for (i = 0; i < num_tokens; ++i) {
        int32_t r = req_id[i], k;
        for (k = 0; k < topk; ++k) {
            int32_t p = token_indices[i * topk + k];
            int64_t column, block;
            out[i * topk + k] = -1;
            if (p < 0) continue;
            if (r < 0 || r >= num_requests) { ++skipped; continue; }
            column = p / block_size;
            if (column >= block_table_width) { ++skipped; continue; }
            block = block_table[(int64_t)r * block_table_stride + column];
            if (block < 0 || block >= num_blocks) { ++skipped; continue; }
            out[i * topk + k] = (int32_t)(block * block_size + p % block_size);
        }
    }
    return skipped;
}

/* ========================================================================== */
/* Sparse MLA attention straight from the nvfp4_ds_mla cache                  */
/* ========================================================================== */

/* The consumer of the cache: [P1] "Key source snippets" (flashmla_sparse.py:
 * the quantized DS-MLA formats are served by the sparse decode kernel path,
 * which reads the cache itself and infers the format from the bytes per
 * token) and [P3] "Implementation breakdown" item 3 (the decode side runs as
 * MQA over the latent cache).  Reading of the MQA step: every head h of
 * token t holds one 576-wide query q[t,h] (512 latent + 64 RoPE) and attends
 * over the token's top-k list of global slots; the key of slot j is its whole
 * decoded entry k_j (576 values), the value its 512 NoPE values.
 *   s_j = softmax_scale * (q[t,h] . k_j)
 *   o[t,h] = sum_j exp(s_j - m) k_j[0:512] / sum_j exp(s_j - m),  m = max_j s_j
 *   lse[t,h] = m + log(sum_j exp(s_j - m))            (natural logarithm)
 * over the valid entries of indices[t] (negative entries are unused; a slot
 * beyond the cache is skipped and counted).  A token with no valid entry
 * gets o = 0 and lse = -inf.  Everything in double, entries decoded exactly. */
/* Softmax attention of the heads of one query token over n decoded keys
 * (576 values each): s_j = scale * q . k_j, o = sum_j exp(s_j - m) k_j[0:512]
 * / sum_j exp(s_j - m), lse = m + log sum_j exp(s_j - m), all in double;
 * n = 0 gives o = 0, lse = -inf.  s is scratch for n scores. */
static void attend_token(const uint16_t* q_t, int64_t q_stride_h, int32_t num_heads, const double* keys, int32_t n,
                         double softmax_scale, double* s, double* out_t, int64_t out_stride_h, double* lse_t) {
    const int dim = NV_NOPE_DIM + NV_ROPE_DIM;
    int32_t h;
    for (h = 0; h < num_heads; ++h) {
        const uint16_t* qh = q_t + (int64_t)h * q_stride_h;
        double* oh = out_t + (int64_t)h * out_stride_h;
        double m = -INFINITY, l = 0.0;
        int d, j;
        for (d = 0; d < NV_NOPE_DIM; ++d) oh[d] = 0.0;
        for (j = 0; j < n; ++j) {
            double dot = 0.0;
            for (d = 0; d < dim; ++d) dot += (double)kvqo_bf16_value(qh[d]) * keys[(int64_t)j * dim + d];
            s[j] = softmax_scale * dot;
            if (s[j] > m) m = s[j];
        }
        for (j = 0; j < n; ++j) {
            double w = exp(s[j] - m);
            l += w;
            for (d = 0; d < NV_NOPE_DIM; ++d) oh[d] += w * keys[(int64_t)j * dim + d];
        }
        if (n > 0)
            for (d = 0; d < NV_NOPE_DIM; ++d) oh[d] /= l;
        if (lse_t) lse_t[h] = (n > 0) ? m + log(l) : -INFINITY;
    }
}

static int64_t sparse_mla_attention(
    void (*decode)(const uint8_t*, double*),
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t t_begin, int64_t t_end, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    const int dim = NV_NOPE_DIM + NV_ROPE_DIM;
    int64_t t, skipped = 0;
    double* keys = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * dim);
    double* s = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    if (!keys || !s) { free(keys); free(s); return -1; }
    for (t = t_begin; t < t_end; ++t) {
        int32_t n = 0, k;
        for (k = 0; k < topk; ++k) {
            int64_t slot = indices[t * indices_stride + k];
            if (slot < 0) continue;
            if (slot >= num_blocks * (int64_t)block_size) { ++skipped; continue; }
            decode(cache + (slot / block_size) * block_stride + (slot % block_size) * entry_stride,
                   keys + (int64_t)n * dim);
            ++n;
        }
        attend_token(q + t * q_stride_t, q_stride_h, num_heads, keys, n, softmax_scale, s, out + t * out_stride_t,
                     out_stride_h, lse ? lse + t * lse_stride_t : NULL);
    }
    free(keys);
    free(s);
    return skipped;
}

int64_t kvqo_sparse_mla_attention_nvfp4_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t t_begin, int64_t t_end, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    return sparse_mla_attention(kvqo_decode_nvfp4_ds_mla_entry, q, q_stride_t, q_stride_h, t_begin, t_end,
                                num_heads, indices, indices_stride, topk, cache, num_blocks, block_size,
                                block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h,
                                lse, lse_stride_t);
}

/* The same consumer over the 656-byte fp8_ds_mla cache ([P1] "Key source
 * snippets": the sparse decode path serves both quantized DS-MLA formats).
 * A slot's key is the fp8 gather's upconvert of its entry: NoPE value k =
 * bf16_rn(fp32(e4m3(n_k)) * s_{k/128}), RoPE bf16 as stored. */
void kvqo_decode_fp8_ds_mla_entry(const uint8_t* entry, double* out576) {
    int k;
    for (k = 0; k < NV_NOPE_DIM; ++k) {
        float s;
        memcpy(&s, &entry[F8_SCALE_OFF + 4 * (k / F8_TILE)], 4);
        out576[k] = kvqo_bf16_value(kvqo_bf16_rn((float)kvqo_e4m3_value(entry[k]) * s));
    }
    for (k = 0; k < NV_ROPE_DIM; ++k)
        out576[NV_NOPE_DIM + k] = kvqo_bf16_value(
            (uint16_t)(entry[F8_ROPE_OFF + 2 * k] | (entry[F8_ROPE_OFF + 2 * k + 1] << 8)));
}

int64_t kvqo_sparse_mla_attention_fp8_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h,
    int64_t t_begin, int64_t t_end, int32_t num_heads,
    const int32_t* indices, int64_t indices_stride, int32_t topk,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    return sparse_mla_attention(kvqo_decode_fp8_ds_mla_entry, q, q_stride_t, q_stride_h, t_begin, t_end,
                                num_heads, indices, indices_stride, topk, cache, num_blocks, block_size,
                                block_stride, entry_stride, softmax_scale, out, out_stride_t, out_stride_h,
                                lse, lse_stride_t);
}

/* Dense prefill over the quantized cache ([P3] "Function and motivation" and
 * "Key source snippets", _compute_prefill_context: a request's whole context
 * is read through its block-table row and attended densely; the MQA form of
 * the sparse decode, reading 21 of the build's spec).  Request b (b_begin <=
 * b < b_end) owns the query tokens [query_start[b], query_start[b+1]); each of
 * them attends, with every head, to the positions p < context_lens[b] of its
 * context, position p being entry p % block_size of block
 * block_table[b][p / block_size].  Positions whose block-table column or block
 * id is out of range are skipped and counted. */
static int64_t prefill_mla_attention(
    void (*decode)(const uint8_t*, double*),
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int64_t b_begin, int64_t b_end,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    const int dim = NV_NOPE_DIM + NV_ROPE_DIM;
    int64_t b, skipped = 0;
    for (b = b_begin; b < b_end; ++b) {
        const int32_t ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        double* keys = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * dim);
        double* s = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
        int32_t n = 0, p;
        int64_t t;
        if (!keys || !s) { free(keys); free(s); return -1; }
        for (p = 0; p < ctx; ++p) {
            const int32_t col = p / block_size;
            int64_t id;
            if (col >= block_table_width) { ++skipped; continue; }
            id = block_table[b * block_table_stride + col];
            if (id < 0 || id >= num_blocks) { ++skipped; continue; }
            decode(cache + id * block_stride + (int64_t)(p % block_size) * entry_stride, keys + (int64_t)n * dim);
            ++n;
        }
        for (t = query_start[b]; t < query_start[b + 1]; ++t)
            attend_token(q + t * q_stride_t, q_stride_h, num_heads, keys, n, softmax_scale, s,
                         out + t * out_stride_t, out_stride_h, lse ? lse + t * lse_stride_t : NULL);
        free(keys);
        free(s);
    }
    return skipped;
}

int64_t kvqo_prefill_mla_attention_nvfp4_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int64_t b_begin, int64_t b_end,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    return prefill_mla_attention(kvqo_decode_nvfp4_ds_mla_entry, q, q_stride_t, q_stride_h, num_heads, query_start,
                                 context_lens, block_table, block_table_stride, block_table_width, b_begin, b_end,
                                 cache, num_blocks, block_size, block_stride, entry_stride, softmax_scale, out,
                                 out_stride_t, out_stride_h, lse, lse_stride_t);
}

int64_t kvqo_prefill_mla_attention_fp8_ds_mla(
    const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int32_t num_heads,
    const int32_t* query_start, const int32_t* context_lens,
    const int32_t* block_table, int64_t block_table_stride, int32_t block_table_width,
    int64_t b_begin, int64_t b_end,
    const uint8_t* cache, int64_t num_blocks, int32_t block_size,
    int64_t block_stride, int64_t entry_stride, double softmax_scale,
    double* out, int64_t out_stride_t, int64_t out_stride_h,
    double* lse, int64_t lse_stride_t) {
    return prefill_mla_attention(kvqo_decode_fp8_ds_mla_entry, q, q_stride_t, q_stride_h, num_heads, query_start,
                                 context_lens, block_table, block_table_stride, block_table_width, b_begin, b_end,
                                 cache, num_blocks, block_size, block_stride, entry_stride, softmax_scale, out,
                                 out_stride_t, out_stride_h, lse, lse_stride_t);
}
