/*
 * bsq_oracle.c -- the CPU oracle for the block-scaled packed-precision path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * restatement of what the GPU path computes.  Only the tests, the smoke check
 * and the benchmark's cpu_baseline leg load it.  It shares no code, header,
 * table or constant generator with the CUDA library; neither side includes or
 * links the other.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (no FMA contraction: every f32 step below is one IEEE-754 operation, as the
 * elementwise-parity page does with `volatile` -- Winery-Strata
 * elementwise_parity.cpp, "packed embedding rows" block).
 *
 * Sources (page title, then function / section):
 *   [P1] cubecl-tile tests/tile/packed.rs: nvfp4_shaped_matmul,
 *        nvfp4_shaped_decode, check_fp4_codes_unpack, check_fp8_codes_unpack,
 *        words_of_bytes, check_ue8m0_scales, packed_one_row_product.
 *   [P2] b12x _lib/fp6.py: FLOAT6_E3M2_MAX .. FLOAT8_E4M3_MAX constants,
 *        mx_gs_numerator, _decode_fp6_e3m2, _decode_fp6_e2m3,
 *        _encode_fp6_nearest, pack_4_fp6_codes, mxfp6_swizzled_scale_offset,
 *        unswizzle_mxfp6_scales, dequant_mxfp6_torch,
 *        quantize_grouped_mxfp6_torch, fp6_block_ue8m0_exact,
 *        ue8m0_output_scale_exact, quantize_block_fp6_*_fast,
 *        relu2_quantize_grouped_mxfp6_torch, silu_mul_quantize_grouped_mxfp6_torch.
 *   [P3] Winery-Strata elementwise_parity.cpp: the f32 -> bf16 RNE rule.
 *
 * Parity status of each function (what pins it is in tests/test_oracle_*.py):
 *   decoders, encoders, packers, swizzle, MX quantizer, products: pinned.
 *   NVFP4 quantizer: the pages give no NVFP4 recipe; the recipe here is the
 *   MX recipe carried over by analogy (a reading).  It is pinned only by
 *   invariants (power-of-two equivariance, error bound, zero blocks), so its
 *   recipe choice itself is "parity unpinned" by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define BSQO_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Formats.  fmt ids used across the oracle API.                              */
/* ------------------------------------------------------------------------ */
enum { FMT_E3M2 = 0, FMT_E2M3 = 1, FMT_E4M3 = 2, FMT_E2M1 = 3, FMT_UE4M3 = 4 };

/* [P2] constants: the largest finite magnitude of each element format.       */
static const float FMT_MAX_E3M2 = 28.0f;
static const float FMT_MAX_E2M3 = 7.5f;
static const float FMT_MAX_E4M3 = 448.0f;
/* e2m1's largest value, 2^(3-1) * (1 + 1/2); the pages reach e2m1 only
 * through its decoder ([P1] check_fp4_codes_unpack), so this is its closed form. */
static const float FMT_MAX_E2M1 = 6.0f;

static inline float f32_of_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static inline uint32_t bits_of_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the top half of an f32. */
static inline float bf16_to_f32(uint16_t b) { return f32_of_bits((uint32_t)b << 16); }

/* ------------------------------------------------------------------------ */
/* Decoders: closed forms, exact in double.                                   */
/* ------------------------------------------------------------------------ */

/* [P2] _decode_fp6_e3m2: 1 sign, 3 exponent (bias 3), 2 mantissa bits, no
 * inf/nan; exponent 0 is subnormal 2^(1-3) * m/4.                            */
BSQO_API double bsqo_decode_e3m2(unsigned c) {
    c &= 0x3F;
    double s = (c >> 5) & 1 ? -1.0 : 1.0;
    int e = (c >> 2) & 7, m = c & 3;
    if (e == 0) return s * ldexp(m / 4.0, 1 - 3);
    return s * ldexp(1.0 + m / 4.0, e - 3);
}

/* [P2] _decode_fp6_e2m3: 1 sign, 2 exponent (bias 1), 3 mantissa bits.       */
BSQO_API double bsqo_decode_e2m3(unsigned c) {
    c &= 0x3F;
    double s = (c >> 5) & 1 ? -1.0 : 1.0;
    int e = (c >> 3) & 3, m = c & 7;
    if (e == 0) return s * ldexp(m / 8.0, 1 - 1);
    return s * ldexp(1.0 + m / 8.0, e - 1);
}

/* OCP e2m1 (the nvfp4 field of [P1] nvfp4_shaped_decode): 1 sign, 2 exponent
 * (bias 1), 1 mantissa bit; exponent 0 is subnormal m/2.                     */
BSQO_API double bsqo_decode_e2m1(unsigned c) {
    c &= 0xF;
    double s = (c >> 3) & 1 ? -1.0 : 1.0;
    int e = (c >> 1) & 3, m = c & 1;
    if (e == 0) return s * ldexp(m / 2.0, 1 - 1);
    return s * ldexp(1.0 + m / 2.0, e - 1);
}

/* OCP e4m3 "fn" ([P1] check_fp8_codes_unpack decodes every non-NaN code):
 * bias 7, 3 mantissa bits, S.1111.111 is NaN, no infinities.                  */
BSQO_API double bsqo_decode_e4m3(unsigned c) {
    c &= 0xFF;
    double s = (c >> 7) & 1 ? -1.0 : 1.0;
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return s * ldexp(m / 8.0, 1 - 7);
    return s * ldexp(1.0 + m / 8.0, e - 7);
}

/* ue4m3: e4m3 without a sign (the nvfp4 block scale).  A set top bit is
 * outside the format; it decodes as NaN so that a caller cannot miss it.     */
BSQO_API double bsqo_decode_ue4m3(unsigned c) {
    c &= 0xFF;
    if (c & 0x80) return NAN;
    return bsqo_decode_e4m3(c);
}

/* UE8M0: a bare biased exponent, value 2^(c-127); 0xFF is NaN ([P1]
 * check_ue8m0_scales: "the code is the exponent biased by 127").             */
BSQO_API double bsqo_decode_ue8m0(unsigned c) {
    c &= 0xFF;
    if (c == 0xFF) return NAN;
    return ldexp(1.0, (int)c - 127);
}

BSQO_API double bsqo_decode(int fmt, unsigned c) {
    switch (fmt) {
    case FMT_E3M2: return bsqo_decode_e3m2(c);
    case FMT_E2M3: return bsqo_decode_e2m3(c);
    case FMT_E4M3: return bsqo_decode_e4m3(c);
    case FMT_E2M1: return bsqo_decode_e2m1(c);
    case FMT_UE4M3: return bsqo_decode_ue4m3(c);
    default: return NAN;
    }
}

static int fmt_bits(int fmt) {
    switch (fmt) {
    case FMT_E3M2: case FMT_E2M3: return 6;
    case FMT_E4M3: return 8;
    case FMT_E2M1: return 4;
    default: return 0;
    }
}

static float fmt_max(int fmt) {
    switch (fmt) {
    case FMT_E3M2: return FMT_MAX_E3M2;
    case FMT_E2M3: return FMT_MAX_E2M3;
    case FMT_E4M3: return FMT_MAX_E4M3;
    case FMT_E2M1: return FMT_MAX_E2M1;
    default: return 0.0f;
    }
}

/* ------------------------------------------------------------------------ */
/* Encoder.                                                                   */
/* ------------------------------------------------------------------------ */

/* Values of the magnitude codes, filled once when the library loads. */
static double mag_table[4][128];
__attribute__((constructor)) static void fill_mag_tables(void) {
    for (int f = 0; f < 4; ++f)
        for (unsigned c = 0; c < 128; ++c)
            mag_table[f][c] = c < (1u << (fmt_bits(f) - 1)) ? bsqo_decode(f, c) : NAN;
}

/* [P2] _encode_fp6_nearest, restated for every element format: clamp to the
 * format's largest magnitude, then take the code whose value is nearest; on a
 * tie take the code whose lowest bit (the mantissa LSB) is even.
 *
 * Reading (sign of zero): the search runs over the magnitude codes of |v| and
 * the sign bit is then copied from v, so -0.0 and negatives that round to
 * zero give the negative-zero code.  This is what an IEEE round-to-nearest
 * conversion with saturation does; the page's own loop returns +0 for them.
 * The two choices decode to the same value.                                  */
BSQO_API unsigned bsqo_encode(int fmt, float v) {
    int bits = fmt_bits(fmt);
    unsigned sign_bit = 1u << (bits - 1);
    unsigned n_mag = sign_bit;              /* magnitude codes 0 .. sign_bit-1 */
    double mag = fabs((double)v);
    double mx = fmt_max(fmt);
    if (mag > mx) mag = mx;                 /* clamp (saturate) */
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < n_mag; ++c) {
        double val = mag_table[fmt][c];
        if (isnan(val)) continue;           /* e4m3's 0x7F */
        double d = fabs(val - mag);
        if (d < best_d) { best_d = d; best = c; }
        else if (d == best_d && (c & 1) == 0 && (best & 1) == 1) best = c;
    }
    if (signbit(v)) best |= sign_bit;
    return best;
}

/* ------------------------------------------------------------------------ */
/* Packing.                                                                   */
/* ------------------------------------------------------------------------ */

/* [P2] pack_4_fp6_codes: four 6-bit codes in a little-endian 24-bit lane,
 * c0 | c1<<6 | c2<<12 | c3<<18, stored as three bytes, low byte first.     */
BSQO_API void bsqo_pack_fp6(const uint8_t* codes, int64_t n, uint8_t* out) {
    for (int64_t g = 0; g < n / 4; ++g) {
        uint32_t bits = (uint32_t)(codes[4 * g] & 0x3F)
                      | (uint32_t)(codes[4 * g + 1] & 0x3F) << 6
                      | (uint32_t)(codes[4 * g + 2] & 0x3F) << 12
                      | (uint32_t)(codes[4 * g + 3] & 0x3F) << 18;
        out[3 * g] = bits & 0xFF;
        out[3 * g + 1] = (bits >> 8) & 0xFF;
        out[3 * g + 2] = (bits >> 16) & 0xFF;
    }
}

/* [P2] unpack_4_fp6_codes: the inverse.                                      */
BSQO_API void bsqo_unpack_fp6(const uint8_t* packed, int64_t n, uint8_t* codes) {
    for (int64_t g = 0; g < n / 4; ++g) {
        uint32_t bits = (uint32_t)packed[3 * g] | (uint32_t)packed[3 * g + 1] << 8
                      | (uint32_t)packed[3 * g + 2] << 16;
        codes[4 * g] = bits & 0x3F;
        codes[4 * g + 1] = (bits >> 6) & 0x3F;
        codes[4 * g + 2] = (bits >> 12) & 0x3F;
        codes[4 * g + 3] = (bits >> 18) & 0x3F;
    }
}

/* [P1] module doc + nvfp4_shaped_decode: a packed word holds 32/bits values,
 * low field first; e2m1 is eight to a 32-bit word.                           */
static inline unsigned nvfp4_code_at(const uint32_t* words, int64_t row_words, int64_t r, int64_t k) {
    uint32_t w = words[r * row_words + k / 8];
    return (w >> (4 * (k % 8))) & 0xF;
}

/* One code of an MX operand: fp6 rows are 3K/4 packed bytes, e4m3 rows K bytes. */
static inline unsigned mx_code_at(const uint8_t* codes, int fmt, int64_t K, int64_t r, int64_t k) {
    if (fmt == FMT_E4M3) return codes[r * K + k];
    const uint8_t* p = codes + r * (3 * K / 4) + 3 * (k / 4);
    uint32_t bits = (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16;
    return (bits >> (6 * (k % 4))) & 0x3F;
}

/* ------------------------------------------------------------------------ */
/* Block-scale layout.                                                        */
/* ------------------------------------------------------------------------ */

static inline int64_t pad_to(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

/* [P2] mxfp6_swizzled_scale_offset: byte offset of the scale of (row, block)
 * in a buffer of pad128(rows) x pad4(blocks) bytes:
 *   ((((row/128)*(pad4(blocks)/4) + block/4)*32 + row%32)*4 + (row%128)/32)*4 + block%4
 * Reading: the same layout serves every block-scale buffer here (UE8M0 per 32
 * and the nvfp4 ue4m3 per 16).                                              */
BSQO_API int64_t bsqo_swz_offset(int64_t row, int64_t block, int64_t n_blocks) {
    int64_t cpd4 = pad_to(n_blocks, 4) / 4;
    return ((((row / 128) * cpd4 + block / 4) * 32 + row % 32) * 4 + (row % 128) / 32) * 4 + block % 4;
}

BSQO_API int64_t bsqo_scale_bytes(int64_t rows, int64_t n_blocks) {
    return pad_to(rows, 128) * pad_to(n_blocks, 4);
}

/* ------------------------------------------------------------------------ */
/* Scale arithmetic of the quantizers, one IEEE f32 operation per step.       */
/* ------------------------------------------------------------------------ */

/* [P2] mx_gs_numerator: gs = numerator / amax, numerator = 448 * fmt_max.
 * Reading: for nvfp4 the numerator is 448 * 6 = 2688 by the same rule.     */
BSQO_API float bsqo_gs_numerator(int fmt) { return FMT_MAX_E4M3 * fmt_max(fmt); }

/* [P2] fp6_block_ue8m0_exact: ratio = (amax_b * gs) / fmt_max with a rounded
 * multiply and a rounded divide; the byte is the ratio's exponent field plus
 * one if its mantissa is non-zero (an exact ceil(log2)), clamped to [0, 255];
 * a ratio <= 0 gives 0.                                                     */
BSQO_API unsigned bsqo_ue8m0_from_block_max(float amax_b, float gs, float fmax) {
    volatile float t = amax_b * gs;
    volatile float ratio = t / fmax;
    uint32_t b = bits_of_f32(ratio);
    int32_t expf = (int32_t)((b & 0x7F800000u) >> 23);
    int32_t r = expf + ((b & 0x007FFFFFu) != 0 ? 1 : 0);
    if (r < 0) r = 0;
    if (r > 255) r = 255;
    if (ratio <= 0.0f) r = 0;
    return (unsigned)r;
}

/* [P2] ue8m0_output_scale_exact: gs * 2^(127-ue), with the power of two built
 * from its bits (exponent field 254-ue, zero mantissa); 0 when ue == 0.      */
BSQO_API float bsqo_ue8m0_output_scale(unsigned ue, float gs) {
    if (ue == 0) return 0.0f;
    float p = f32_of_bits((uint32_t)(254 - (int32_t)ue) << 23);
    volatile float r = p * gs;
    return r;
}

static float tensor_amax(const uint16_t* x, int64_t n) {
    float a = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = fabsf(bf16_to_f32(x[i]));
        if (v > a) a = v;
    }
    return a;
}

/* ------------------------------------------------------------------------ */
/* MX quantizer (e3m2 / e2m3 / e4m3, UE8M0 per 32).                           */
/* ------------------------------------------------------------------------ */

/* [P2] quantize_grouped_mxfp6_torch (one group, every row valid) with the
 * exact scale steps of fp6_block_ue8m0_exact / ue8m0_output_scale_exact and
 * the block quantizer quantize_block_fp6_*_fast:
 *   amax over the tensor; gs = num / amax (0 if amax == 0);
 *   per 32-block: amax_b; ue from (amax_b*gs)/fmt_max by the exact ceil;
 *   inv = gs * 2^(127-ue); code_i = nearest(x_i * inv) if inv != 0, else 0;
 *   fp6 codes packed 4-in-3, e4m3 codes one byte each; scales swizzled.
 * Reading (single rounding): x_i * inv is encoded from f32 directly, not via
 * bf16 (bf16_round=False).  Reading (dequant factor): the library hands out
 * s_global = 1/gs (f32 divide), 0 if gs == 0, which dequant multiplies by.
 * codes: [M, 3K/4] (fp6) or [M, K] (e4m3); scales: pad128(M)*pad4(K/32).    */
/* One row of the MX quantizer: codes (packed row) and the row's UE8M0 bytes. */
static void quantize_mx_row(const uint16_t* xr, int64_t K, int fmt, float gs,
                            uint8_t* codes_row, uint8_t* ue_row, int containers) {
    const float fmax = fmt_max(fmt);
    uint8_t blk[32];
    for (int64_t b = 0; b < K / 32; ++b) {
        const uint16_t* xb = xr + b * 32;
        float amax_b = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float v = fabsf(bf16_to_f32(xb[i]));
            if (v > amax_b) amax_b = v;
        }
        unsigned ue = 0;
        float inv = 0.0f;
        if (gs != 0.0f) {
            ue = bsqo_ue8m0_from_block_max(amax_b, gs, fmax);
            inv = bsqo_ue8m0_output_scale(ue, gs);
        }
        memset(blk, 0, sizeof blk);
        if (inv != 0.0f) {
            for (int i = 0; i < 32; ++i) {
                volatile float q = bf16_to_f32(xb[i]) * inv;
                blk[i] = (uint8_t)bsqo_encode(fmt, q);
            }
        }
        if (fmt == FMT_E4M3 || containers) memcpy(codes_row + b * 32, blk, 32);
        else bsqo_pack_fp6(blk, 32, codes_row + b * 24);
        ue_row[b] = (uint8_t)ue;
    }
}

static float mx_global_scale(const uint16_t* x, int64_t n, int fmt) {
    const float amax = tensor_amax(x, n);
    volatile float gs = 0.0f;
    if (amax > 0.0f) gs = bsqo_gs_numerator(fmt) / amax;
    return gs;
}

/* [P2] quantize_grouped_mxfp6_torch (one group, every row valid) with the
 * exact scale steps of fp6_block_ue8m0_exact / ue8m0_output_scale_exact and
 * the block quantizer quantize_block_fp6_*_fast:
 *   amax over the tensor; gs = num / amax (0 if amax == 0);
 *   per 32-block: amax_b; ue from (amax_b*gs)/fmt_max by the exact ceil;
 *   inv = gs * 2^(127-ue); code_i = nearest(x_i * inv) if inv != 0, else 0;
 *   fp6 codes packed 4-in-3, e4m3 codes one byte each; scales swizzled.
 * Reading (single rounding): x_i * inv is encoded from f32 directly, not via
 * bf16 (bf16_round=False).  Reading (dequant factor): the library hands out
 * s_global = 1/gs (f32 divide), 0 if gs == 0, which dequant multiplies by.
 * codes: [M, 3K/4] (fp6) or [M, K] (e4m3); scales: pad128(M)*pad4(K/32).    */
BSQO_API int bsqo_quantize_mx(const uint16_t* x, int64_t M, int64_t K, int fmt,
                              uint8_t* codes, uint8_t* scales, float* s_global) {
    if (fmt != FMT_E3M2 && fmt != FMT_E2M3 && fmt != FMT_E4M3) return 1;
    if (M < 0 || K < 0 || K % 32) return 1;
    const int64_t nb = K / 32;
    const int64_t row_bytes = fmt == FMT_E4M3 ? K : 3 * K / 4;
    const float gs = mx_global_scale(x, M * K, fmt);
    memset(scales, 0, (size_t)bsqo_scale_bytes(M, nb));
    uint8_t* ue_row = (uint8_t*)malloc((size_t)(nb > 0 ? nb : 1));
    for (int64_t r = 0; r < M; ++r) {
        quantize_mx_row(x + r * K, K, fmt, gs, codes + r * row_bytes, ue_row, 0);
        for (int64_t b = 0; b < nb; ++b) scales[bsqo_swz_offset(r, b, nb)] = ue_row[b];
    }
    free(ue_row);
    *s_global = gs != 0.0f ? 1.0f / gs : 0.0f;
    return 0;
}

/* [P2] quantize_block_fp6_e3m2_bytes / _e2m3_bytes with
 * pack_32_byte_containers_to_4xu64: the same quantizer, fp6 codes written one
 * per byte (bits [5:0], bits [7:6] zero) in K order instead of four in three
 * bytes.  codes: [M, K] bytes; scales and s_global as bsqo_quantize_mx.      */
BSQO_API int bsqo_quantize_mx_containers(const uint16_t* x, int64_t M, int64_t K, int fmt,
                                         uint8_t* codes, uint8_t* scales, float* s_global) {
    if (fmt != FMT_E3M2 && fmt != FMT_E2M3) return 1;
    if (M < 0 || K < 0 || K % 32) return 1;
    const int64_t nb = K / 32;
    const float gs = mx_global_scale(x, M * K, fmt);
    memset(scales, 0, (size_t)bsqo_scale_bytes(M, nb));
    uint8_t* ue_row = (uint8_t*)malloc((size_t)(nb > 0 ? nb : 1));
    for (int64_t r = 0; r < M; ++r) {
        quantize_mx_row(x + r * K, K, fmt, gs, codes + r * K, ue_row, 1);
        for (int64_t b = 0; b < nb; ++b) scales[bsqo_swz_offset(r, b, nb)] = ue_row[b];
    }
    free(ue_row);
    *s_global = gs != 0.0f ? 1.0f / gs : 0.0f;
    return 0;
}

/* [P2] quantize_grouped_mxfp6_torch (several groups) and
 * as_grouped_mxfp6_scale_view: x [G, R, C] bf16; group g's first row_counts[g]
 * rows are quantized with the group's own global scale gs[g] (given, as on the
 * page -- not derived from an amax), rows past row_counts[g] are zero codes and
 * zero scales.  codes: [G, R, row_bytes] group-major (the page stores
 * [R, 3C/4, G]; codes_page[r, j, g] = codes[g, r, j]); scales: G consecutive
 * swizzled buffers of pad128(R)*pad4(C/32) bytes (the page's 6-D view is this
 * storage); s_global[g] = 1/gs[g] (0 if gs[g] == 0).                        */
BSQO_API int bsqo_quantize_grouped_mx(const uint16_t* x, int64_t G, int64_t R, int64_t C,
                                      const int64_t* row_counts, const float* gs, int fmt,
                                      uint8_t* codes, uint8_t* scales, float* s_global) {
    if (fmt != FMT_E3M2 && fmt != FMT_E2M3 && fmt != FMT_E4M3) return 1;
    if (G < 1 || R < 1 || C < 32 || C % 32) return 1;
    const int64_t nb = C / 32;
    const int64_t row_bytes = fmt == FMT_E4M3 ? C : 3 * C / 4;
    const int64_t sbytes = bsqo_scale_bytes(R, nb);
    memset(codes, 0, (size_t)(G * R * row_bytes));
    memset(scales, 0, (size_t)(G * sbytes));
    uint8_t* ue_row = (uint8_t*)malloc((size_t)nb);
    for (int64_t g = 0; g < G; ++g) {
        const int64_t valid = row_counts[g] < 0 ? 0 : (row_counts[g] > R ? R : row_counts[g]);
        for (int64_t r = 0; r < valid; ++r) {
            quantize_mx_row(x + (g * R + r) * C, C, fmt, gs[g], codes + (g * R + r) * row_bytes, ue_row, 0);
            for (int64_t b = 0; b < nb; ++b) scales[g * sbytes + bsqo_swz_offset(r, b, nb)] = ue_row[b];
        }
        volatile float inv = 0.0f;
        if (gs[g] != 0.0f) inv = 1.0f / gs[g];
        s_global[g] = inv;
    }
    free(ue_row);
    return 0;
}

/* The same quantizer for a subset of rows (the tensor amax still spans all
 * M rows): codes [n_rows, row_bytes] and plain row-major scales [n_rows, K/32]. */
BSQO_API int bsqo_quantize_mx_rows(const uint16_t* x, int64_t M, int64_t K, int fmt,
                                   const int64_t* rows, int64_t n_rows,
                                   uint8_t* codes, uint8_t* ue, float* s_global) {
    if (fmt != FMT_E3M2 && fmt != FMT_E2M3 && fmt != FMT_E4M3) return 1;
    if (M < 0 || K < 0 || K % 32) return 1;
    const int64_t row_bytes = fmt == FMT_E4M3 ? K : 3 * K / 4;
    const float gs = mx_global_scale(x, M * K, fmt);
    for (int64_t i = 0; i < n_rows; ++i)
        quantize_mx_row(x + rows[i] * K, K, fmt, gs, codes + i * row_bytes, ue + i * (K / 32), 0);
    *s_global = gs != 0.0f ? 1.0f / gs : 0.0f;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantizer (e2m1, ue4m3 per 16, one f32 tensor factor).               */
/* ------------------------------------------------------------------------ */

/* One row of the nvfp4 quantizer: eight codes per u32 word, low nibble first,
 * and the row's ue4m3 bytes.                                                */
static void quantize_nvfp4_row(const uint16_t* xr, int64_t K, float gs,
                               uint32_t* words_row, uint8_t* s_row) {
    memset(words_row, 0, (size_t)(K / 8) * 4);
    for (int64_t b = 0; b < K / 16; ++b) {
        const uint16_t* xb = xr + b * 16;
        float amax_b = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float v = fabsf(bf16_to_f32(xb[i]));
            if (v > amax_b) amax_b = v;
        }
        unsigned sb = 0;
        float inv = 0.0f;
        if (gs != 0.0f) {
            volatile float t = amax_b * gs;
            volatile float ratio = t / FMT_MAX_E2M1;
            sb = bsqo_encode(FMT_E4M3, ratio);      /* ratio >= +0: sign bit clear */
            if (sb != 0) {
                volatile float sv = (float)bsqo_decode_e4m3(sb);
                inv = gs / sv;
            }
        }
        if (inv != 0.0f) {
            for (int i = 0; i < 16; ++i) {
                volatile float q = bf16_to_f32(xb[i]) * inv;
                int64_t k = b * 16 + i;
                words_row[k / 8] |= (uint32_t)bsqo_encode(FMT_E2M1, q) << (4 * (k % 8));
            }
        }
        s_row[b] = (uint8_t)sb;
    }
}

static float nvfp4_global_scale(const uint16_t* x, int64_t n) {
    const float amax = tensor_amax(x, n);
    volatile float gs = 0.0f;
    if (amax > 0.0f) gs = bsqo_gs_numerator(FMT_E2M1) / amax;
    return gs;
}

/* Reading (the pages give no nvfp4 recipe): the MX recipe above with e2m1's
 * maximum 6 and an e4m3 block scale rounded to nearest (no ceil):
 *   gs = (448*6) / amax; s_b = e4m3_rn_sat((amax_b*gs) / 6);
 *   inv = gs / s_b (f32 divide), 0 if s_b == 0;
 *   code_i = e2m1_rn_sat(x_i * inv) if inv != 0, else 0.
 * codes: [M, K/8] u32, low nibble first; scales: pad128(M)*pad4(K/16).
 * Parity of the recipe choice is unpinned by the pages.                     */
BSQO_API int bsqo_quantize_nvfp4(const uint16_t* x, int64_t M, int64_t K,
                                 uint32_t* codes, uint8_t* scales, float* s_global) {
    if (M < 0 || K < 0 || K % 16) return 1;
    const int64_t nb = K / 16;
    const float gs = nvfp4_global_scale(x, M * K);
    memset(scales, 0, (size_t)bsqo_scale_bytes(M, nb));
    uint8_t* s_row = (uint8_t*)malloc((size_t)(nb > 0 ? nb : 1));
    for (int64_t r = 0; r < M; ++r) {
        quantize_nvfp4_row(x + r * K, K, gs, codes + r * (K / 8), s_row);
        for (int64_t b = 0; b < nb; ++b) scales[bsqo_swz_offset(r, b, nb)] = s_row[b];
    }
    free(s_row);
    *s_global = gs != 0.0f ? 1.0f / gs : 0.0f;
    return 0;
}

/* Row-subset form, as bsqo_quantize_mx_rows. */
BSQO_API int bsqo_quantize_nvfp4_rows(const uint16_t* x, int64_t M, int64_t K,
                                      const int64_t* rows, int64_t n_rows,
                                      uint32_t* codes, uint8_t* sb, float* s_global) {
    if (M < 0 || K < 0 || K % 16) return 1;
    const float gs = nvfp4_global_scale(x, M * K);
    for (int64_t i = 0; i < n_rows; ++i)
        quantize_nvfp4_row(x + rows[i] * K, K, gs, codes + i * (K / 8), sb + i * (K / 16));
    *s_global = gs != 0.0f ? 1.0f / gs : 0.0f;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization ([P1] packed_scaled_copy, [P2] dequant_mxfp6_torch).        */
/* ------------------------------------------------------------------------ */

/* value = decode(code) * scale(row, block) * g, in double (exact).
 * Reading (UE8M0 byte 0): 2^(0-127), the closed form; the page's dequant
 * maps it to 0.  The quantizer only writes byte 0 for blocks whose codes are
 * all zero, where the two readings agree.                                    */
BSQO_API int bsqo_dequant_mx(const uint8_t* codes, int fmt, const uint8_t* scales, double g,
                             int64_t R, int64_t K, double* out) {
    if (K % 32) return 1;
    const int64_t nb = K / 32;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            double s = bsqo_decode_ue8m0(scales[bsqo_swz_offset(r, k / 32, nb)]);
            out[r * K + k] = bsqo_decode(fmt, mx_code_at(codes, fmt, K, r, k)) * s * g;
        }
    return 0;
}

BSQO_API int bsqo_dequant_nvfp4(const uint32_t* codes, const uint8_t* scales, double g,
                                int64_t R, int64_t K, double* out) {
    if (K % 16) return 1;
    const int64_t nb = K / 16;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            double s = bsqo_decode_ue4m3(scales[bsqo_swz_offset(r, k / 16, nb)]);
            out[r * K + k] = bsqo_decode_e2m1(nvfp4_code_at(codes, K / 8, r, k)) * s * g;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Products: the plain definition, sum in double.                             */
/* ------------------------------------------------------------------------ */

/* Operand descriptors for the product oracle.  kind: 0 = bf16 values,
 * 1 = nvfp4 (u32 words + ue4m3 per 16), 2 = MX (fmt codes + UE8M0 per 32).  */
typedef struct {
    int kind;
    int fmt;
    const void* data;
    const uint8_t* scales;
    double g;
} operand;

static inline double operand_at(const operand* op, int64_t K, int64_t r, int64_t k) {
    switch (op->kind) {
    case 0:
        return (double)bf16_to_f32(((const uint16_t*)op->data)[r * K + k]);
    case 1: {
        double s = bsqo_decode_ue4m3(op->scales[bsqo_swz_offset(r, k / 16, K / 16)]);
        return bsqo_decode_e2m1(nvfp4_code_at((const uint32_t*)op->data, K / 8, r, k)) * s;
    }
    default: {
        double s = bsqo_decode_ue8m0(op->scales[bsqo_swz_offset(r, k / 32, K / 32)]);
        return bsqo_decode(op->fmt, mx_code_at((const uint8_t*)op->data, op->fmt, K, r, k)) * s;
    }
    }
}

/* [P1] nvfp4_shaped_matmul / packed_matmul_rhs, orientation Y = A * W^T:
 *   Y[m,n] = gA * gW * sum_k A[m,k] * W[n,k]
 * for the listed (m, n) pairs; S[i] = |gA*gW| * sum_k |A[m,k] * W[n,k]|, the
 * scale the error bound is stated against.                                   */
static void product_at(const operand* a, const operand* w, int64_t K,
                       const int64_t* mi, const int64_t* ni, int64_t cnt,
                       double* y, double* s, int nthreads) {
#ifdef _OPENMP
    /* nthreads <= 0: every processor (set explicitly: an earlier call's count
     * would otherwise persist) */
    omp_set_num_threads(nthreads > 0 ? nthreads : omp_get_num_procs());
#pragma omp parallel for schedule(dynamic, 16) if (nthreads != 1)
#endif
    for (int64_t i = 0; i < cnt; ++i) {
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = operand_at(a, K, mi[i], k) * operand_at(w, K, ni[i], k);
            acc += p;
            aacc += fabs(p);
        }
        double g = a->g * w->g;
        y[i] = acc * g;
        if (s) s[i] = aacc * fabs(g);
    }
}

/* GEMM, nvfp4 x nvfp4 (gA/gW are the tensor factors). */
BSQO_API int bsqo_gemm_nvfp4_at(const uint32_t* A, const uint8_t* sA, double gA,
                                const uint32_t* W, const uint8_t* sW, double gW, int64_t K,
                                const int64_t* mi, const int64_t* ni, int64_t cnt,
                                double* y, double* s, int nthreads) {
    if (K % 16) return 1;
    operand a = {1, FMT_E2M1, A, sA, gA}, w = {1, FMT_E2M1, W, sW, gW};
    product_at(&a, &w, K, mi, ni, cnt, y, s, nthreads);
    return 0;
}

/* GEMM, MX x MX (either side e3m2 / e2m3 / e4m3). */
BSQO_API int bsqo_gemm_mx_at(const uint8_t* A, int fa, const uint8_t* sA, double gA,
                             const uint8_t* W, int fw, const uint8_t* sW, double gW, int64_t K,
                             const int64_t* mi, const int64_t* ni, int64_t cnt,
                             double* y, double* s, int nthreads) {
    if (K % 32) return 1;
    operand a = {2, fa, A, sA, gA}, w = {2, fw, W, sW, gW};
    product_at(&a, &w, K, mi, ni, cnt, y, s, nthreads);
    return 0;
}

/* GEMV, bf16 activations x nvfp4 weight ([P1] packed_one_row_product). */
BSQO_API int bsqo_gemv_nvfp4_at(const uint16_t* x, const uint32_t* W, const uint8_t* sW, double gW,
                                int64_t K, const int64_t* mi, const int64_t* ni, int64_t cnt,
                                double* y, double* s, int nthreads) {
    if (K % 16) return 1;
    operand a = {0, 0, x, NULL, 1.0}, w = {1, FMT_E2M1, W, sW, gW};
    product_at(&a, &w, K, mi, ni, cnt, y, s, nthreads);
    return 0;
}

/* GEMV, bf16 activations x MX weight. */
BSQO_API int bsqo_gemv_mx_at(const uint16_t* x, const uint8_t* W, int fw, const uint8_t* sW, double gW,
                             int64_t K, const int64_t* mi, const int64_t* ni, int64_t cnt,
                             double* y, double* s, int nthreads) {
    if (K % 32) return 1;
    operand a = {0, 0, x, NULL, 1.0}, w = {2, fw, W, sW, gW};
    product_at(&a, &w, K, mi, ni, cnt, y, s, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fused activation + quantize ([P2] relu2_quantize_grouped_mxfp6_torch and  */
/* silu_mul_quantize_grouped_mxfp6_torch): the activation is evaluated in f32 */
/* and rounded to the input dtype (bf16), and that bf16 tensor is quantized   */
/* by the MX recipe above.                                                    */
/*   ReLU^2:    a = max(x, 0)^2 (one f32 product; exact, <= 16 significant    */
/*              bits), rounded to bf16.                                        */
/*   SiLU * up: the input row holds gate [0, K) then up [K, 2K);              */
/*              a = fl(fl(g / fl(1 + exp(-g))) * u), rounded to bf16.  SiLU   */
/*              is written as one division, g / (1 + e^-g), the logistic form */
/*              of g * sigmoid(g); exp is the C library's expf.               */
/* ------------------------------------------------------------------------ */
enum { BSQO_ACT_RELU2 = 1, BSQO_ACT_SILU_MUL = 2 };

BSQO_API uint16_t bsqo_f32_to_bf16(float f);

BSQO_API int bsqo_activate(const uint16_t* x, int64_t M, int64_t K, int act, uint16_t* out) {
    if (!x || !out || M < 1 || K < 1 || (act != BSQO_ACT_RELU2 && act != BSQO_ACT_SILU_MUL)) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            volatile float a;
            if (act == BSQO_ACT_RELU2) {
                const float v = bf16_to_f32(x[m * K + k]);
                const float r = v > 0.0f ? v : 0.0f;
                a = r * r;
            } else {
                const float g = bf16_to_f32(x[m * 2 * K + k]);
                const float u = bf16_to_f32(x[m * 2 * K + K + k]);
                volatile float e = expf(-g);
                volatile float d = 1.0f + e;
                volatile float sg = g / d;
                a = sg * u;
            }
            out[m * K + k] = bsqo_f32_to_bf16(a);
        }
    return 0;
}

BSQO_API int bsqo_quantize_mx_act(const uint16_t* x, int64_t M, int64_t K, int act, int fmt, uint8_t* codes,
                                  uint8_t* scales, float* s_global, uint16_t* act_out) {
    if (M < 1 || K < 32 || K % 32) return -1;
    uint16_t* a = act_out ? act_out : (uint16_t*)malloc((size_t)(M * K) * sizeof(uint16_t));
    if (!a) return -1;
    int rc = bsqo_activate(x, M, K, act, a);
    if (rc == 0) rc = bsqo_quantize_mx(a, M, K, fmt, codes, scales, s_global);
    if (!act_out) free(a);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Output rounding.                                                           */
/* ------------------------------------------------------------------------ */

/* [P3] "THE f32 -> bf16 CONVERSIONS KEEP A NaN A NaN": for a non-NaN f32 u,
 * bf16 = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 (round to nearest even);
 * a NaN keeps its top half with the quiet bit set.                           */
BSQO_API uint16_t bsqo_f32_to_bf16(float f) {
    uint32_t u = bits_of_f32(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 64);
    return (uint16_t)((u + (0x7FFFu + ((u >> 16) & 1u))) >> 16);
}

/* The same rounding taken once from a double (no intermediate f32): round to
 * 8 significant bits, ties to even, with bf16's subnormal step 2^-133 and
 * overflow to infinity.                                                     */
BSQO_API uint16_t bsqo_double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                            /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                           /* step of 8 significant bits */
    if (q < -133) q = -133;                  /* subnormal step */
    double n = nearbyint(ldexp(a, -q));      /* ties to even under the default mode */
    double r = ldexp(n, q);
    if (r >= 0x1p128) return sign | 0x7F80;  /* rounded past the largest bf16 */
    float rf = (float)r;                     /* exact: r has <= 8 significant bits */
    return sign | (uint16_t)(bits_of_f32(rf) >> 16);
}

/* bsqo_double_to_bf16 over an array (no arithmetic of its own). */
BSQO_API void bsqo_double_to_bf16_n(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bsqo_double_to_bf16(v[i]);
}
