// mx_encode.cuh -- the MX block encode shared by the quantizers (quantize.cu)
// and the GEMM that quantizes its bf16 activations in its prologue (gemm.cu):
// block amax, the exact ceil UE8M0 block scale and its encode multiplier
// (b12x _lib/fp6.py fp6_block_ue8m0_exact, ue8m0_output_scale_exact), and the
// RNE-satfinite encode of 32 values into packed words
// (quantize_block_fp6_*_fast; four-in-three packing, pack_fp6_values).
#pragma once

#include "bsq_device.cuh"

namespace bsq {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (lo * k, hi * k) in one packed fp32 multiply (two IEEE RN products).
__device__ __forceinline__ void mul2_rn(float lo, float hi, float k, float& r_lo, float& r_hi) {
    asm("{ .reg .b64 a, b, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %4}; mul.rn.f32x2 d, a, b; mov.b64 {%0, %1}, d; }"
        : "=f"(r_lo), "=f"(r_hi) : "f"(lo), "f"(hi), "f"(k));
}

// Largest |bf16| magnitude bits among the 32 values of one 64-byte unit.
__device__ __forceinline__ uint32_t absmax32_bits(const uint4 (&v)[4]) {
    const uint32_t m = 0x7FFF7FFFu;
    const uint32_t a = __vmaxu2(__vmaxu2(v[0].x & m, v[0].y & m), __vmaxu2(v[0].z & m, v[0].w & m));
    const uint32_t b = __vmaxu2(__vmaxu2(v[1].x & m, v[1].y & m), __vmaxu2(v[1].z & m, v[1].w & m));
    const uint32_t c = __vmaxu2(__vmaxu2(v[2].x & m, v[2].y & m), __vmaxu2(v[2].z & m, v[2].w & m));
    const uint32_t d = __vmaxu2(__vmaxu2(v[3].x & m, v[3].y & m), __vmaxu2(v[3].z & m, v[3].w & m));
    const uint32_t e = __vmaxu2(__vmaxu2(a, b), __vmaxu2(c, d));
    return max(e & 0xFFFFu, e >> 16);
}

// MX block scale from the block's amax (bf16 magnitude bits): the UE8M0 byte by
// the exact ceil rule and the encode multiplier inv = gs * 2^(127-ue).
template <int FMT>
__device__ __forceinline__ void mx_block_scale(uint32_t amax_bits, float gs, uint32_t& ue, float& inv) {
    ue = 0;
    inv = 0.0f;
    if (gs != 0.0f) {
        ue = ue8m0_from_block_max(bf16_bits_to_f32(amax_bits), gs, fmt_max(FMT));
        inv = ue8m0_output_scale(ue, gs);
    }
}

// The 32 codes of one MX block as output words: 6 (fp6, four codes in three
// bytes, c0 | c1<<6 | c2<<12 | c3<<18 little-endian) or 8 (e4m3, a byte each).
// All zero when inv == 0.  The conversion leaves each 6-bit code in its own
// byte with the top two bits clear, so a pair p = c0 | c1<<8 compacts to
// c0 | c1<<6 as p - (p>>8)*192, and disjoint fields combine by multiply-add.
// CONT: fp6 codes left one per byte (b12x fp6.py pack_32_byte_containers_to_4xu64).
template <int FMT, bool CONT = false>
__device__ __forceinline__ void mx_encode_words(const uint4 (&v)[4], float inv, uint32_t (&w)[8]) {
    if (inv == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0;
        return;
    }
    uint32_t p[16];   // p[i]: codes 2i (low byte) and 2i+1
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t x2 = (&v[i >> 2].x)[i & 3];
        float lo, hi;
        mul2_rn(bf16_lo(x2), bf16_hi(x2), inv, lo, hi);
        p[i] = cvt_x2<FMT>(lo, hi);
    }
    if constexpr (FMT == kE4M3 || CONT) {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = p[2 * k] + (p[2 * k + 1] << 16);
    } else {
        uint32_t g[8];    // g[j]: codes 4j..4j+3 -> 24 bits
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t a = p[2 * j] - (p[2 * j] >> 8) * 192u;
            const uint32_t b = p[2 * j + 1] - (p[2 * j + 1] >> 8) * 192u;
            g[j] = a + b * 4096u;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            w[3 * h + 0] = g[4 * h + 0] + (g[4 * h + 1] << 24);
            w[3 * h + 1] = (g[4 * h + 1] >> 8) + (g[4 * h + 2] << 16);
            w[3 * h + 2] = (g[4 * h + 2] >> 16) + (g[4 * h + 3] << 8);
        }
    }
}

}  // namespace bsq
