// dequant.cu -- out[r, k] = decode(code) * block_scale * g in fp32 (a test and
// debugging aid: cubecl-tile tests/tile/packed.rs packed_scaled_copy; b12x
// _lib/fp6.py dequant_mxfp6_torch).  decode * scale is exact in fp32, so the
// only rounding is the multiply by g.
#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

// Closed-form decoders (OCP minifloat fields; b12x _lib/fp6.py _decode_fp6_*).
__device__ __forceinline__ float dec_minifloat(uint32_t c, int ebits, int mbits, int bias) {
    const uint32_t sign = (c >> (ebits + mbits)) & 1u;
    const uint32_t e = (c >> mbits) & ((1u << ebits) - 1u), m = c & ((1u << mbits) - 1u);
    float v;
    if (e == 0) v = (float)m * __uint_as_float((uint32_t)(127 + 1 - bias - mbits) << 23);
    else v = __uint_as_float(((e + 127u - (uint32_t)bias) << 23) | (m << (23 - mbits)));
    return sign ? -v : v;
}

__device__ __forceinline__ float dec_e2m1(uint32_t c) { return dec_minifloat(c & 0xF, 2, 1, 1); }
__device__ __forceinline__ float dec_e3m2(uint32_t c) { return dec_minifloat(c & 0x3F, 3, 2, 3); }
__device__ __forceinline__ float dec_e2m3(uint32_t c) { return dec_minifloat(c & 0x3F, 2, 3, 1); }
__device__ __forceinline__ float dec_e4m3(uint32_t c) {
    c &= 0xFF;
    if ((c & 0x7F) == 0x7F) return __uint_as_float(0x7FC00000u);
    return dec_minifloat(c, 4, 3, 7);
}
__device__ __forceinline__ float dec_ue8m0(uint32_t c) {
    c &= 0xFF;
    if (c == 0xFF) return __uint_as_float(0x7FC00000u);
    return c == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(c << 23);
}

template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                               const float* __restrict__ g, float* __restrict__ out, int64_t R, int64_t K,
                               uint32_t* __restrict__ err) {
    const float gg = g ? __ldg(g) : 1.0f;
    const int64_t blk = FMT == kNvfp4 ? 16 : 32;
    const int64_t cpd4 = pad_to(K / blk, 4) / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < R * K; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K, k = i % K;
        [[maybe_unused]] constexpr int64_t kRowNum = FMT == kNvfp4 ? 2 : FMT == kE4M3 ? 4 : 3;   // code bytes per 4 values
        [[maybe_unused]] const int64_t cbyte = FMT == kNvfp4 ? 4 * (r * (K / 8) + k / 8) : FMT == kE4M3 ? r * K + k
                                                                          : r * (3 * K / 4) + 3 * (k / 4);
        if (!BSQ_IN_BUFFER(err, kChkDequantIn, swz_offset(r, k / blk, cpd4), 1, pad_to(R, 128) * 4 * cpd4) ||
            !BSQ_IN_BUFFER(err, kChkDequantIn, cbyte, FMT == kNvfp4 ? 4 : FMT == kE4M3 ? 1 : 3, R * (kRowNum * K / 4)) ||
            !BSQ_IN_BUFFER(err, kChkDequantOut, i, 1, R * K))
            continue;
        const uint32_t sc = scales[swz_offset(r, k / blk, cpd4)];
        float v, s;
        if constexpr (FMT == kNvfp4) {
            const uint32_t w = reinterpret_cast<const uint32_t*>(codes)[r * (K / 8) + k / 8];
            v = dec_e2m1(w >> (4 * (k % 8)));
            s = (sc & 0x80) ? __uint_as_float(0x7FC00000u) : dec_e4m3(sc);
        } else if constexpr (FMT == kE4M3) {
            v = dec_e4m3(codes[r * K + k]);
            s = dec_ue8m0(sc);
        } else {
            const uint8_t* p = codes + r * (3 * K / 4) + 3 * (k / 4);
            const uint32_t bits = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
            const uint32_t c = (bits >> (6 * (k % 4))) & 0x3F;
            v = FMT == kE3M2 ? dec_e3m2(c) : dec_e2m3(c);
            s = dec_ue8m0(sc);
        }
        out[i] = __fmul_rn(__fmul_rn(v, s), gg);
    }
}

}  // namespace

bsq_status dequant_launch(const void* codes, int fmt, const uint8_t* scales, const float* g, float* out,
                          int64_t R, int64_t K, bool nvfp4, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const uint8_t* c = static_cast<const uint8_t*>(codes);
    int64_t blocks = (R * K + 255) / 256;
    const int64_t cap = (int64_t)info->num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (nvfp4) dequant_kernel<kNvfp4><<<(unsigned)blocks, 256, 0, s>>>(c, scales, g, out, R, K, info->err);
    else if (fmt == kE3M2) dequant_kernel<kE3M2><<<(unsigned)blocks, 256, 0, s>>>(c, scales, g, out, R, K, info->err);
    else if (fmt == kE2M3) dequant_kernel<kE2M3><<<(unsigned)blocks, 256, 0, s>>>(c, scales, g, out, R, K, info->err);
    else dequant_kernel<kE4M3><<<(unsigned)blocks, 256, 0, s>>>(c, scales, g, out, R, K, info->err);
    count_launch(BSQ_KERNEL_DEQUANT);
    return launch_status();
}

}  // namespace bsq
