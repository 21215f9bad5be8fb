// gemv.cu -- the decode product y[m, n] = gW * sum_k x[m, k] * W[n, k] for
// 1 <= M <= 32 bf16 activation rows against a packed weight streamed from HBM
// (cubecl-tile tests/tile/packed.rs, packed_one_row_product: the decode step's
// one-row product, N spread across CTAs, the accumulator held in registers
// for the whole K walk and drained once).
//
// Design (sm_103a):
//  * A CTA owns 128 weight rows (8 warps x 16 rows) and walks all of K.
//  * The weight is dequantized in registers, never staged: each thread loads
//    its rows' packed bytes straight from global memory (16-byte loads,
//    prefetched a 256-element chunk ahead) and turns them into bf16 pairs.
//  * Products run on the tensor cores as mma.sync m16n8k16 bf16 -> f32, weight
//    rows as the A operand (16 rows), activation rows as B (8 per n-tile).
//  * Exact decode: a code's bits are "placed" into a bf16 (its exponent and
//    mantissa fields dropped into the low bf16 fields and its sign into the
//    sign bit), which is the code's value times a fixed power of two (bf16
//    subnormals included).  One bf16x2 multiply by (block scale * 2^c) then
//    yields value*scale*2^c' exactly: every e2m1*ue4m3 and fp6*2^k product
//    fits bf16's 8-bit significand.  The fixed power is undone in fp32 at the
//    end.  No rounding happens before the tensor-core accumulate.
//  * K inside a 32-element thread range is permuted consistently for both
//    operands (pairs (j, j+4) of each 8-code group share a bf16x2 register);
//    the activation chunk is staged in shared memory in that order with a
//    bank-conflict-free layout.
#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kThreads = 256;            // 8 warps
constexpr int kRowsPerCta = 128;         // 16 rows per warp
constexpr int kChunk = 256;              // K elements staged per step (2 sub-chunks of 128)
constexpr int kPitch = kChunk / 8 + 4;   // 16-byte units per staged x row (== 4 mod 8)

template <int WFMT>
struct WTraits;
// nvfp4: 4-bit codes, 16 per block, 32 codes of a thread = 16 bytes.
template <>
struct WTraits<kNvfp4> { static constexpr int kRegs = 4; static constexpr int kBlock = 16; };
template <>
struct WTraits<kE3M2> { static constexpr int kRegs = 6; static constexpr int kBlock = 32; };
template <>
struct WTraits<kE2M3> { static constexpr int kRegs = 6; static constexpr int kBlock = 32; };
template <>
struct WTraits<kE4M3> { static constexpr int kRegs = 8; static constexpr int kBlock = 32; };

// Raw packed bytes of one thread's 32-code range of one row, plus its scales.
template <int WFMT>
struct RowRaw {
    uint32_t w[WTraits<WFMT>::kRegs];
    uint32_t s;   // nvfp4: two ue4m3 bytes (blocks 2t', 2t'+1); MX: one UE8M0 byte
};

template <int WFMT>
__device__ __forceinline__ void load_row(RowRaw<WFMT>& rr, const uint8_t* __restrict__ W, const uint8_t* __restrict__ sW,
                                         int64_t row, int64_t k, bool valid, int64_t K, int64_t cpd4) {
    if (!valid) {
#pragma unroll
        for (int i = 0; i < WTraits<WFMT>::kRegs; ++i) rr.w[i] = 0;
        rr.s = 0;
        return;
    }
    if constexpr (WFMT == kNvfp4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(W + row * (K / 2) + k / 2));
        rr.w[0] = v.x; rr.w[1] = v.y; rr.w[2] = v.z; rr.w[3] = v.w;
        rr.s = __ldg(reinterpret_cast<const uint16_t*>(sW + swz_offset(row, k / 16, cpd4)));
    } else if constexpr (WFMT == kE4M3) {
        const uint4* p = reinterpret_cast<const uint4*>(W + row * K + k);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        rr.w[0] = a.x; rr.w[1] = a.y; rr.w[2] = a.z; rr.w[3] = a.w;
        rr.w[4] = b.x; rr.w[5] = b.y; rr.w[6] = b.z; rr.w[7] = b.w;
        rr.s = __ldg(sW + swz_offset(row, k / 32, cpd4));
    } else {
        const uint2* p = reinterpret_cast<const uint2*>(W + row * (3 * K / 4) + (3 * k) / 4);
        const uint2 a = __ldg(p), b = __ldg(p + 1), c = __ldg(p + 2);
        rr.w[0] = a.x; rr.w[1] = a.y; rr.w[2] = b.x; rr.w[3] = b.y; rr.w[4] = c.x; rr.w[5] = c.y;
        rr.s = __ldg(sW + swz_offset(row, k / 32, cpd4));
    }
}

// Four fp6 codes of a 24-bit little-endian lane -> four byte containers.
__device__ __forceinline__ uint32_t fp6_to_containers(uint32_t bits24) {
    return (bits24 & 0x3Fu) | ((bits24 << 2) & 0x3F00u) | ((bits24 << 4) & 0x3F0000u) | ((bits24 << 6) & 0x3F000000u);
}

// Place two codes (code A in bits 0..7 of u, code B in bits 16..23) into a
// bf16x2: value(code) * 2^-P with P = 126 (e2m1, e2m3), 124 (e3m2), 120 (e4m3).
template <int WFMT>
__device__ __forceinline__ uint32_t place_pair(uint32_t u) {
    if constexpr (WFMT == kNvfp4) return ((u << 6) & 0x01C001C0u) | ((u << 12) & 0x80008000u);
    else if constexpr (WFMT == kE3M2) return ((u << 5) & 0x03E003E0u) | ((u << 10) & 0x80008000u);
    else if constexpr (WFMT == kE2M3) return ((u << 4) & 0x01F001F0u) | ((u << 10) & 0x80008000u);
    else return ((u << 4) & 0x07F007F0u) | ((u << 8) & 0x80008000u);
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// bf16x2 scale multiplier for one block: nvfp4 -> s * 2^119 (so the product is
// value*s*2^-7); MX -> 2^(ue-11) (product value*2^(ue-127)*2^(116-P)).
template <int WFMT>
__device__ __forceinline__ uint32_t scale_mult(uint32_t code) {
    uint32_t b;
    if constexpr (WFMT == kNvfp4) {
        const float f = __fmul_rn(e4m3_to_f32(code & 0xFF), 0x1p119f);
        b = f32_to_bf16_bits(f);   // exact: at most 4 significant bits
    } else {
        b = ((code & 0xFF) + 116u) << 7;
    }
    return b | (b << 16);
}

// The weight operand of one thread for one 128-element sub-chunk of one row:
// P[q][j] holds codes (8q+j, 8q+j+4) of its 32-code range, scaled.
template <int WFMT>
__device__ __forceinline__ void decode_row(const RowRaw<WFMT>& rr, uint32_t (&P)[4][4]) {
    if constexpr (WFMT == kNvfp4) {
        const uint32_t s0 = scale_mult<kNvfp4>(rr.s & 0xFF), s1 = scale_mult<kNvfp4>(rr.s >> 8);
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) P[q][j] = bmul2(place_pair<kNvfp4>(rr.w[q] >> (4 * j)), q < 2 ? s0 : s1);
    } else {
        const uint32_t sm = scale_mult<WFMT>(rr.s);
        uint32_t C[8];   // byte containers of the 32 codes, 4 per word
        if constexpr (WFMT == kE4M3) {
#pragma unroll
            for (int i = 0; i < 8; ++i) C[i] = rr.w[i];
        } else {
            // 24 bytes = 8 lanes of 3 bytes; w[] holds them little-endian.
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int byte = 3 * g, wi = byte >> 2, sh = (byte & 3) * 8;
                uint32_t bits = rr.w[wi] >> sh;
                if (sh > 8) bits |= rr.w[wi + 1] << (32 - sh);
                C[g] = fp6_to_containers(bits & 0xFFFFFFu);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t u = __byte_perm(C[2 * q], C[2 * q + 1], (uint32_t)(j | ((4 + j) << 8)));
                P[q][j] = bmul2(place_pair<WFMT>(u), sm);
            }
    }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NT, int WFMT>
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ W, const uint8_t* __restrict__ sW,
            const float* __restrict__ gW, void* __restrict__ y, int out_bf16, int64_t M, int64_t N, int64_t K) {
    constexpr int kRowsX = 8 * NT;
    __shared__ __align__(16) uint4 xs[2][kRowsX * kPitch];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta + warp * 16 + g;
    const int64_t row1 = row0 + 8;
    const int64_t cpd4 = pad_to(K / WTraits<WFMT>::kBlock, 4) / 4;
    const int64_t nck = (K + kChunk - 1) / kChunk;

    // ---- activation staging: 16-byte group u of row r of a chunk ----
    auto stage_load = [&](int64_t ck, uint4 (&xr)[NT]) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int idx = threadIdx.x + i * kThreads;     // < kRowsX * 32
            const int r = idx >> 5, u = idx & 31;
            const int64_t k = ck * kChunk + u * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < M && k < K) v = __ldg(reinterpret_cast<const uint4*>(x + r * K + k));
            // [x0..x7] -> [(x0,x4), (x1,x5), (x2,x6), (x3,x7)]
            xr[i] = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                               __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
        }
    };
    auto stage_store = [&](int buf, const uint4 (&xr)[NT]) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int idx = threadIdx.x + i * kThreads;
            const int r = idx >> 5, u = idx & 31;
            const int h = u >> 4, tt = (u >> 2) & 3, q = u & 3;
            xs[buf][r * kPitch + 16 * h + 4 * q + tt] = xr[i];
        }
    };
    auto load_w = [&](int64_t ck, RowRaw<WFMT> (&rr)[2][2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t k = ck * kChunk + 128 * h + 32 * t;
            const bool kv = ck < nck && k < K;
            load_row<WFMT>(rr[h][0], W, sW, row0, k, kv && row0 < N, K, cpd4);
            load_row<WFMT>(rr[h][1], W, sW, row1, k, kv && row1 < N, K, cpd4);
        }
    };

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    RowRaw<WFMT> wcur[2][2], wnext[2][2];
    {
        uint4 xr[NT];
        stage_load(0, xr);
        stage_store(0, xr);
        load_w(0, wcur);
    }
    __syncthreads();

    for (int64_t ck = 0; ck < nck; ++ck) {
        const int buf = (int)(ck & 1);
        uint4 xr[NT];
        if (ck + 1 < nck) stage_load(ck + 1, xr);
        load_w(ck + 1, wnext);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t P0[4][4], P1[4][4];
            decode_row<WFMT>(wcur[h][0], P0);
            decode_row<WFMT>(wcur[h][1], P1);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 xb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xb[nt] = xs[buf][(8 * nt + g) * kPitch + 16 * h + 4 * q + t];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int j0 = 2 * half;
                    const uint32_t a[4] = {P0[q][j0], P1[q][j0], P0[q][j0 + 1], P1[q][j0 + 1]};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint32_t b0 = half ? xb[nt].z : xb[nt].x;
                        const uint32_t b1 = half ? xb[nt].w : xb[nt].y;
                        mma_bf16(acc[nt], a, b0, b1);
                    }
                }
            }
        }
        if (ck + 1 < nck) stage_store(buf ^ 1, xr);
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) { wcur[h][0] = wnext[h][0]; wcur[h][1] = wnext[h][1]; }
    }

    // ---- epilogue: undo the fixed power of two, apply gW, store y[m, n] ----
    constexpr float kLift = WFMT == kNvfp4 ? 0x1p7f : WFMT == kE3M2 ? 0x1p8f : WFMT == kE2M3 ? 0x1p10f : 0x1p4f;
    const float f = __fmul_rn(kLift, gW ? __ldg(gW) : 1.0f);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = 8 * nt + 2 * t + (i & 1);
            const int64_t n = (i < 2) ? row0 : row1;
            if (m < M && n < N) {
                const float v = __fmul_rn(acc[nt][i], f);
                if (out_bf16) reinterpret_cast<uint16_t*>(y)[m * N + n] = f32_to_bf16_bits(v);
                else reinterpret_cast<float*>(y)[m * N + n] = v;
            }
        }
    }
}

template <int WFMT>
bsq_status launch_fmt(const uint16_t* x, const uint8_t* W, const uint8_t* sW, const float* gW, void* y, int out,
                      int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    const dim3 grid((unsigned)((N + kRowsPerCta - 1) / kRowsPerCta));
    if (M <= 8) gemv_kernel<1, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K);
    else if (M <= 16) gemv_kernel<2, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K);
    else gemv_kernel<4, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K);
    return launch_status();
}

}  // namespace

bsq_status gemv_launch(const uint16_t* x, const void* W, int fw, const uint8_t* sW, const float* gW, void* y,
                       int out, int64_t M, int64_t N, int64_t K, bool nvfp4, cudaStream_t s) {
    bsq_status st;
    if (!device_info(&st)) return st;
    const uint8_t* Wb = static_cast<const uint8_t*>(W);
    bsq_status r;
    if (nvfp4) {
        r = launch_fmt<kNvfp4>(x, Wb, sW, gW, y, out, M, N, K, s);
        count_launch(BSQ_KERNEL_GEMV_NVFP4);
    } else {
        if (fw == kE3M2) r = launch_fmt<kE3M2>(x, Wb, sW, gW, y, out, M, N, K, s);
        else if (fw == kE2M3) r = launch_fmt<kE2M3>(x, Wb, sW, gW, y, out, M, N, K, s);
        else r = launch_fmt<kE4M3>(x, Wb, sW, gW, y, out, M, N, K, s);
        count_launch(BSQ_KERNEL_GEMV_MX);
    }
    return r;
}

}  // namespace bsq
