// gemv.cu -- the decode product y[m, n] = gW * sum_k x[m, k] * W[n, k] for
// 1 <= M <= 32 bf16 activation rows against a packed weight streamed from HBM
// (cubecl-tile tests/tile/packed.rs, packed_one_row_product: the decode step's
// one-row product, N spread across CTAs, the accumulator held in registers
// for the whole K walk and drained once).
//
// Two kernels (sm_103a):
//  * nvfp4 (gemv_nvf4_kernel, gemv_nvf4_res_kernel, below): the weight
//    streams through a TMA ring in shared memory and is decoded with the
//    hardware e2m1 -> f16 conversion; see the comment at its namespace.
//  * MX formats (gemv_kernel, here): a CTA owns 128 weight rows (8 warps x 16
//    rows) and walks all of K; the weight is dequantized in registers, never
//    staged: each thread loads its rows' packed bytes straight from global
//    memory (prefetched a 256-element chunk ahead) and turns them into bf16
//    pairs.  Products run on the tensor cores as mma.sync m16n8k16 bf16 -> f32,
//    weight rows as the A operand (16 rows), activation rows as B (8 per
//    n-tile).
//  * Exact decode ("placed" bf16): a code's bits are dropped into the low
//    bf16 exponent/mantissa fields and its sign into the sign bit, which is
//    the code's value times a fixed power of two (bf16 subnormals included);
//    one bf16x2 multiply by a constant power of two makes it the code's value
//    (at most 4 significant bits: exact).  No rounding happens before the
//    tensor-core accumulate.
//  * MX block scales are applied in fp32 to per-block partial sums: the two
//    MMAs of a K slice cover exactly one 32-code block (each thread of a quad
//    holds 8 of its codes), so any UE8M0 byte scales its block exactly.
#include <climits>
#include <mutex>
#include <type_traits>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kThreads = 256;            // 8 warps
constexpr int kRowsPerCta = 128;         // 16 rows per warp
constexpr int kChunk = 256;              // K elements staged per step (2 sub-chunks of 128)
constexpr int kPitch = kChunk / 8 + 4;   // 16-byte units per staged x row (== 4 mod 8)

// y[i] (i = m N + n, `size` = M N) in the output type: bf16 bits or f32.
__device__ __forceinline__ void store_y(void* y, int out_bf16, int64_t i, float v, uint32_t* err, int64_t size) {
    if (!BSQ_IN_BUFFER(err, kChkGemvY, i, 1, size)) return;
    if (out_bf16) reinterpret_cast<uint16_t*>(y)[i] = f32_to_bf16_bits(v);
    else reinterpret_cast<float*>(y)[i] = v;
}

// Raw packed bytes of one thread's share of one row's 128-element sub-chunk:
// codes 8t..8t+7 of each of the sub-chunk's four MX blocks (thread t of the
// quad), plus the four blocks' UE8M0 bytes.
template <int WFMT>
struct RowRaw {
    uint32_t w[8];   // block b: w[2b] codes 0..3 of the thread's eight, w[2b+1] codes 4..7 (packed bits)
    uint32_t s;      // the sub-chunk's four UE8M0 bytes, block b in byte b
};

template <int WFMT>
__device__ __forceinline__ void load_row(RowRaw<WFMT>& rr, const uint8_t* __restrict__ W, const uint8_t* __restrict__ sW,
                                         int64_t row, int64_t k, int t, bool valid, int64_t N, int64_t K, int64_t cpd4,
                                         uint32_t* err) {
    [[maybe_unused]] constexpr int64_t kRowNum = WFMT == kE4M3 ? 4 : 3;   // row bytes = kRowNum K / 4
    valid = valid && BSQ_IN_BUFFER(err, kChkGemvW, row * (kRowNum * K / 4) + (kRowNum * k) / 4,
                                   kRowNum * 32, N * (kRowNum * K / 4)) &&
            BSQ_IN_BUFFER(err, kChkGemvScales, swz_offset(row, k / 32, cpd4), 4, pad_to(N, 128) * 4 * cpd4);
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i) rr.w[i] = 0;
        rr.s = 0;
        return;
    }
    if constexpr (WFMT == kE4M3) {
        // block b's codes 8t..8t+7: bytes 32b + 8t .. +8 of the sub-chunk
        const uint8_t* base = W + row * K + k + 8 * t;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(base + 32 * b));
            rr.w[2 * b] = v.x;
            rr.w[2 * b + 1] = v.y;
        }
    } else {
        // block b's codes 8t..8t+7: 6 bytes at 24b + 6t, read as the two aligned
        // words that hold them (rows of 3K/4 bytes, K % 128 == 0: 4-byte aligned)
        const uint8_t* rowp = W + row * (3 * K / 4) + (3 * k) / 4;
        const int off = 6 * t;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowp + 24 * b + (off & ~3));
            const uint32_t lo = __ldg(wp), hi = __ldg(wp + 1);
            const uint32_t b0 = (off & 2) ? __funnelshift_r(lo, hi, 16) : lo;     // bits 0..31 of the 48
            const uint32_t b1 = (off & 2) ? (hi >> 16) : (hi & 0xFFFFu);         // bits 32..47
            rr.w[2 * b] = b0 & 0xFFFFFFu;                                         // codes 0..3
            rr.w[2 * b + 1] = (b0 >> 24) | (b1 << 8);                             // codes 4..7
        }
    }
    // the four blocks' scale bytes are consecutive in the swizzled buffer
    rr.s = __ldg(reinterpret_cast<const uint32_t*>(sW + swz_offset(row, k / 32, cpd4)));
}

// Four fp6 codes of a 24-bit little-endian lane -> four byte containers.
__device__ __forceinline__ uint32_t fp6_to_containers(uint32_t bits24) {
    return (bits24 & 0x3Fu) | ((bits24 << 2) & 0x3F00u) | ((bits24 << 4) & 0x3F0000u) | ((bits24 << 6) & 0x3F000000u);
}

// Place two codes (code A in bits 0..7 of u, code B in bits 16..23) into a
// bf16x2: value(code) * 2^-P with P = 126 (e2m3), 124 (e3m2), 120 (e4m3).
template <int WFMT>
__device__ __forceinline__ uint32_t place_pair(uint32_t u) {
    if constexpr (WFMT == kE3M2) return ((u << 5) & 0x03E003E0u) | ((u << 10) & 0x80008000u);
    else if constexpr (WFMT == kE2M3) return ((u << 4) & 0x01F001F0u) | ((u << 10) & 0x80008000u);
    else return ((u << 4) & 0x07F007F0u) | ((u << 8) & 0x80008000u);
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 2^P in both bf16 halves: a placed code times this is the code's value
// (an exact bf16: at most 4 significant bits, inside the normal range).
template <int WFMT>
__device__ __forceinline__ constexpr uint32_t unplace_mult() {
    constexpr uint32_t p = WFMT == kE3M2 ? 124u : WFMT == kE2M3 ? 126u : 120u;
    return ((p + 127u) << 7) | (((p + 127u) << 7) << 16);
}

// The UE8M0 byte's value 2^(ue-127) as an fp32, built from its bits (byte 0 is
// the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t ue) {
    return ue == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(ue << 23);
}

// One row's sub-chunk as MMA A-operand registers: V[b][j] holds codes
// (8t+2j, 8t+2j+1) of block b as exact bf16 values; sc[b] the block scale.
template <int WFMT>
__device__ __forceinline__ void decode_row(const RowRaw<WFMT>& rr, uint32_t (&V)[4][4], float (&sc)[4]) {
    constexpr uint32_t kUnplace = unplace_mult<WFMT>();
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t c0 = rr.w[2 * b], c1 = rr.w[2 * b + 1];     // byte containers of codes 0..3 / 4..7
        if constexpr (WFMT != kE4M3) {
            c0 = fp6_to_containers(c0);
            c1 = fp6_to_containers(c1);
        }
        V[b][0] = bmul2(place_pair<WFMT>(__byte_perm(c0, 0, 0x4140)), kUnplace);
        V[b][1] = bmul2(place_pair<WFMT>(__byte_perm(c0, 0, 0x4342)), kUnplace);
        V[b][2] = bmul2(place_pair<WFMT>(__byte_perm(c1, 0, 0x4140)), kUnplace);
        V[b][3] = bmul2(place_pair<WFMT>(__byte_perm(c1, 0, 0x4342)), kUnplace);
        sc[b] = ue8m0_value((rr.s >> (8 * b)) & 0xFFu);
    }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The MX kernel.  Each quad of a warp (rows g and g + 8) walks K in 128-element
// sub-chunks = four MX blocks; thread t holds codes 8t..8t+7 of every block, so
// the two m16n8k16 MMAs of a block (MMA s: K slots 2t, 2t+1 <- codes 8t+4s,
// +1; slots 2t+8, 2t+9 <- codes 8t+4s+2, +3) sum that block alone.  Each
// block's sum starts from zero and is added to the fp32 accumulator times the
// block's scale 2^(ue-127): every UE8M0 byte is applied exactly in fp32, and
// the operands are the codes' exact values.  x is staged in its natural order
// (16 bytes = x[8t .. 8t+8) of a block per thread and activation row).
template <int NT, int WFMT>
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ W, const uint8_t* __restrict__ sW,
            const float* __restrict__ gW, void* __restrict__ y, int out_bf16, int64_t M, int64_t N, int64_t K,
            uint32_t* __restrict__ err) {
    constexpr int kRowsX = 8 * NT;
    __shared__ __align__(16) uint4 xs[2][kRowsX * kPitch];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta + warp * 16 + g;
    const int64_t row1 = row0 + 8;
    const int64_t cpd4 = pad_to(K / 32, 4) / 4;
    const int64_t nck = (K + kChunk - 1) / kChunk;

    // ---- activation staging: 16-byte group u of row r of a chunk, natural order ----
    auto stage_load = [&](int64_t ck, uint4 (&xr)[NT]) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int idx = threadIdx.x + i * kThreads;     // < kRowsX * 32
            const int r = idx >> 5, u = idx & 31;
            const int64_t k = ck * kChunk + u * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < M && k < K && BSQ_IN_BUFFER(err, kChkGemvX, r * K + k, 8, M * K))
                v = __ldg(reinterpret_cast<const uint4*>(x + r * K + k));
            xr[i] = v;
        }
    };
    auto stage_store = [&](int buf, const uint4 (&xr)[NT]) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int idx = threadIdx.x + i * kThreads;
            xs[buf][(idx >> 5) * kPitch + (idx & 31)] = xr[i];
        }
    };
    auto load_w = [&](int64_t ck, RowRaw<WFMT> (&rr)[2][2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t k = ck * kChunk + 128 * h;
            const bool kv = ck < nck && k < K;
            load_row<WFMT>(rr[h][0], W, sW, row0, k, t, kv && row0 < N, N, K, cpd4, err);
            load_row<WFMT>(rr[h][1], W, sW, row1, k, t, kv && row1 < N, N, K, cpd4, err);
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
            uint32_t V0[4][4], V1[4][4];
            float s0[4], s1[4];
            decode_row<WFMT>(wcur[h][0], V0, s0);
            decode_row<WFMT>(wcur[h][1], V1, s1);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xb = xs[buf][(8 * nt + g) * kPitch + 16 * h + 4 * b + t];
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    const uint32_t a0[4] = {V0[b][0], V1[b][0], V0[b][1], V1[b][1]};
                    const uint32_t a1[4] = {V0[b][2], V1[b][2], V0[b][3], V1[b][3]};
                    mma_bf16(d, a0, xb.x, xb.y);
                    mma_bf16(d, a1, xb.z, xb.w);
                    acc[nt][0] = __fmaf_rn(d[0], s0[b], acc[nt][0]);
                    acc[nt][1] = __fmaf_rn(d[1], s0[b], acc[nt][1]);
                    acc[nt][2] = __fmaf_rn(d[2], s1[b], acc[nt][2]);
                    acc[nt][3] = __fmaf_rn(d[3], s1[b], acc[nt][3]);
                }
            }
        }
        if (ck + 1 < nck) stage_store(buf ^ 1, xr);
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) { wcur[h][0] = wnext[h][0]; wcur[h][1] = wnext[h][1]; }
    }

    // ---- epilogue: apply gW, store y[m, n] ----
    const float f = gW ? __ldg(gW) : 1.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = 8 * nt + 2 * t + (i & 1);
            const int64_t n = (i < 2) ? row0 : row1;
            if (m < M && n < N) store_y(y, out_bf16, m * N + n, __fmul_rn(acc[nt][i], f), err, M * N);
        }
    }
}

// ------------------------------------------------------------- nvfp4 ----
// The nvfp4 decode GEMV.  Weight bytes stream HBM -> shared memory through a
// TMA ring (the bytes in flight per SM, not the instruction count, bound a
// decode GEMV), so the SM's load window is the ring, not registers.
//
//  * CTA = CW consumer warps x 16 weight rows + one producer warp.  R = 16 CW
//    rows per CTA, chosen on the host so the CTAs fill the SMs in whole waves.
//  * Stage = 256 codes of every row: a 2-D TMA box {128 B, R rows} with the
//    128-byte swizzle, plus the block-scale atoms of those 16 blocks (one bulk
//    copy of up to 4 atoms per 128-row block the tile touches).
//  * Consumers read their 16 rows with ldmatrix (eight rows x 16 B per matrix;
//    the swizzle puts the eight rows' chunks in eight bank groups), so thread
//    (g, t) holds codes 8t..8t+7 of a 32-code chunk for rows g and g+8.
//  * x is staged per stage by the consumer threads (loaded two stages ahead
//    into registers), natural K order, row pitch 36 x 16 B.
//
// Exact decode, two ways, chosen per stage (uniform in the CTA):
//  * f16: when every activation of the stage is zero or an f16 normal, x is
//    staged as f16 and each code pair (one byte, two e2m1 codes) goes through
//    the hardware e2m1x2 -> f16x2 conversion and one f16x2 multiply by the
//    block scale (ue4m3 -> f16, exact).  value * scale lies in [2^-10, 2688]
//    with at most 5 significant bits: exact, an f16 normal; x * w is then exact
//    in the f32 MMA accumulate.
//  * bf16 (any other stage): x is staged as raw bf16 and the codes are
//    "placed" into bf16 (value * 2^-126) and multiplied by scale * 2^119 in
//    bf16x2, exact; those products carry 2^-7, so they accumulate separately
//    and are lifted by 2^7 at the end.
namespace nvf4 {

constexpr int kMaxRowBlocks = 3;    // 128-row scale blocks one tile can touch (R <= 256)
constexpr int kSmemLimit = 232448;  // opt-in shared memory per CTA

// the four code pairs (bytes) of a word -> four f16x2
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "  mov.b32 {b0, b1, b2, b3}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, b0;\n  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "  cvt.rn.f16x2.e2m1x2 %2, b2;\n  cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// codes (2j, 2j+1) of one byte placed into a bf16x2: value * 2^-126 each
__device__ __forceinline__ uint32_t place_byte_bf16x2(uint32_t b) {
    return ((b & 7u) << 6) | ((b & 8u) << 12) | ((b & 0x70u) << 18) | ((b & 0x80u) << 24);
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// AND of `ok` over the nthreads threads that meet at named barrier `id`.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool ok) {
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 q, %1, 0; barrier.red.and.pred p, %2, %3, q; selp.u32 %0, 1, 0, p; }"
                 : "=r"(r) : "r"((uint32_t)ok), "r"(id), "r"(nthreads) : "memory");
    return r != 0;
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Bits 15 and 31 are set when the low / high bf16 half of w is exactly an f16
// value: zero, or exponent field 110..142 (the f16 normals, and the f16
// subnormals on which a bf16 value's 8 significant bits land exactly: values
// of at least 2^-17).  Both halves are tested at once, a guard bit in each
// sign position keeping borrows from crossing into the other half: for a
// half's 15 magnitude bits m, (0x8000 + m) - 1 keeps bit 15 iff m != 0,
// - (110 << 7) iff m >= 110 << 7, - (143 << 7) iff m >= 143 << 7.  AND the
// results over many words and test once with f16_exact.
__device__ __forceinline__ uint32_t f16_exact_bits(uint32_t w) {
    const uint32_t a = w | 0x80008000u;
    return ~(a - 0x00010001u) | ((a - 0x37003700u) & ~(a - 0x47804780u));
}
__device__ __forceinline__ bool f16_exact(uint32_t bits) { return (bits & 0x80008000u) == 0x80008000u; }
__device__ __forceinline__ uint32_t f16_exact_bits4(const uint4& v) {
    return f16_exact_bits(v.x) & f16_exact_bits(v.y) & f16_exact_bits(v.z) & f16_exact_bits(v.w);
}
// bf16x2 -> f16x2, round to nearest (exact whenever f16_exact holds)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
    return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}

// A stage's scale atoms of n_rb consecutive 128-row tiles from rb0: one load of
// a 2-tile box per pair of tiles, a 1-tile box for an odd remainder, into
// [tile][atom][512 B] at dst; tiles past the weight's rows and atoms past K
// read as zeros (the maps are {128 words, atoms, tiles} of the scale buffer).
__device__ __forceinline__ void load_scale_tiles(uint32_t dst, const CUtensorMap* tmS2, const CUtensorMap* tmS1,
                                                 uint32_t bar, int i, int rb0, int n_rb) {
    int j = 0;
    for (; j + 2 <= n_rb; j += 2) tma_load_3d(dst + (uint32_t)j * 2048u, tmS2, bar, 0, 4 * i, rb0 + j);
    if (j < n_rb) tma_load_3d(dst + (uint32_t)j * 2048u, tmS1, bar, 0, 4 * i, rb0 + j);
}
// Programmatic dependent launch: the prologue above overlaps the previous
// kernel; nothing that kernel writes is read before this wait.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct Args {
    const uint16_t* x;
    const uint8_t* sW;
    const float* gW;
    void* y;
    uint32_t* err;
    int64_t M, N, K;
    int64_t cpd4;        // scale atoms per 128-row block
    int out_bf16;
};

// Shared memory plan: ring stages (codes, x, scale atoms), barriers and the
// per-stage x flags; as many stages as fit, at most 8.  A stage's x is four
// {64 values, 8 NT rows} boxes with the 128-byte swizzle (rows >= M and
// values past K read as zeros).
template <int NT, int CW>
struct Plan {
    static constexpr int kXBox = 8 * NT * 128;                      // one {64, 8 NT} bf16 box
    static constexpr int kWBytes = 16 * CW * 128;
    static constexpr int kSBytes = kMaxRowBlocks * 2048;
    static constexpr int kStageBytes = kWBytes + 4 * kXBox + kSBytes;   // codes first: 1024-aligned
    static constexpr int kFixed = 1024 + 512;
    static constexpr int kFit = (kSmemLimit - kFixed) / kStageBytes;
    static constexpr int kStages = kFit < 8 ? kFit : 8;
    static constexpr int kBytes = kFixed + kStages * kStageBytes;
    static_assert(kStages >= 3, "too little shared memory for the ring");
    static_assert(kWBytes % 1024 == 0 && kXBox % 1024 == 0, "128-byte-swizzled boxes start 1024-aligned");
    static_assert((3 * kStages + 1) * 8 + kStages * 4 <= 512, "barrier area");
};

// Staged kernel (M >= 3, or M <= 2 when x does not fit beside the resident
// kernel's ring).  Per stage the producer warp loads the codes, the scale
// atoms and x (four 2-D boxes of 8 NT rows); four dedicated x warps check the
// stage's x (is every value zero or exact in f16?  one AND over the x warps),
// convert it in place to f16 when it is, record the choice in a per-stage flag
// and release the stage to the consumers with an mbarrier.  The consumer warps
// so never stage x themselves nor wait for one another: each walks the ring at
// its own pace.  (A single x warp per CTA fell behind the consumers.)
constexpr int kXWarps = 4;

template <int NT, int CW>
__global__ void __launch_bounds__((CW + 1 + kXWarps) * 32, 1)
gemv_nvf4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS2,
                 const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmX, const Args args) {
    using P = Plan<NT, CW>;
    constexpr int R = 16 * CW;
    constexpr int kStages = P::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // stage s: codes at s * kStageBytes, x boxes after them, then the scale atoms
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * P::kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* xready = empty + kStages;                      // [kStages]: x checked (and converted)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xready + kStages);
    uint32_t* xflag = reinterpret_cast<uint32_t*>(xready + kStages + 1);   // [kStages]: 1 = x is f16

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t row_base = (int64_t)blockIdx.x * R;
    const int nst = (int)((K + 255) / 256);
    const int rb0 = (int)(row_base >> 7);
    const int rb1 = (int)((row_base + R - 1) >> 7);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), CW);
            mbar_init(smem_u32(xready + s), kXWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait_then_release();

    if (warp == CW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmS2);
            prefetch_tmap(&tmS1);
            prefetch_tmap(&tmX);
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(smem_u32(empty + s), ((i / kStages) - 1) & 1, args.err, abort_flag, kErrGemvProducer))
                    break;
                uint8_t* st = smem + s * P::kStageBytes;
                const int n_rb = rb1 - rb0 + 1;
                const uint32_t fb = smem_u32(full + s);
                mbar_arrive_expect_tx(fb, P::kWBytes + 4 * P::kXBox + (uint32_t)n_rb * 2048u);
                tma_load_2d(smem_u32(st), &tmW, fb, i * 128, (int32_t)row_base);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_2d(smem_u32(st + P::kWBytes + b * P::kXBox), &tmX, fb, i * 256 + 64 * b, 0);
                load_scale_tiles(smem_u32(st + P::kWBytes + 4 * P::kXBox), &tmS2, &tmS1, fb, i, rb0, n_rb);
                issued = i + 1;
            }
            if (*abort_flag) {
                // leave no copy in flight into this CTA's shared memory
                for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(full + i % kStages), (i / kStages) & 1) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        return;
    }

    if (warp > CW) {
        // ---------------- x warps ----------------
        // A stage's x is 4 boxes x 8 NT rows x 8 slots of 16 bytes; x warp j takes
        // slots [j kPer * 32, (j + 1) kPer * 32), kPer per lane.
        constexpr int kXW = kXWarps;
        constexpr int kPer = 256 * NT / (32 * kXW);
        const int j = warp - CW - 1;
        for (int i = 0; i < nst; ++i) {
            const int s = i % kStages;
            uint8_t* xs = smem + s * P::kStageBytes + P::kWBytes;
            const bool have = mbar_wait(smem_u32(full + s), (i / kStages) & 1, args.err, abort_flag, kErrGemvConsumer);
            // slot u: byte offset 16 u within the stage's four boxes (the check and the
            // conversion are per value, so the swizzled order is immaterial)
            uint4 h[kPer];
            uint32_t okb = ~0u;
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int u = 32 * (j * kPer + q) + lane;
                const uint4 v = have ? *reinterpret_cast<const uint4*>(xs + 16 * u) : make_uint4(0, 0, 0, 0);
                okb &= f16_exact_bits4(v);
                h[q] = bf16x8_to_f16x8(v);
            }
            const bool f16 = bar_and(1, 32 * kXW, f16_exact(okb));
            if (have && f16) {
#pragma unroll
                for (int q = 0; q < kPer; ++q) *reinterpret_cast<uint4*>(xs + 16 * (32 * (j * kPer + q) + lane)) = h[q];
            }
            // the slot is refilled by TMA (the async proxy) after the consumers release it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                if (j == 0) xflag[s] = f16 ? 1u : 0u;
                mbar_arrive(smem_u32(xready + s));
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, t = lane & 3;
    const int64_t row0 = row_base + warp * 16 + g, row1 = row0 + 8;
    const int nblocks32 = (int)(K / 16);     // K < 2^31: the entry point bounds every dimension

    float acc_h[NT][4], acc_b[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc_h[i][j] = acc_b[i][j] = 0.0f;

    // ldmatrix addresses: lane L supplies row (L & 7) of matrix L >> 3:
    // matrices {rows 0-7, chunk c}, {rows 8-15, c}, {rows 0-7, c+1}, {rows 8-15, c+1}
    const int mrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);   // row within the tile
    const int mcol = lane >> 4;                                        // 0: chunk c, 1: chunk c+1
    // scale word of rows g, g+8 (chunk pair c, c+1 share one 4-byte group)
    int soff[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int64_t row = r ? row1 : row0;
        soff[r] = (int)((row >> 7) - rb0) * 2048 + (int)(row & 31) * 16 + (int)((row >> 5) & 3) * 4;
    }
    const uint32_t ssel = (t >> 1) ? 0x31u : 0x20u;   // bytes (t>>1) and 2 + (t>>1) of the group

    // one stage of MMAs: chunk pairs (c, c+1) = (2cp, 2cp+1), each one
    // ldmatrix.x4 of codes (rows g, g+8 x chunks c, c+1) and one 4-byte scale
    // group per row.  F16 selects the decode (and the accumulator set).
    auto consume = [&](auto f16_tag, auto tail_tag, uint32_t wst, uint32_t sst, uint32_t xs, int i,
                       float (&acc)[NT][4]) {
        constexpr bool F16 = decltype(f16_tag)::value;
        constexpr bool TAIL = decltype(tail_tag)::value;   // zero the multipliers of blocks past K
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
            uint32_t wr[4];
            ldmatrix_x4(wst + mrow * 128 + (((2 * cp + mcol) ^ (mrow & 7)) << 4), wr);
            uint32_t S[2][2];   // [row][chunk] pair multipliers
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t two = __byte_perm(lds32(sst + soff[r] + cp * 512), 0, ssel);
                if constexpr (F16) {
                    const uint32_t sf = e4m3x2_to_f16x2(two);
                    S[r][0] = __byte_perm(sf, sf, 0x1010);
                    S[r][1] = __byte_perm(sf, sf, 0x3232);
                } else {
                    const uint32_t b0 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32(two & 0xFF), 0x1p119f));
                    const uint32_t b1 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32((two >> 8) & 0xFF), 0x1p119f));
                    S[r][0] = b0 | (b0 << 16);
                    S[r][1] = b1 | (b1 << 16);
                }
                if constexpr (TAIL) {
                    const int blk0 = 16 * i + 4 * cp + (t >> 1);        // chunk 2cp; chunk 2cp+1 is blk0 + 2
                    if (blk0 >= nblocks32) S[r][0] = 0;
                    if (blk0 + 2 >= nblocks32) S[r][1] = 0;
                }
            }
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {               // chunk 2cp + ch
                uint32_t P2[2][4];   // pairs j = 0..3 of rows g (wr[2ch]) and g+8 (wr[2ch+1])
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if constexpr (F16) {
                        e2m1x8_to_f16x2(wr[2 * ch + r], P2[r]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) P2[r][j] = hmul2(P2[r][j], S[r][ch]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            P2[r][j] = bmul2(place_byte_bf16x2((wr[2 * ch + r] >> (8 * j)) & 0xFFu), S[r][ch]);
                    }
                }
                // x units 4 (2cp + ch) + t of rows 8 nt + g: box (2cp + ch) >> 1, piece
                // (4 (2cp + ch) + t) & 7, 128-byte swizzle by the row
                const int c = 4 * (2 * cp + ch) + t;
                uint4 xv[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    xv[nt] = lds128(xs + (uint32_t)((c >> 3) * P::kXBox + (8 * nt + g) * 128 + (((c & 7) ^ g) << 4)));
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t a[4] = {P2[0][2 * e], P2[1][2 * e], P2[0][2 * e + 1], P2[1][2 * e + 1]};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<F16>(acc[nt], a, e ? xv[nt].z : xv[nt].x, e ? xv[nt].w : xv[nt].y);
                }
            }
        }
    };

    for (int i = 0; i < nst; ++i) {
        const int s = i % kStages;
        const uint32_t par = (i / kStages) & 1;
        // xready orders the stage's codes and scales too: the x warps waited for `full`
        // before they arrived (after a failed wait they arrive with the abort flag set)
        const bool have = mbar_wait(smem_u32(xready + s), par, args.err, abort_flag, kErrGemvConsumer) && !*abort_flag;
        if (have) {
            const uint32_t wst = smem_u32(smem + s * P::kStageBytes);
            const uint32_t xs = wst + P::kWBytes;
            const uint32_t sst = xs + 4 * P::kXBox;
            const bool tail = 16 * (i + 1) > nblocks32;
            if (xflag[s]) {
                if (tail) consume(std::true_type{}, std::true_type{}, wst, sst, xs, i, acc_h);
                else consume(std::true_type{}, std::false_type{}, wst, sst, xs, i, acc_h);
            } else {
                if (tail) consume(std::false_type{}, std::true_type{}, wst, sst, xs, i, acc_b);
                else consume(std::false_type{}, std::false_type{}, wst, sst, xs, i, acc_b);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }

    // ---- epilogue: acc_h + 2^7 acc_b, times gW ----
    if (*abort_flag) return;
    const float gw = args.gW ? __ldg(args.gW) : 1.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = 8 * nt + 2 * t + (i & 1);
            const int64_t n = (i < 2) ? row0 : row1;
            if (m < M && n < N)
                store_y(args.y, args.out_bf16, m * N + n, __fmul_rn(__fmaf_rn(acc_b[nt][i], 0x1p7f, acc_h[nt][i]), gw),
                        args.err, M * N);
        }
    }
}

// Resident-x variant (small M, when M x K fits next to a 6-stage ring): x is
// checked once, staged once (f16 when every value is zero or an f16 normal,
// else raw bf16) and stays in shared memory for the whole K walk, so the
// stage loop has no x staging and no consumer-wide barrier.  The ring depth is
// whatever the rest of shared memory holds (6..8 stages).
//
// SLOT (M = 1, f16 path): the block scale leaves the decode.  With one
// activation row, seven of the MMA's eight B columns would be zero, so column j
// instead carries x only for the K positions of blocks b with b % 8 == j (the
// lane holding a column's fragment loads x or zero).  After every eight blocks
// the fp32 tile holds, per weight row, the eight block partial sums
// sum_k w[n, k] x[k] of unscaled e2m1 values; each is multiplied by its ue4m3
// scale (decoded exactly to fp32 from its bits) and added to the row's
// accumulators.  The per-pair f16 scale multiply and the per-chunk scale
// conversions drop out of the stage loop.
constexpr int kResMaxStages = 8;


// ue4m3 byte -> fp32, exact: its 7 bits placed as an fp32 exponent/mantissa
// (normal or subnormal) are the value times 2^-120.
__device__ __forceinline__ float ue4m3_bits_to_f32(uint32_t b) {
    return __fmul_rn(__uint_as_float((b & 0x7Fu) << 20), 0x1p120f);
}

template <int CW, bool SLOT>
__global__ void __launch_bounds__((CW + 1) * 32, 1)
gemv_nvf4_res_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS2,
                     const __grid_constant__ CUtensorMap tmS1, const Args args, int n_stages, uint32_t x_pitch) {
    constexpr int R = 16 * CW;
    constexpr int kCons = CW * 32;
    constexpr int kWBytes = R * 128;
    constexpr int kSBytes = kMaxRowBlocks * 2048;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int64_t M = args.M, N = args.N, K = args.K;
    uint8_t* sWst = smem;
    uint8_t* sSst = sWst + n_stages * kWBytes;
    uint8_t* sX = sSst + n_stages * kSBytes;                            // M rows x x_pitch bytes
    uint64_t* full = reinterpret_cast<uint64_t*>(sX + M * x_pitch);      // x_pitch % 16 == 0
    uint64_t* empty = full + kResMaxStages;
    uint64_t* xbar = empty + kResMaxStages;                              // x has landed in shared memory
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xbar + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row_base = (int64_t)blockIdx.x * R;
    const int nst = (int)((K + 255) / 256);
    const int rb0 = (int)(row_base >> 7);
    const int rb1 = (int)((row_base + R - 1) >> 7);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int st = 0; st < n_stages; ++st) {
            mbar_init(smem_u32(full + st), 1);
            mbar_init(smem_u32(empty + st), CW);
        }
        mbar_init(smem_u32(xbar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait_then_release();

    if (warp == CW) {
        // ---------------- producer (as in gemv_nvf4_kernel) ----------------
        if (lane == 0) {
            // x first, before the weight ring's traffic: each row one bulk copy
            // of its K bf16 values into its shared-memory row (a row a device
            // check skips leaves the barrier short: its bounded wait ends it)
            mbar_arrive_expect_tx(smem_u32(xbar), (uint32_t)(M * K * 2));
            for (int64_t r = 0; r < M; ++r)
                if (BSQ_IN_BUFFER(args.err, kChkGemvX, r * K, K, M * K))
                    bulk_load(smem_u32(sX + r * x_pitch), args.x + r * K, (uint32_t)(K * 2), smem_u32(xbar));
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmS2);
            prefetch_tmap(&tmS1);
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int st = i % n_stages;
                if (i >= n_stages &&
                    !mbar_wait(smem_u32(empty + st), ((i / n_stages) - 1) & 1, args.err, abort_flag, kErrGemvProducer))
                    break;
                const int n_rb = rb1 - rb0 + 1;
                mbar_arrive_expect_tx(smem_u32(full + st), kWBytes + (uint32_t)n_rb * 2048u);
                tma_load_2d(smem_u32(sWst + st * kWBytes), &tmW, smem_u32(full + st), i * 128, (int32_t)row_base);
                load_scale_tiles(smem_u32(sSst + st * kSBytes), &tmS2, &tmS1, smem_u32(full + st), i, rb0, n_rb);
                issued = i + 1;
            }
            if (*abort_flag) {
                for (int i = issued - n_stages < 0 ? 0 : issued - n_stages; i < issued; ++i) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(full + i % n_stages), (i / n_stages) & 1) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
            {   // the x copy too
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(xbar), 0) && globaltimer() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    // 1. x has been copied into shared memory (the producer's first transfer):
    //    check every value (one AND over the consumer threads), then convert it
    //    in place to f16 or leave it raw bf16.  A row holds nst * 256 values
    //    (the K tail zero, as the weight's TMA fill there is zero) plus 64 bytes
    //    of padding.
    const bool x_ok = mbar_wait(smem_u32(xbar), 0, args.err, abort_flag, kErrGemvConsumer);
    const int64_t row_units = (int64_t)nst * 32;                        // 16-byte units per staged row
    uint32_t okb = ~0u;
    for (int64_t u = threadIdx.x; u < M * row_units; u += kCons) {
        const int64_t r = u / row_units, c = u - r * row_units;
        if (c < K / 8) okb &= f16_exact_bits4(*reinterpret_cast<const uint4*>(sX + r * x_pitch + 16 * c));
    }
    const bool use_f16 = bar_and(1, kCons, f16_exact(okb));
    for (int64_t u = threadIdx.x; u < M * row_units; u += kCons) {
        const int64_t r = u / row_units, c = u - r * row_units;
        uint4* p = reinterpret_cast<uint4*>(sX + r * x_pitch + 16 * c);
        if (c >= K / 8) {
            *p = make_uint4(0, 0, 0, 0);
        } else if (use_f16) {
            const uint4 v = *p;
            *p = bf16x8_to_f16x8(v);
        }
    }
    bar_and(1, kCons, x_ok);                                            // x staged for every warp

    const int g = lane >> 2, t = lane & 3;
    const int64_t row0 = row_base + warp * 16 + g, row1 = row0 + 8;
    const int nblocks32 = (int)(K / 16);     // K < 2^31: the entry point bounds every dimension
    const int mrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
    const int mcol = lane >> 4;
    int soff[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int64_t row = r ? row1 : row0;
        soff[r] = (int)((row >> 7) - rb0) * 2048 + (int)(row & 31) * 16 + (int)((row >> 5) & 3) * 4;
    }
    const uint32_t ssel = (t >> 1) ? 0x31u : 0x20u;
    const bool x_row = g < M;                                           // B rows past M are zero
    const uint32_t xrow = smem_u32(sX) + (uint32_t)(x_row ? g : 0) * x_pitch + 16 * t;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    auto consume = [&](auto f16_tag, auto tail_tag, uint32_t wst, uint32_t sst, int i) {
        constexpr bool F16 = decltype(f16_tag)::value;
        constexpr bool TAIL = decltype(tail_tag)::value;
        const uint32_t xs = xrow + (uint32_t)i * 512;                   // 256 values of this stage
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
            uint32_t wr[4];
            ldmatrix_x4(wst + mrow * 128 + (((2 * cp + mcol) ^ (mrow & 7)) << 4), wr);
            uint32_t S[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t two = __byte_perm(lds32(sst + soff[r] + cp * 512), 0, ssel);
                if constexpr (F16) {
                    const uint32_t sf = e4m3x2_to_f16x2(two);
                    S[r][0] = __byte_perm(sf, sf, 0x1010);
                    S[r][1] = __byte_perm(sf, sf, 0x3232);
                } else {
                    const uint32_t b0 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32(two & 0xFF), 0x1p119f));
                    const uint32_t b1 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32((two >> 8) & 0xFF), 0x1p119f));
                    S[r][0] = b0 | (b0 << 16);
                    S[r][1] = b1 | (b1 << 16);
                }
                if constexpr (TAIL) {
                    const int blk0 = 16 * i + 4 * cp + (t >> 1);
                    if (blk0 >= nblocks32) S[r][0] = 0;
                    if (blk0 + 2 >= nblocks32) S[r][1] = 0;
                }
            }
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t Pp[2][4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if constexpr (F16) {
                        e2m1x8_to_f16x2(wr[2 * ch + r], Pp[r]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) Pp[r][j] = hmul2(Pp[r][j], S[r][ch]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            Pp[r][j] = bmul2(place_byte_bf16x2((wr[2 * ch + r] >> (8 * j)) & 0xFFu), S[r][ch]);
                    }
                }
                const uint4 xv = x_row ? lds128(xs + 64 * (2 * cp + ch)) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t a[4] = {Pp[0][2 * e], Pp[1][2 * e], Pp[0][2 * e + 1], Pp[1][2 * e + 1]};
                    mma16816<F16>(acc, a, e ? xv.z : xv.x, e ? xv.w : xv.y);
                }
            }
        }
    };

    // SLOT: per-row block partial sums (columns 2t, 2t+1 of rows g, g+8), scaled
    float acc_s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t xrow0 = smem_u32(sX) + 16 * t;                       // x row 0
    auto consume_slot = [&](auto tail_tag, uint32_t wst, uint32_t sst, int i) {
        constexpr bool TAIL = decltype(tail_tag)::value;
        const uint32_t xs = xrow0 + (uint32_t)i * 512;
#pragma unroll
        for (int G = 0; G < 2; ++G) {                                   // blocks 8G .. 8G+7 of the stage
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int cq = 0; cq < 2; ++cq) {
                const int cp = 2 * G + cq;
                uint32_t wr[4];
                ldmatrix_x4(wst + mrow * 128 + (((2 * cp + mcol) ^ (mrow & 7)) << 4), wr);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int chunk = 2 * cp + ch;                      // 32 codes: blocks 2chunk, 2chunk+1
                    uint32_t Pp[2][4];
                    e2m1x8_to_f16x2(wr[2 * ch], Pp[0]);
                    e2m1x8_to_f16x2(wr[2 * ch + 1], Pp[1]);
                    // this lane's codes 8t..8t+7 lie in block 2chunk + (t >> 1): column (that block) % 8
                    const bool mine = g == ((2 * chunk + (t >> 1)) & 7);
                    const uint4 xv = mine ? lds128(xs + 64 * chunk) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t a[4] = {Pp[0][2 * e], Pp[1][2 * e], Pp[0][2 * e + 1], Pp[1][2 * e + 1]};
                        mma16816<true>(d, a, e ? xv.z : xv.x, e ? xv.w : xv.y);
                    }
                }
            }
            // columns 2t, 2t+1 of this group are blocks 8G + 2t + {0, 1}
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t two = lds32(sst + soff[r] + (2 * G + (t >> 1)) * 512) >> (16 * (t & 1));
                float s0 = ue4m3_bits_to_f32(two & 0xFFu), s1 = ue4m3_bits_to_f32((two >> 8) & 0xFFu);
                if constexpr (TAIL) {
                    const int blk0 = 16 * i + 8 * G + 2 * t;
                    if (blk0 >= nblocks32) s0 = 0.0f;
                    if (blk0 + 1 >= nblocks32) s1 = 0.0f;
                }
                acc_s[2 * r] = __fmaf_rn(s0, d[2 * r], acc_s[2 * r]);
                acc_s[2 * r + 1] = __fmaf_rn(s1, d[2 * r + 1], acc_s[2 * r + 1]);
            }
        }
    };

    for (int i = 0; i < nst; ++i) {
        const int st = i % n_stages;
        if (mbar_wait(smem_u32(full + st), (i / n_stages) & 1, args.err, abort_flag, kErrGemvConsumer)) {
            const uint32_t wst = smem_u32(sWst + st * kWBytes), sst = smem_u32(sSst + st * kSBytes);
            const bool tail = 16 * (i + 1) > nblocks32;
            if (SLOT && use_f16) {
                if (tail) consume_slot(std::true_type{}, wst, sst, i);
                else consume_slot(std::false_type{}, wst, sst, i);
            } else if (use_f16) {
                if (tail) consume(std::true_type{}, std::true_type{}, wst, sst, i);
                else consume(std::true_type{}, std::false_type{}, wst, sst, i);
            } else {
                if (tail) consume(std::false_type{}, std::true_type{}, wst, sst, i);
                else consume(std::false_type{}, std::false_type{}, wst, sst, i);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + st));
    }

    // ---- epilogue: the bf16 path's products carry 2^-7 ----
    if (*abort_flag) return;
    const float gw = __fmul_rn(args.gW ? __ldg(args.gW) : 1.0f, use_f16 ? 1.0f : 0x1p7f);
    if (SLOT && use_f16) {
        // a row's sum over its eight block columns: two per lane, then the four lanes t
        float v0 = acc_s[0] + acc_s[1], v1 = acc_s[2] + acc_s[3];
        v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
        v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
        v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
        v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
        if (t == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int64_t n = r ? row1 : row0;
                if (n < N) store_y(args.y, args.out_bf16, n, __fmul_rn(r ? v1 : v0, gw), args.err, M * N);
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = 2 * t + (i & 1);
        const int64_t n = (i < 2) ? row0 : row1;
        if (m < M && n < N) store_y(args.y, args.out_bf16, m * N + n, __fmul_rn(acc[i], gw), args.err, M * N);
    }
}


// Tensor-core variant (17 <= M <= 32): the decoded weight becomes the A operand
// of tcgen05.mma kind::f16 straight from tensor memory, so the warps that
// decode do no MMA work, no x fragment loads and hold no accumulators.
//  * CTA = 192 weight rows, one CTA per SM (28672 rows: 150 CTAs).  Tile 0 =
//    rows 0..127 in TMEM lanes 0..127, tile 1 = rows 128..191 in lanes 0..63
//    of a second set of A columns; each tile is one M = 128 MMA (tile 1's
//    lanes 64..127 carry nothing and their accumulator lanes are never read).
//    x is checked, converted and read from L2 once per 192 rows: with two
//    96-row CTAs per SM each did it for itself, and that x work, not the
//    decode, set the kernel's time.
//  * Warp 0 issues TMA, warp 1 owns TMEM and issues tile 0's MMAs, warp 18
//    issues tile 1's (on another scheduler: one thread issuing both tiles'
//    small MMAs was the slower design), warps 2..17 decode: per TMEM lane
//    quarter q four warps, (h, p) = K half h of every
//    256-code stage (a "granule") and part p.  Quarters 0, 1 (which hold rows
//    of both tiles): part p decodes its lane's row of tile p, all four
//    32-code chunks of the granule.  Quarters 2, 3 (tile 0 only): part p
//    decodes chunks 2p, 2p + 1 of its lane's row and, with the other three
//    such warps of half h, checks and converts the granule's x.
//  * Stage (256 codes): the codes (2-D box {128 B, 192 rows}, 128-byte
//    swizzle), the scale atoms of the two 128-row tiles the rows span (one
//    3-D tensor-map load) and x as four 2-D boxes {64 values, NP rows}
//    (128-byte swizzle, rows >= M zero-filled) -- x is already the K-major B
//    operand of the MMA (N = NP = 32).
//  * Granule (128 codes of every row): the x warps check whether its
//    2 x NP x 64 x values are exact in f16 (one AND over the half's four x
//    warps), publish the decision for that stage and half (a flag and an
//    mbarrier) and, if so, rewrite x in place as f16; then every row's codes
//    take the hardware e2m1 -> f16 conversion times the ue4m3 scale (exact).
//    Else x stays bf16 and the codes take the placed-bf16 decode (value *
//    scale * 2^-7, exact), accumulating into a second fp32 tile lifted by 2^7
//    at the end.  Quarters 0, 1 do not wait for the decision: they decode for
//    f16 x at once and decode again when the decision is bf16.  Decoded
//    chunks go by tcgen05.st into the row's TMEM lane (column j holds K
//    values 2j, 2j + 1) in one of three granule slots.
//  * MMA: per granule and tile eight kind::f16 MMAs (M = 128, N = NP, K = 16,
//    A from TMEM) into that tile's f16 or bf16 accumulator (zeroed by the
//    decode warps first); a granule slot is released by a commit, a stage
//    after its second granule.
//  * Epilogue: the decode warps read both accumulators of their tile
//    (tcgen05.ld), combine, scale by gW and store y[m, n] for m < M.
// Every wait is bounded (2 s); a timeout records its site in the device error
// word and the CTA drains what it issued before it leaves.
namespace tc {

constexpr int kStages = 4;
constexpr int kRows = 192;
constexpr int kDecWarps = 16;
constexpr int kMmaWarp1 = 2 + kDecWarps;  // issues tile 1's MMAs (warp 1 issues tile 0's), on another scheduler
constexpr int kThreads = (3 + kDecWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kSlots = 3;                 // granule slots: two tiles x 64 columns each
constexpr uint32_t kColAcc = 384;         // tile t: f16 accumulator at kColAcc + 64 t, bf16 at + 32

template <int NP>
struct Plan {
    static constexpr int kW = kRows * 128;
    static constexpr int kS = 2 * 4 * 512;                // the atoms of the two 128-row tiles the rows span
    static constexpr int kXBox = NP * 128;
    static constexpr int kX = 4 * kXBox;
    static constexpr int kStage = kW + kS + kX;          // a multiple of 1024
    static constexpr int kBytes = 1024 + kStages * kStage + 256;
    static_assert(kStage % 1024 == 0, "1024-byte aligned stages (128-byte swizzle)");
    static_assert(NP == 32, "the accumulator columns hold 32 activation rows");
    static_assert((4 * kStages + 2 * kSlots + 3) * 8 + 2 * kStages * 4 + 8 <= 256, "barrier area");
};

__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc) {
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;"
                 :: "r"(d), "r"(a_tmem), "l"(bdesc), "r"(idesc) : "memory");
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
gemv_nvf4_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmS2, const Args args) {
    using P = Plan<NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * P::kStage);
    uint64_t* empty = full + kStages;
    uint64_t* a_full = empty + kStages;
    uint64_t* a_empty = a_full + kSlots;
    uint64_t* acc_full = a_empty + kSlots;
    uint64_t* drain = acc_full + 1;                                  // [2]: one per MMA warp
    uint64_t* xready = drain + 2;                                    // [stage][half]: that xflag is set
    uint32_t* xflag = reinterpret_cast<uint32_t*>(xready + 2 * kStages);   // [stage][half]: its x is f16
    uint32_t* tmem_base_s = xflag + 2 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t row_base = (int64_t)blockIdx.x * kRows;
    const int nst = (int)((K + 255) / 256);
    const int ngr = 2 * nst;
    const int nblocks = (int)(K / 16);
    const int64_t rb = row_base >> 7;                 // first 128-row scale tile the rows touch

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 2);                // both MMA warps' commits
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(smem_u32(a_full + i), kDecWarps / 2);
            mbar_init(smem_u32(a_empty + i), 2);
        }
        mbar_init(smem_u32(acc_full), 2);
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(drain + 1), 1);
        for (int i = 0; i < 2 * kStages; ++i) mbar_init(smem_u32(xready + i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_base_s), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    pdl_wait_then_release();

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            prefetch_tmap(&tmS2);
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(smem_u32(empty + s), ((i / kStages) - 1) & 1, args.err, abort_flag, kErrGemvProducer))
                    break;
                uint8_t* st = smem + s * P::kStage;
                const uint32_t fb = smem_u32(full + s);
                mbar_arrive_expect_tx(fb, P::kW + P::kS + P::kX);
                tma_load_2d(smem_u32(st), &tmW, fb, i * 128, (int32_t)row_base);
                tma_load_3d(smem_u32(st + P::kW), &tmS2, fb, 0, 4 * i, (int32_t)rb);   // tiles rb, rb + 1 (zeros past N)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tma_load_2d(smem_u32(st + P::kW + P::kS + j * P::kXBox), &tmX, fb, i * 256 + 64 * j, 0);
                issued = i + 1;
            }
            if (*abort_flag) {
                for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(full + i % kStages), (i / kStages) & 1) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1 || warp == kMmaWarp1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            const int t = warp == 1 ? 0 : 1;                // this warp's tile
            const uint32_t id_h = (1u << 4) | ((uint32_t)(NP >> 3) << 17) | ((128u >> 4) << 24);
            const uint32_t id_b = id_h | (1u << 7) | (1u << 10);
            const uint64_t dX0 = smem_desc(smem_u32(smem + P::kW + P::kS), 16, 1024, 2);
            for (int gi = 0; gi < ngr; ++gi) {
                const int slot = gi % kSlots, i = gi >> 1, h = gi & 1, s = i % kStages;
                // a_full orders the stage's TMA data too: every decode warp waited for `full`
                // before it arrived, so the stage's x (the B operand) has landed
                if (!mbar_wait(smem_u32(a_full + slot), (gi / kSlots) & 1, args.err, abort_flag, kErrGemvConsumer))
                    break;
                tc_fence_after();
                const bool f16 = xflag[2 * s + h] != 0;
                const uint32_t idesc = f16 ? id_h : id_b;
                const uint64_t xs = dX0 + (uint64_t)((s * P::kStage) >> 4);
                const uint32_t d = tmem + kColAcc + 64 * t + (f16 ? 0 : 32);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int box = 2 * h + (kk >> 2);
                    mma_f16_ts(d, tmem + 128 * slot + 64 * t + 8 * kk, xs + (uint64_t)((box * P::kXBox) >> 4) + 2 * (kk & 3),
                               idesc);
                }
                tc_commit(smem_u32(a_empty + slot));
                if (h == 1 || gi == ngr - 1) tc_commit(smem_u32(empty + s));
            }
            tc_commit(smem_u32(acc_full));
            tc_commit(smem_u32(drain + t));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(drain + t), 0)) {
                if (globaltimer() - t0 > kWaitLimitNs) { atomicCAS(args.err, 0u, (uint32_t)kErrGemvConsumer); break; }
            }
        }
    } else {
        // --------------------------------------------------------- decode --
        const int q = warp & 3;                        // TMEM lane quarter
        const int grp = (warp - 2) >> 2;               // 0..3: every group has one warp of each quarter
        const int h = grp & 1, p = grp >> 1;           // K half of every stage, part
        const bool xw = q >= 2;                        // quarters 2, 3 also do the granule's x
        const int tile = xw ? 0 : p;
        const int r = 128 * tile + 32 * q + lane;      // CTA row
        const int cc0 = xw ? 2 * p : 0, ncc = xw ? 2 : 4;   // this warp's chunks of the granule
        const int xtid = ((q & 1) + 2 * p) * 32 + lane;     // 0..127 over the half's four x warps
        const bool xlead = q == 2 && p == 0;                // publishes the half's x decision
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t acc_col = kColAcc + 64 * tile;
        if (h == 0 && (!xw || p == 0)) {   // this tile's accumulators start at zero (every MMA
                                           // accumulates), before the first granule reaches the MMA warp
            uint32_t z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0;
            tc_st_cols(lane_base + acc_col, z);
            tc_st_cols(lane_base + acc_col + 32, z);
            tc_wait_st();
        }
        const int64_t nrow = row_base + r;                 // this thread's weight row
        const uint32_t soff = (uint32_t)(((nrow >> 7) - rb) * 2048 + (nrow & 31) * 16 + ((nrow >> 5) & 3) * 4);
        const int xunits = (int)(16 * M);            // 16-byte x units of rows < M in the granule's two boxes
        constexpr int kXPer = NP / 8;                  // at most this many per x thread
        for (int gi = h; gi < ngr; gi += 2) {
            const int slot = gi % kSlots, i = gi >> 1, s = i % kStages;
            uint8_t* st = smem + s * P::kStage;
            const bool have = mbar_wait(smem_u32(full + s), (i / kStages) & 1, args.err, abort_flag, kErrGemvConsumer);
            // the row's chunks of this granule: chunk c = 4h + cc (32 codes, blocks 2c, 2c + 1 of the stage)
            const uint32_t wrow = smem_u32(st) + r * 128;
            const uint8_t* srow = st + P::kW + soff;
            const bool tail = 16 * (i + 1) > nblocks;        // uniform: only the last stage
            auto decode = [&](bool f16) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k >= ncc) break;
                    const int cc = cc0 + k;
                    const int c = 4 * h + cc;
                    const uint4 w = lds128(wrow + ((c ^ (r & 7)) << 4));
                    uint32_t two = *reinterpret_cast<const uint16_t*>(srow + (c >> 1) * 512 + ((2 * c) & 3));
                    if (tail) {                               // blocks past K: scale 0
                        const int blk0 = 16 * i + 2 * c;
                        if (blk0 >= nblocks) two &= 0xFF00u;
                        if (blk0 + 1 >= nblocks) two &= 0x00FFu;
                    }
                    uint32_t a[16];
                    if (f16) {
                        const uint32_t sf = e4m3x2_to_f16x2(two);
                        const uint32_t s0 = __byte_perm(sf, sf, 0x1010), s1 = __byte_perm(sf, sf, 0x3232);
                        uint32_t t4[4];
                        e2m1x8_to_f16x2(w.x, t4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) a[j] = hmul2(t4[j], s0);
                        e2m1x8_to_f16x2(w.y, t4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) a[4 + j] = hmul2(t4[j], s0);
                        e2m1x8_to_f16x2(w.z, t4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) a[8 + j] = hmul2(t4[j], s1);
                        e2m1x8_to_f16x2(w.w, t4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) a[12 + j] = hmul2(t4[j], s1);
                    } else {
                        const uint32_t b0 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32(two & 0xFF), 0x1p119f));
                        const uint32_t b1 = f32_to_bf16_bits(__fmul_rn(e4m3_to_f32((two >> 8) & 0xFF), 0x1p119f));
                        const uint32_t s0 = b0 | (b0 << 16), s1 = b1 | (b1 << 16);
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int kw = 0; kw < 4; ++kw)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                a[4 * kw + j] = bmul2(place_byte_bf16x2((ww[kw] >> (8 * j)) & 0xFFu), kw < 2 ? s0 : s1);
                    }
                    tc_st_cols(lane_base + 128 * slot + 64 * tile + 16 * cc, a);
                }
            };
            if (xw) {
                // x boxes 2h, 2h + 1: exact in f16?  One AND over the half's four x warps (run
                // even after a failed wait).  Unit v: box 2h + v / (8M), row (v % (8M)) / 8,
                // 16-byte piece v % 8 (rows >= M are zero fill).
                uint8_t* xb = st + P::kW + P::kS + 2 * h * P::kXBox;
                auto xaddr = [&](int v) {                   // v < 16M: two boxes of 8M units
                    const int half = 8 * (int)M;
                    return v < half ? xb + v * 16 : xb + P::kXBox + (v - half) * 16;
                };
                uint4 xv[kXPer];
                uint32_t okb = ~0u;
#pragma unroll
                for (int u = 0; u < kXPer; ++u) {
                    const int v = xtid + 128 * u;
                    xv[u] = make_uint4(0, 0, 0, 0);
                    if (have && v < xunits) xv[u] = *reinterpret_cast<const uint4*>(xaddr(v));
                    okb &= f16_exact_bits4(xv[u]);
                }
                const bool f16 = bar_and(1 + h, 128, f16_exact(okb));
                if (!have) continue;
                // the decision for the other warps of the half and the MMA warps (this stage's
                // previous readers of the flag are done: the stage was refilled after its MMAs)
                if (xlead && lane == 0) {
                    xflag[2 * s + h] = f16 ? 1u : 0u;
                    mbar_arrive(smem_u32(xready + 2 * s + h));
                }
                if (f16) {      // in place, before the slot wait: only this granule's MMAs read it
#pragma unroll
                    for (int u = 0; u < kXPer; ++u) {
                        const int v = xtid + 128 * u;
                        if (v < xunits)
                            *reinterpret_cast<uint4*>(xaddr(v)) = bf16x8_to_f16x8(xv[u]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                if (gi >= kSlots &&
                    !mbar_wait(smem_u32(a_empty + slot), ((gi / kSlots) - 1) & 1, args.err, abort_flag, kErrGemvConsumer))
                    continue;
                decode(f16);
            } else {
                // decode for f16 x at once (activations nearly always are), then take the x
                // warps' decision and decode again the rare granule whose x is not
                if (gi >= kSlots &&
                    !mbar_wait(smem_u32(a_empty + slot), ((gi / kSlots) - 1) & 1, args.err, abort_flag, kErrGemvConsumer))
                    continue;
                if (!have) continue;
                decode(true);
                if (!mbar_wait(smem_u32(xready + 2 * s + h), (i / kStages) & 1, args.err, abort_flag, kErrGemvConsumer))
                    continue;
                if (xflag[2 * s + h] == 0) {
                    tc_wait_st();
                    decode(false);
                }
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(a_full + slot));
        }
        // ------------------------------------------------------- epilogue --
        // The warps that share a (tile, quarter) split its NP activation
        // columns: quarters 0, 1 by h (16 each), quarters 2, 3 by (p, h) (8 each).
        if (mbar_wait(smem_u32(acc_full), 0, args.err, abort_flag, kErrGemvConsumer) && !*abort_flag) {
            tc_fence_after();
            const float gw = args.gW ? __ldg(args.gW) : 1.0f;
            const int64_t n = row_base + r;
            const int c16 = xw ? 16 * p : 16 * h;          // the 16 columns this warp loads
            uint32_t dh[16], db[16];
            tc_ld_32x32b_x16(lane_base + acc_col + c16, dh);
            tc_ld_32x32b_x16(lane_base + acc_col + 32 + c16, db);
            tc_wait_ld();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fmaf_rn(__uint_as_float(db[j]), 0x1p7f, __uint_as_float(dh[j]));
            const int j0 = xw ? 8 * h : 0, nj = xw ? 8 : 16;     // of the 16 loaded, the columns stored
            if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int64_t m = c16 + j;
                    if (j >= j0 && j < j0 + nj && m < M)
                        store_y(args.y, args.out_bf16, m * N + n, __fmul_rn(v[j], gw), args.err, M * N);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace tc

}  // namespace nvf4

// Consumer warps per CTA (16 rows each) for the nvfp4 GEMV: the choice in
// {4, 6, 8, 12} with the least rows per SM over whole waves (one CTA per SM).
int nvf4_warps(int64_t N, int sms) {
    const int cand[4] = {12, 8, 6, 4};
    int best = 8;
    int64_t best_cost = INT64_MAX;
    for (int w : cand) {
        const int64_t tiles = (N + 16 * w - 1) / (16 * w);
        const int64_t cost = (tiles + sms - 1) / sms * w;
        if (cost < best_cost) { best_cost = cost; best = w; }
    }
    return best;
}

// The weight's tensor map and its scale buffer's (2-tile and 1-tile boxes).
struct NvfMaps {
    CUtensorMap w, s2, s1;
};

// Programmatic dependent launch: the kernel's prologue may overlap the
// previous kernel on the stream; the kernel waits (griddepcontrol.wait)
// before reading anything that kernel wrote.
template <typename KernelT, typename... Args>
cudaError_t launch_pdl(KernelT kernel, dim3 grid, int threads, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int NT, int CW>
bsq_status launch_nvf4_cfg(const NvfMaps& mp, const uint16_t* x, const nvf4::Args& a, cudaStream_t s) {
    constexpr int R = 16 * CW;
    constexpr size_t smem = nvf4::Plan<NT, CW>::kBytes;
    auto kern = nvf4::gemv_nvf4_kernel<NT, CW>;
    // x [M, K] bf16 as {64 values, 8 NT rows} boxes, 128-byte swizzle; rows >= M
    // and values past K are zero fill
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return BSQ_ERR_UNSUPPORTED;
    CUtensorMap tmX;
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K * 2)};
    const cuuint32_t box[2] = {64, (cuuint32_t)(8 * NT)};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BSQ_ERR_UNSUPPORTED;
    static std::once_flag once[64];
    static bool ok_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSQ_ERR_CUDA;
    std::call_once(once[dev], [&] {
        ok_dev[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
    });
    if (!ok_dev[dev]) { (void)cudaGetLastError(); return BSQ_ERR_UNSUPPORTED; }
    const dim3 grid((unsigned)((a.N + R - 1) / R));
    if (launch_pdl(kern, grid, (CW + 1 + nvf4::kXWarps) * 32, smem, s, mp.w, mp.s2, mp.s1, tmX, a) != cudaSuccess) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    return launch_status();
}

template <int NT>
bsq_status launch_nvf4_nt(int cw, const NvfMaps& mp, const uint16_t* x, const nvf4::Args& a, cudaStream_t s) {
    switch (cw) {
    case 12: return launch_nvf4_cfg<NT, 12>(mp, x, a, s);
    case 8: return launch_nvf4_cfg<NT, 8>(mp, x, a, s);
    case 6: return launch_nvf4_cfg<NT, 6>(mp, x, a, s);
    default: return launch_nvf4_cfg<NT, 4>(mp, x, a, s);
    }
}

// The resident-x kernel when x and a ring of >= 6 stages fit (M <= 2 at K = 8192);
// returns -1 (nothing launched) when they do not.
template <int CW, bool SLOT>
int launch_nvf4_res_cfg(const NvfMaps& mp, const nvf4::Args& a, cudaStream_t s) {
    constexpr int R = 16 * CW;
    constexpr int64_t kStage = R * 128 + nvf4::kMaxRowBlocks * 2048;
    // nst * 256 values per row (the K tail zero) + 64 bytes: == 64 mod 128, conflict-free B reads
    const int64_t pitch = (a.K + 255) / 256 * 512 + 64;
    const int64_t fixed = 1024 + a.M * pitch + (2 * nvf4::kResMaxStages + 1) * 8 + 16;
    int64_t stages = (nvf4::kSmemLimit - fixed) / kStage;
    if (stages > nvf4::kResMaxStages) stages = nvf4::kResMaxStages;
    if (stages < 6) return -1;                               // a shallower ring starves the consumers
    const size_t smem = (size_t)(fixed + stages * kStage);
    auto kern = nvf4::gemv_nvf4_res_kernel<CW, SLOT>;
    static std::once_flag once[64];
    static bool ok_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSQ_ERR_CUDA;
    std::call_once(once[dev], [&] {
        ok_dev[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, nvf4::kSmemLimit) ==
                      cudaSuccess;
    });
    if (!ok_dev[dev]) { (void)cudaGetLastError(); return -1; }
    const dim3 grid((unsigned)((a.N + R - 1) / R));
    if (launch_pdl(kern, grid, (CW + 1) * 32, smem, s, mp.w, mp.s2, mp.s1, a, (int)stages, (uint32_t)pitch) != cudaSuccess) { (void)cudaGetLastError(); return (int)BSQ_ERR_CUDA; }
    return (int)launch_status();
}

template <bool SLOT>
int launch_nvf4_res_slot(int cw, const NvfMaps& mp, const nvf4::Args& a, cudaStream_t s) {
    switch (cw) {
    case 12: return launch_nvf4_res_cfg<12, SLOT>(mp, a, s);
    case 8: return launch_nvf4_res_cfg<8, SLOT>(mp, a, s);
    case 6: return launch_nvf4_res_cfg<6, SLOT>(mp, a, s);
    default: return launch_nvf4_res_cfg<4, SLOT>(mp, a, s);
    }
}

int launch_nvf4_res(int cw, const NvfMaps& mp, const nvf4::Args& a, cudaStream_t s) {
    return a.M == 1 ? launch_nvf4_res_slot<true>(cw, mp, a, s) : launch_nvf4_res_slot<false>(cw, mp, a, s);
}


// The tensor-core kernel (17 <= M <= 32); -1 when it cannot be launched here.
template <int NP>
int launch_nvf4_tc_cfg(const DeviceInfo* info, const NvfMaps& mp, const uint16_t* x, const nvf4::Args& a,
                       cudaStream_t s) {
    using P = nvf4::tc::Plan<NP>;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return -1;
    CUtensorMap tmX;
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K * 2)};
    const cuuint32_t box[2] = {64, (cuuint32_t)NP};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return -1;
    auto kern = nvf4::tc::gemv_nvf4_tc_kernel<NP>;
    static std::once_flag once[64];
    static bool ok_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSQ_ERR_CUDA;
    std::call_once(once[dev], [&] {
        ok_dev[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kBytes) == cudaSuccess;
    });
    if (!ok_dev[dev]) { (void)cudaGetLastError(); return -1; }
    (void)info;
    const dim3 grid((unsigned)((a.N + nvf4::tc::kRows - 1) / nvf4::tc::kRows));
    if (launch_pdl(kern, grid, nvf4::tc::kThreads, P::kBytes, s, mp.w, tmX, mp.s2, a) != cudaSuccess) { (void)cudaGetLastError(); return (int)BSQ_ERR_CUDA; }
    return (int)launch_status();
}

bsq_status launch_nvf4(const DeviceInfo* info, const uint16_t* x, const uint8_t* W, const uint8_t* sW,
                       const float* gW, void* y, int out, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    const int cw = nvf4_warps(N, info->num_sms);
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return BSQ_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    const cuuint32_t es[3] = {1, 1, 1};
    auto weight_map = [&](CUtensorMap* m, uint32_t rows) {
        const cuuint32_t box[2] = {128, rows};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // the scale buffer as 32-bit words {128 of an atom, atoms along K, 128-row tiles}
    const int64_t cpd4 = pad_to(K / 16, 4) / 4;
    auto scale_map = [&](CUtensorMap* m, uint32_t tiles) {
        const cuuint64_t sd[3] = {128, (cuuint64_t)cpd4, (cuuint64_t)(pad_to(N, 128) / 128)};
        const cuuint64_t ss[2] = {512, (cuuint64_t)(cpd4 * 512)};
        const cuuint32_t sb[3] = {128, 4, tiles};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(sW), sd, ss, sb, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    NvfMaps mp;
    if (!scale_map(&mp.s2, 2) || !scale_map(&mp.s1, 1)) return BSQ_ERR_UNSUPPORTED;
    nvf4::Args a;
    a.x = x; a.sW = sW; a.gW = gW; a.y = y; a.err = info->err; a.M = M; a.N = N; a.K = K;
    a.cpd4 = cpd4;
    a.out_bf16 = out;
    if (M > 16) {
        // 17..32 activation rows: the tensor-core kernel (mma.sync issue would
        // bound the register-decode kernels); it reads the weight in 192-row boxes
        if (weight_map(&mp.w, (uint32_t)nvf4::tc::kRows)) {
            const int st = launch_nvf4_tc_cfg<32>(info, mp, x, a, s);
            if (st >= 0) return (bsq_status)st;
        }
    }
    if (!weight_map(&mp.w, (uint32_t)(16 * cw))) return BSQ_ERR_UNSUPPORTED;
    if (M <= 8) {
        const int st = launch_nvf4_res(cw, mp, a, s);
        if (st >= 0) return (bsq_status)st;
        return launch_nvf4_nt<1>(cw, mp, x, a, s);
    }
    if (M <= 16) return launch_nvf4_nt<2>(cw, mp, x, a, s);
    return launch_nvf4_nt<4>(cw, mp, x, a, s);
}

template <int WFMT>
bsq_status launch_fmt(const uint16_t* x, const uint8_t* W, const uint8_t* sW, const float* gW, void* y, int out,
                      int64_t M, int64_t N, int64_t K, uint32_t* err, cudaStream_t s) {
    const dim3 grid((unsigned)((N + kRowsPerCta - 1) / kRowsPerCta));
    if (M <= 8) gemv_kernel<1, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K, err);
    else if (M <= 16) gemv_kernel<2, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K, err);
    else gemv_kernel<4, WFMT><<<grid, kThreads, 0, s>>>(x, W, sW, gW, y, out, M, N, K, err);
    return launch_status();
}

}  // namespace

bsq_status gemv_launch(const uint16_t* x, const void* W, int fw, const uint8_t* sW, const float* gW, void* y,
                       int out, int64_t M, int64_t N, int64_t K, bool nvfp4, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const uint8_t* Wb = static_cast<const uint8_t*>(W);
    bsq_status r;
    if (nvfp4) {
        r = launch_nvf4(info, x, Wb, sW, gW, y, out, M, N, K, s);
        count_launch(BSQ_KERNEL_GEMV_NVFP4);
    } else {
        if (fw == kE3M2) r = launch_fmt<kE3M2>(x, Wb, sW, gW, y, out, M, N, K, info->err, s);
        else if (fw == kE2M3) r = launch_fmt<kE2M3>(x, Wb, sW, gW, y, out, M, N, K, info->err, s);
        else r = launch_fmt<kE4M3>(x, Wb, sW, gW, y, out, M, N, K, info->err, s);
        count_launch(BSQ_KERNEL_GEMV_MX);
    }
    return r;
}

}  // namespace bsq
