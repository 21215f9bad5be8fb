// quantize.cu -- bf16 -> MX (e3m2 / e2m3 / e4m3, UE8M0 per 32) and
// bf16 -> nvfp4 (e2m1, ue4m3 per 16) block quantizers.
//
// Recipe: b12x _lib/fp6.py, quantize_grouped_mxfp6_torch with the exact scale
// steps of fp6_block_ue8m0_exact / ue8m0_output_scale_exact and the per-block
// quantizers quantize_block_fp6_*_fast (the nvfp4 variant is the same recipe
// with e2m1's maximum and a round-to-nearest e4m3 block scale).
//
// Two launch shapes:
//  * small tensors (M*K <= kFusedMaxElems): ONE launch of a 16-CTA thread-block
//    cluster.  Each CTA reduces the amax of its slice, the cluster exchanges
//    the partial maxima through distributed shared memory, and every CTA then
//    encodes its share of the blocks.  No workspace, no grid-wide wait.
//  * large tensors: an amax pass writes per-CTA partial maxima to the caller's
//    workspace; the encode pass reduces them (a few hundred words) in every
//    CTA and encodes.  The second read of x is normally an L2 hit.  The encode
//    pass is a programmatic dependent launch: it is scheduled while the amax
//    pass runs and waits for it (griddepcontrol) before reading the partials.
//
// Encode mapping: one warp per (row, 1024-element chunk); each lane owns 32
// consecutive values (one MX block, or two nvfp4 blocks) = 64 contiguous bytes,
// so the block amax and scale math run once per 32 values without shuffles.
#include <cstdio>
#include <atomic>
#include <mutex>

#include "bsq_device.cuh"
#include "bsq_internal.h"
#include "mx_encode.cuh"

namespace bsq {
namespace {

constexpr int kThreads = 256;                // amax pass and the fused cluster launch
constexpr int kEncThreads = 1024;            // encode pass: one CTA per SM
constexpr int kMaxPartials = 2048;
constexpr int64_t kFusedMaxElems = 1 << 16;    // 128 KiB of bf16
constexpr int kFusedCluster = 16;   // non-portable size; 8 where 16 is refused

// Largest |bf16| magnitude bits among the 8 values of a 16-byte load.
// For non-NaN bf16, (bits & 0x7FFF) orders like |value|.
__device__ __forceinline__ uint32_t absmax8_bits(uint4 v) {
    uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
    uint32_t m = __vmaxu2(a, b);
    return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Max over the CTA; every thread gets the result.
__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* red) {
    v = warp_max(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
    return warp_max(v);
}

// Lets the dependent encode pass (launched with programmatic stream
// serialization) start its launch now; it waits for this grid's completion
// before reading the partials.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisite_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads) amax_partial_kernel(const uint4* __restrict__ x, int64_t n8,
                                                                uint32_t* __restrict__ partial) {
    __shared__ uint32_t red[32];
    launch_dependents();
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n8; i += 8 * stride) {
        uint4 v[8];                                   // eight 16-byte loads in flight per thread
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = i + u * stride < n8 ? __ldg(x + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 8; ++u) m = max(m, absmax8_bits(v[u]));
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

// ---- cluster helpers (distributed shared memory) ----
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// The tensor amax (as bf16 magnitude bits), either from the workspace
// partials or, in the fused cluster launch, computed here.
template <bool FUSED>
__device__ __forceinline__ uint32_t tensor_amax_bits(const uint16_t* __restrict__ x, int64_t n,
                                                     const uint32_t* __restrict__ partial, int n_partial,
                                                     uint32_t* red, uint32_t* xchg) {
    if constexpr (FUSED) {
        const uint32_t rank = cluster_rank(), csize = cluster_size();
        const int64_t n8 = n / 8;
        const int64_t lo = n8 * rank / csize, hi = n8 * (rank + 1) / csize;
        const uint4* x4 = reinterpret_cast<const uint4*>(x);
        uint32_t m = 0;
        const int64_t bd = blockDim.x;
        int64_t i = lo + threadIdx.x;
        for (; i + 3 * bd < hi; i += 4 * bd) {
            const uint4 a = __ldg(x4 + i), b = __ldg(x4 + i + bd), c = __ldg(x4 + i + 2 * bd), d = __ldg(x4 + i + 3 * bd);
            m = max(m, max(max(absmax8_bits(a), absmax8_bits(b)), max(absmax8_bits(c), absmax8_bits(d))));
        }
        for (; i < hi; i += bd) m = max(m, absmax8_bits(__ldg(x4 + i)));
        m = block_max(m, red);
        if (threadIdx.x == 0) *xchg = m;
        cluster_sync();                              // every CTA's partial is visible
        uint32_t all = 0;
        if (threadIdx.x < csize) all = ld_dsmem_u32(smem_u32(xchg), threadIdx.x);
        all = block_max(all, red);
        cluster_sync();                              // no CTA leaves while others read it
        return all;
    } else {
        wait_prerequisite_grid();
        uint32_t m = 0;
        for (int i = threadIdx.x; i < n_partial; i += blockDim.x) m = max(m, partial[i]);
        return block_max(m, red);
    }
}

// ------------------------------------------------------- per-block encode ----
// The MX block encode (amax, scale, encode words) lives in mx_encode.cuh.

// Store one MX block's words at codes + row offset + block offset (24 or 32 bytes).
template <int FMT, bool CONT = false>
__device__ __forceinline__ void mx_store_words(uint8_t* __restrict__ dst, const uint32_t (&w)[8]) {
    if constexpr (FMT == kE4M3 || CONT) {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        reinterpret_cast<uint2*>(dst)[0] = make_uint2(w[0], w[1]);
        reinterpret_cast<uint2*>(dst)[1] = make_uint2(w[2], w[3]);
        reinterpret_cast<uint2*>(dst)[2] = make_uint2(w[4], w[5]);
    }
}

// One nvfp4 block (16 values: two uint4) from its amax bits: the ue4m3 scale
// (round to nearest of fl(fl(amax*gs)/6)) and two words of eight e2m1 codes.
__device__ __forceinline__ void nvfp4_encode_block(uint4 v0, uint4 v1, uint32_t amax_bits, float gs, uint32_t& sc,
                                                   uint32_t& w0, uint32_t& w1) {
    sc = 0;
    w0 = w1 = 0;
    if (gs == 0.0f) return;
    const float t = __fmul_rn(bf16_bits_to_f32(amax_bits), gs);
    sc = cvt_x2<kE4M3>(__fdiv_rn(t, kMaxE2M1), 0.0f) & 0xFFu;
    if (sc == 0) return;
    const float inv = __fdiv_rn(gs, e4m3_to_f32(sc));
    const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float lo, hi;
        mul2_rn(bf16_lo(in[i]), bf16_hi(in[i]), inv, lo, hi);
        c[i] = cvt_e2m1x2(lo, hi);
    }
    w0 = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    w1 = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
}

// ------------------------------------------------------------------ MX ----
// Each lane owns whole blocks: block slot gb = (row, b) of a row-major grid of
// pad128(M) x pad4(K/32) slots, walked with a grid-wide stride so every lane
// gets the same work (+-1 block).  A block is 32 values = 64 contiguous bytes
// (four 16-byte loads whose sectors the neighbouring lanes' loads share); the
// block amax needs no shuffle and the scale math is done once per 32 values.
template <int FMT, bool FUSED, bool CONT = false>
__global__ void __launch_bounds__(kEncThreads)
quant_mx_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, const uint32_t* __restrict__ partial,
                int n_partial, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                float* __restrict__ s_global, uint32_t* __restrict__ err) {
    __shared__ uint32_t red[32];
    __shared__ uint32_t xchg;
    const uint32_t am_bits = tensor_amax_bits<FUSED>(x, M * K, partial, n_partial, red, &xchg);
    const float amax = bf16_bits_to_f32(am_bits);
    const float gs = amax > 0.0f ? __fdiv_rn(gs_numerator(FMT), amax) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    const int lane = threadIdx.x & 31;
    const uint32_t nb = (uint32_t)(K / 32);
    const int64_t cpd4 = pad_to(nb, 4) / 4;
    const uint32_t nbp = (uint32_t)pad_to(nb, 4);                 // block slots per row
    const uint32_t total = (uint32_t)pad_to(M, 128) * nbp;        // a multiple of 128
    const int64_t row_bytes = FMT == kE4M3 || CONT ? K : 3 * K / 4;
    const uint32_t stride = gridDim.x * blockDim.x;

    for (uint32_t gb = blockIdx.x * blockDim.x + threadIdx.x; gb < total; gb += stride) {
        const uint32_t r = gb / nbp, b = gb - r * nbp;
        const bool valid = r < M && b < nb;
        uint4 v[4];
        if (valid && BSQ_IN_BUFFER(err, kChkQuantX, (int64_t)r * K + 32 * (int64_t)b, 32, M * K)) {
            const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)r * K + 32 * (int64_t)b);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
        }
        uint32_t ue;
        float inv;
        mx_block_scale<FMT>(absmax32_bits(v), gs, ue, inv);
        uint32_t w[8];
        mx_encode_words<FMT, CONT>(v, inv, w);
        constexpr int kBlockBytes = FMT == kE4M3 || CONT ? 32 : 24;
        if (valid && BSQ_IN_BUFFER(err, kChkQuantCodes, (int64_t)r * row_bytes + kBlockBytes * (int64_t)b, kBlockBytes,
                                   M * row_bytes))
            mx_store_words<FMT, CONT>(codes + (int64_t)r * row_bytes + kBlockBytes * (int64_t)b, w);
        // four consecutive blocks' scale bytes (four consecutive lanes, the same
        // row: nbp % 4 == 0) -> one 32-bit store
        const uint32_t s4 = ue | (__shfl_down_sync(0xFFFFFFFFu, ue, 1) << 8) |
                            (__shfl_down_sync(0xFFFFFFFFu, ue, 2) << 16) | (__shfl_down_sync(0xFFFFFFFFu, ue, 3) << 24);
        if ((lane & 3) == 0 && BSQ_IN_BUFFER(err, kChkQuantScales, swz_offset(r, b, cpd4), 4, (int64_t)total))
            *reinterpret_cast<uint32_t*>(scales + swz_offset(r, b, cpd4)) = s4;
    }
}

// --------------------------------------------------------------- nvfp4 ----
// Each lane owns two consecutive blocks of 16 (32 values, 64 contiguous bytes,
// four output words), pair slots walked with a grid-wide stride as above.
template <bool FUSED>
__global__ void __launch_bounds__(kEncThreads)
quant_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, const uint32_t* __restrict__ partial,
                   int n_partial, uint32_t* __restrict__ codes, uint8_t* __restrict__ scales,
                   float* __restrict__ s_global, uint32_t* __restrict__ err) {
    __shared__ uint32_t red[32];
    __shared__ uint32_t xchg;
    const uint32_t am_bits = tensor_amax_bits<FUSED>(x, M * K, partial, n_partial, red, &xchg);
    const float amax = bf16_bits_to_f32(am_bits);
    const float gs = amax > 0.0f ? __fdiv_rn(kMaxE4M3 * kMaxE2M1, amax) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    const int lane = threadIdx.x & 31;
    const uint32_t nb = (uint32_t)(K / 16);
    const int64_t cpd4 = pad_to(nb, 4) / 4;
    const uint32_t npp = (uint32_t)pad_to(nb, 4) / 2;             // block-pair slots per row
    const uint32_t total = (uint32_t)pad_to(M, 128) * npp;        // a multiple of 256
    const uint32_t stride = gridDim.x * blockDim.x;

    for (uint32_t gp = blockIdx.x * blockDim.x + threadIdx.x; gp < total; gp += stride) {
        const uint32_t r = gp / npp;
        const uint32_t b0 = 2 * (gp - r * npp);                    // this lane's first block
        uint32_t sb[2];
        uint32_t word[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t b = b0 + h;
            const bool valid = r < M && b < nb;
            uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
            if (valid && BSQ_IN_BUFFER(err, kChkQuantX, (int64_t)r * K + 16 * (int64_t)b, 16, M * K)) {
                const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)r * K + 16 * (int64_t)b);
                v0 = __ldg(src);
                v1 = __ldg(src + 1);
            }
            uint32_t w0, w1;
            nvfp4_encode_block(v0, v1, max(absmax8_bits(v0), absmax8_bits(v1)), gs, sb[h], w0, w1);
            word[2 * h] = w0;
            word[2 * h + 1] = w1;
        }
        const int64_t woff = (int64_t)r * (K / 8) + 2 * (int64_t)b0;       // in 32-bit words
        if (r < M && b0 < nb && BSQ_IN_BUFFER(err, kChkQuantCodes, woff, b0 + 1 < nb ? 4 : 2, M * (K / 8))) {
            uint32_t* dst = codes + woff;                                     // 8-byte aligned rows (K % 16 == 0)
            *reinterpret_cast<uint2*>(dst) = make_uint2(word[0], word[1]);
            if (b0 + 1 < nb) *reinterpret_cast<uint2*>(dst + 2) = make_uint2(word[2], word[3]);
        }
        // blocks b0, b0+1 from this lane and b0+2, b0+3 from the next -> one 32-bit store
        const uint32_t s2 = sb[0] | (sb[1] << 8);
        const uint32_t s4 = s2 | (__shfl_down_sync(0xFFFFFFFFu, s2, 1) << 16);
        if ((lane & 1) == 0 && BSQ_IN_BUFFER(err, kChkQuantScales, swz_offset(r, b0, cpd4), 4, 2 * (int64_t)total))
            *reinterpret_cast<uint32_t*>(scales + swz_offset(r, b0, cpd4)) = s4;
    }
}

// -------------------------------------------------------------- one pass ----
// The whole quantizer in ONE cooperative launch, one CTA per SM: each CTA
// bulk-copies its contiguous slice of x into shared memory in 32 KiB chunks
// (one mbarrier each) and reduces the amax of every chunk as it lands,
// publishes its partial maximum, waits at a bounded grid barrier for every
// CTA's partial, then encodes its slice from shared memory.  x is read from
// HBM once.  Used when every slice fits in one SM's shared memory; larger
// tensors take the two-pass path above.
//
// Work unit ("slot") = 32 consecutive values of a row = 64 bytes of x: one MX
// block, or two nvfp4 blocks.  Slots run over a padded grid of pad128(M) rows x
// `slots_per_row` (pad4(K/32) for MX, pad4(K/16)/2 for nvfp4), so the padding of
// the scale buffer is written too; CTA ranges are multiples of four slots, so
// a group of four scale bytes never straddles two CTAs.
//
// Grid barrier: CTA c stores its partial in workspace word 1 + c, then adds to
// the control block's arrival counter with release semantics; after the counter
// reads G (acquire) every partial is visible.  One polling thread per CTA keeps
// the counter's line uncontended.  Each CTA then counts itself out; the last
// one out zeroes both counters for the next call.
//
// Several tensors can share one launch (and one barrier): each owns a range of
// CTAs sized to its share of the slots, and reduces only its own partials, so
// every tensor gets its own amax and s_global exactly as in a launch of its own.
constexpr int kOneThreads = 1024;
constexpr int kOneIters = 4;           // slots per thread: a slice holds <= 4 * kOneThreads slots
constexpr uint32_t kChunkBytes = 32768;
constexpr int kMaxChunks = 8;

constexpr int kMaxBatch = 8;          // tensors per one-pass launch
// One-pass control block, after the partials in the caller's workspace:
// [0..1] a 64-bit magic (valid: the counters below are consistent), [2] arrivals,
// [3] departures.  Every call leaves it valid with both counters zero, so no
// launch needs a memset; a workspace that does not hold the magic (a fresh
// allocation, or one left by a call that timed out) is initialized by CTA 0
// while the other CTAs wait for the magic.
constexpr int kCtlWord = kMaxPartials;
constexpr int kCtlWords = 64;
constexpr uint64_t kCtlMagic = 0x7F4A7C159E3779B9ull;

struct OneTensor {
    const uint16_t* x;
    int64_t M, K;
    void* codes;
    uint8_t* scales;
    float* s_global;
    uint32_t slots_per_row; // padded
    uint32_t slots_per_cta; // a multiple of 4
};

// A batch of tensors in one launch: tensor i owns CTAs [first_cta[i], first_cta[i+1]).
struct OnePassArgs {
    OneTensor t[kMaxBatch];
    uint32_t first_cta[kMaxBatch + 1];
    int n;
    uint32_t* ws;           // [1 + cta] partial maxima; [kCtlWord ..] the control block
    uint32_t* err;
};

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint32_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(uint32_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// swz_offset in 32-bit arithmetic (scale buffers of the one-pass path are < 4 GiB).
__device__ __forceinline__ uint32_t swz_offset32(uint32_t row, uint32_t block, uint32_t cpd4) {
    return ((((row >> 7) * cpd4 + (block >> 2)) * 32 + (row & 31)) * 4 + ((row >> 5) & 3)) * 4 + (block & 3);
}

// Flat index (in 64-byte units of x) of slot s: rows have K/32 units of data.
__device__ __forceinline__ int64_t slot_data_index(uint32_t s, uint32_t spr, int64_t units_row, int64_t M) {
    const int64_t r = s / spr, b = s - r * spr;
    if (r >= M) return M * units_row;
    return r * units_row + (b < units_row ? b : units_row);
}

// The 64-byte unit at shared address `addr` (unit index u within the slice).
// The four 16-byte pieces are read starting at piece (u >> 1) & 3, so the eight
// lanes of a quarter-warp reading consecutive units hit eight different bank
// groups, then put back in order with two select stages.
__device__ __forceinline__ void load_unit(uint32_t addr, uint32_t u, uint4 (&v)[4]) {
    const uint32_t rot = (u >> 1) & 3;
    uint4 w[4], t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = lds128(addr + 16 * ((j + rot) & 3));   // w[j] = piece (j + rot) & 3
    const bool r1 = rot & 1, r2 = rot & 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) t[k] = r1 ? w[(k + 3) & 3] : w[k];              // t[k] = piece (k + (rot & 2)) & 3
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = r2 ? t[(k + 2) & 3] : t[k];              // v[k] = piece k
}

// TRANSPOSE (every row a whole number of 4-slot groups, so slot and 64-byte
// unit offsets coincide): step 2 also rewrites each warp's 32 units piece-major
// (unit u's piece j at (u/32)*2048 + j*512 + (u%32)*16), so step 3 reads its
// pieces in order, conflict-free, with no un-rotation.
template <int FMT, bool TRANSPOSE>   // FMT: kE3M2 / kE2M3 / kE4M3, or kNvfp4
__global__ void __launch_bounds__(kOneThreads, 1) quant_onepass_kernel(const __grid_constant__ OnePassArgs args) {
    extern __shared__ __align__(128) uint8_t slice[];
    __shared__ uint64_t bar[kMaxChunks];
    __shared__ uint32_t red[32];
    __shared__ int abort_flag;
    int ti = 0;
    while (ti + 1 < args.n && blockIdx.x >= args.first_cta[ti + 1]) ++ti;
    const OneTensor a = args.t[ti];                          // this CTA's tensor
    const uint32_t G = gridDim.x;                            // the grid barrier counts every CTA
    const uint32_t p0 = args.first_cta[ti], Gt = args.first_cta[ti + 1] - p0;
    const uint32_t c = blockIdx.x - p0;                      // CTA index within the tensor
    const int lane = threadIdx.x & 31;
    const int64_t units_row = a.K / 32;
    const uint32_t spr = a.slots_per_row;
    const uint32_t total = (uint32_t)pad_to(a.M, 128) * spr;
    const uint32_t s0 = min(total, c * a.slots_per_cta), s1 = min(total, s0 + a.slots_per_cta);
    const int64_t f0 = slot_data_index(s0, spr, units_row, a.M), f1 = slot_data_index(s1, spr, units_row, a.M);
    const uint32_t bytes = (uint32_t)((f1 - f0) * 64);
    const uint32_t n_chunks = (bytes + kChunkBytes - 1) / kChunkBytes;
    const uint32_t slice_addr = smem_u32(slice);

    // 1. the slice -> shared memory, one bulk copy and one barrier per chunk
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (uint32_t k = 0; k < n_chunks; ++k) mbar_init(smem_u32(bar + k), 1);
        fence_mbar_init();
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x) + f0 * 64;
        for (uint32_t k = 0; k < n_chunks; ++k) {
            const uint32_t off = k * kChunkBytes, n = min(kChunkBytes, bytes - off);
            if (BSQ_IN_BUFFER(args.err, kChkQuantX, f0 * 64 + off, n, a.M * a.K * 2)) {
                mbar_arrive_expect_tx(smem_u32(bar + k), n);
                bulk_load(slice_addr + off, src + off, n, smem_u32(bar + k));
            } else {
                mbar_arrive(smem_u32(bar + k));   // skipped: the chunk completes with no bytes
            }
        }
        // control block: initialize it (CTA 0) or wait for it if it is not valid
        uint32_t* ctl = args.ws + kCtlWord;
        if (ld_acquire_u64(ctl) != kCtlMagic) {
            if (blockIdx.x == 0) {
                ctl[2] = 0;
                ctl[3] = 0;
                st_release_u64(ctl, kCtlMagic);          // the zeroed counters before the magic
            } else {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_u64(ctl) != kCtlMagic) {
                    if (globaltimer() - t0 > kWaitLimitNs) {
                        atomicCAS(args.err, 0u, (uint32_t)kErrQuantBarrier);
                        abort_flag = 1;
                        break;
                    }
                }
            }
        }
    }
    __syncthreads();

    // 2. block maxima of this thread's slots as their chunks land, kept in
    //    registers for step 3 (the slot -> thread map is the same there), and the
    //    slice amax.  Iteration it covers units < (it + 1) * kOneThreads.
    //    Thread t's slot in iteration it: s = s0 + it * kOneThreads + t, at
    //    (row, slot-in-row) stepped without a division per iteration.
    const uint32_t s_t = s0 + threadIdx.x;
    const uint32_t r_t = s_t / spr, b_t = s_t - r_t * spr;
    const uint32_t dr = kOneThreads / spr, db = kOneThreads - dr * spr;
    uint32_t bm[kOneIters];   // MX: the block's amax bits; nvfp4: block 2b | block 2b+1 << 16
    uint32_t m = 0;
    {
        uint32_t r = r_t, b = b_t, waited = 0;
#pragma unroll
        for (int it = 0; it < kOneIters; ++it) {
            const uint32_t need = min(n_chunks, ((uint32_t)(it + 1) * kOneThreads * 64 + kChunkBytes - 1) / kChunkBytes);
            while (waited < need) {
                if (!mbar_wait(smem_u32(bar + waited), 0, args.err, &abort_flag, kErrQuantLoad)) {
                    waited = n_chunks;                           // aborted: results are void
                    break;
                }
                ++waited;
            }
            bm[it] = 0;
            const uint32_t s = s_t + it * kOneThreads;
            const bool have = s < s1 && r < a.M && b < units_row;
            const uint32_t u = have ? (uint32_t)(r * units_row + b - f0) : 0u;
            const uint32_t rot = (u >> 1) & 3;
            uint4 pv[4];
            if (have) {
                const uint32_t addr = slice_addr + 64 * u;
                uint32_t mb[2] = {0, 0};
#pragma unroll
                for (int j = 0; j < 4; ++j) {          // rotated piece order: conflict-free
                    const uint32_t pc = (j + rot) & 3;
                    pv[j] = lds128(addr + 16 * pc);
                    const uint32_t x8 = absmax8_bits(pv[j]);
                    if (pc < 2) mb[0] = max(mb[0], x8); else mb[1] = max(mb[1], x8);
                }
                bm[it] = FMT == kNvfp4 ? (mb[0] | (mb[1] << 16)) : max(mb[0], mb[1]);
                m = max(m, max(mb[0], mb[1]));
            }
            if constexpr (TRANSPOSE) {
                __syncwarp();                          // the warp's 32 units are read
                if (have) {
                    const uint32_t gbase = slice_addr + (u >> 5) * 2048 + (u & 31) * 16;
#pragma unroll
                    for (int j = 0; j < 4; ++j) sts128(gbase + ((j + rot) & 3) * 512, pv[j]);
                }
            }
            b += db;
            r += dr;
            if (b >= spr) { b -= spr; ++r; }
        }
    }
    m = block_max(m, red);

    // publish, then the bounded grid barrier: thread 0 stores the partial and
    // counts itself in with a release add, then polls the counter
    if (threadIdx.x == 0) {
        uint32_t* ctl = args.ws + kCtlWord;
        args.ws[1 + blockIdx.x] = m;
#ifdef BSQ_TEST_BARRIER_SKIP_LAST_CTA
        // test build only: the grid's last CTA never counts itself in, so every
        // CTA's bounded wait below runs out (no copy or TMEM is in flight here)
        if (blockIdx.x + 1 != gridDim.x)
#endif
        red_release_add_u32(ctl + 2, 1u);
        if (ld_acquire_u32(ctl + 2) < G) {
            const uint64_t t0 = globaltimer();
            while (ld_acquire_u32(ctl + 2) < G) {
                if (abort_flag || globaltimer() - t0 > kWaitLimitNs) {
                    atomicCAS(args.err, 0u, (uint32_t)kErrQuantBarrier);
                    abort_flag = 1;
                    break;
                }
            }
        }
        if (abort_flag) {
            st_release_u64(ctl, 0ull);                   // the next call re-initializes the block
        } else if (atomicAdd(ctl + 3, 1u) == G - 1) {    // last one out: zero the counters
            ctl[2] = 0;
            ctl[3] = 0;
        }
    }
    __syncthreads();
    launch_dependents();       // the next kernel (a GEMM) may launch; it waits for this grid's results
    uint32_t am = 0;
    if (threadIdx.x < Gt) am = ld_relaxed_u32(args.ws + 1 + p0 + threadIdx.x);   // this tensor's CTAs
    am = block_max(am, red);   // (its barriers also publish abort_flag)
    if (abort_flag) {
        // leave no bulk copy in flight into this CTA's shared memory
        if (threadIdx.x == 0)
            for (uint32_t k = 0; k < n_chunks; ++k) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(bar + k), 0) && globaltimer() - t0 < kWaitLimitNs) {
                }
            }
        return;
    }
    const float amax = bf16_bits_to_f32(am);
    constexpr float kNum = FMT == kNvfp4 ? kMaxE4M3 * kMaxE2M1 : gs_numerator(FMT == kNvfp4 ? 0 : FMT);
    const float gs = amax > 0.0f ? __fdiv_rn(kNum, amax) : 0.0f;
    if (c == 0 && threadIdx.x == 0) *a.s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    // 3. encode from shared memory, one slot per lane
    const int64_t row_bytes = FMT == kNvfp4 ? a.K / 2 : FMT == kE4M3 ? a.K : 3 * a.K / 4;
    const uint32_t nb = FMT == kNvfp4 ? (uint32_t)(a.K / 16) : (uint32_t)units_row;
    const uint32_t cpd4 = (nb + 3) / 4;
    uint32_t r = r_t, b = b_t;
#pragma unroll
    for (int it = 0; it < kOneIters; ++it) {
        const uint32_t s = s_t + it * kOneThreads;
        if (s0 + it * kOneThreads >= s1) break;                     // uniform across the CTA
        const bool in_range = s < s1;
        const bool valid = in_range && r < a.M && b < units_row;
        uint4 v[4];
        if (valid) {
            const uint32_t u = (uint32_t)(r * units_row + b - f0);
            if constexpr (TRANSPOSE) {
                const uint32_t gbase = slice_addr + (u >> 5) * 2048 + (u & 31) * 16;
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = lds128(gbase + j * 512);
            } else {
                load_unit(slice_addr + 64 * u, u, v);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = make_uint4(0, 0, 0, 0);
        }
        uint8_t* const row_codes = static_cast<uint8_t*>(a.codes) + (int64_t)r * row_bytes;
        constexpr int kUnitBytes = FMT == kNvfp4 ? 16 : FMT == kE4M3 ? 32 : 24;   // code bytes of one slot
        const bool store = valid && BSQ_IN_BUFFER(args.err, kChkQuantCodes, (int64_t)r * row_bytes + kUnitBytes * b,
                                                  kUnitBytes, a.M * row_bytes);
        const int64_t scale_bytes = pad_to(a.M, 128) * 4 * (int64_t)cpd4;
        if constexpr (FMT == kNvfp4) {
            uint32_t sb0, sb1, w[4];
            nvfp4_encode_block(v[0], v[1], bm[it] & 0xFFFFu, gs, sb0, w[0], w[1]);
            nvfp4_encode_block(v[2], v[3], bm[it] >> 16, gs, sb1, w[2], w[3]);
            if (store) *reinterpret_cast<uint4*>(row_codes + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
            const uint32_t s2 = sb0 | (sb1 << 8);
            const uint32_t s4 = s2 | (__shfl_down_sync(0xFFFFFFFFu, s2, 1) << 16);
            if (in_range && (lane & 1) == 0 &&
                BSQ_IN_BUFFER(args.err, kChkQuantScales, swz_offset32(r, 2 * b, cpd4), 4, scale_bytes))
                *reinterpret_cast<uint32_t*>(a.scales + swz_offset32(r, 2 * b, cpd4)) = s4;
        } else {
            uint32_t ue, w[8];
            float inv;
            mx_block_scale<FMT>(bm[it], gs, ue, inv);
            mx_encode_words<FMT>(v, inv, w);
            if (store) mx_store_words<FMT>(row_codes + kUnitBytes * b, w);
            const uint32_t s4 = ue | (__shfl_down_sync(0xFFFFFFFFu, ue, 1) << 8) |
                                (__shfl_down_sync(0xFFFFFFFFu, ue, 2) << 16) | (__shfl_down_sync(0xFFFFFFFFu, ue, 3) << 24);
            if (in_range && (lane & 3) == 0 &&
                BSQ_IN_BUFFER(args.err, kChkQuantScales, swz_offset32(r, b, cpd4), 4, scale_bytes))
                *reinterpret_cast<uint32_t*>(a.scales + swz_offset32(r, b, cpd4)) = s4;
        }
        b += db;
        r += dr;
        if (b >= spr) { b -= spr; ++r; }
    }
}

// ------------------------------------------------- fused activation ----
// Activation + MX quantize (b12x _lib/fp6.py relu2_quantize_grouped_mxfp6_torch,
// silu_mul_quantize_grouped_mxfp6_torch): the activation is evaluated in f32
// and rounded to bf16 (the input dtype), and that tensor -- never stored, unless
// the caller asks for it -- goes through the same amax / scale / encode steps.
//   ReLU^2:    max(x, 0)^2 (one f32 product, exact), x [M, K].
//   SiLU * up: fl(fl(g / fl(1 + exp(-g))) * u), x [M, 2K] = gate | up per row;
//              exp is CUDA's expf (not a fast approximation).
// Two launch shapes as for the plain MX quantizer: one 16-CTA cluster for small
// tensors, else an amax pass over the activated values into the workspace and
// an encode pass that evaluates the activation again (same instructions, same
// bits) -- the input is read twice, the activated tensor never.
constexpr int kActRelu2 = 1, kActSiluMul = 2;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float relu2_f32(float v) {
    const float r = v > 0.0f ? v : 0.0f;
    return __fmul_rn(r, r);
}
__device__ __forceinline__ float silu_mul_f32(float g, float u) {
    const float e = expf(-g);
    const float d = __fadd_rn(1.0f, e);
    return __fmul_rn(__fdiv_rn(g, d), u);
}
// Activated outputs (row, col .. col + 7) as bf16 bits; K = output columns,
// M = rows of x (for the device bounds checks).
template <int ACT>
__device__ __forceinline__ uint4 act8(const uint16_t* __restrict__ x, int64_t row, int64_t col, int64_t M, int64_t K,
                                      uint32_t* err) {
    if (!BSQ_IN_BUFFER(err, kChkQuantX, row * (ACT == kActRelu2 ? K : 2 * K) + col, ACT == kActRelu2 ? 8 : K + 8,
                       M * (ACT == kActRelu2 ? K : 2 * K)))
        return make_uint4(0, 0, 0, 0);
    if constexpr (ACT == kActRelu2) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + row * K + col));
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(relu2_f32(bf16_lo(in[i])), relu2_f32(bf16_hi(in[i])));
        return make_uint4(o[0], o[1], o[2], o[3]);
    } else {
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(x + row * 2 * K + col));
        const uint4 uv = __ldg(reinterpret_cast<const uint4*>(x + row * 2 * K + K + col));
        const uint32_t g[4] = {gv.x, gv.y, gv.z, gv.w}, u[4] = {uv.x, uv.y, uv.z, uv.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack_bf16x2(silu_mul_f32(bf16_lo(g[i]), bf16_lo(u[i])), silu_mul_f32(bf16_hi(g[i]), bf16_hi(u[i])));
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}
// Max |activated| over output units [lo, hi) (a unit = 8 outputs of one row).
template <int ACT>
__device__ __forceinline__ uint32_t act_absmax_units(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t lo,
                                                     int64_t hi, int64_t step, uint32_t* err) {
    const int64_t upr = K / 8;
    uint32_t m = 0;
    for (int64_t i = lo; i < hi; i += step) {
        const int64_t row = i / upr, col = 8 * (i - row * upr);
        m = max(m, absmax8_bits(act8<ACT>(x, row, col, M, K, err)));
    }
    return m;
}

template <int ACT>
__global__ void __launch_bounds__(kThreads) act_amax_partial_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                                    int64_t K, uint32_t* __restrict__ partial,
                                                                    uint32_t* __restrict__ err) {
    __shared__ uint32_t red[32];
    launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    uint32_t m = act_absmax_units<ACT>(x, M, K, (int64_t)blockIdx.x * kThreads + threadIdx.x, M * K / 8, stride, err);
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

template <int FMT, bool FUSED, int ACT>
__global__ void __launch_bounds__(kEncThreads)
quant_mx_act_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, const uint32_t* __restrict__ partial,
                    int n_partial, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                    float* __restrict__ s_global, uint16_t* __restrict__ act_out, uint32_t* __restrict__ err) {
    __shared__ uint32_t red[32];
    __shared__ uint32_t xchg;
    uint32_t am_bits;
    if constexpr (FUSED) {
        const uint32_t rank = cluster_rank(), csize = cluster_size();
        const int64_t n8 = M * K / 8;
        const int64_t lo = n8 * rank / csize, hi = n8 * (rank + 1) / csize;
        uint32_t m = act_absmax_units<ACT>(x, M, K, lo + threadIdx.x, hi, blockDim.x, err);
        m = block_max(m, red);
        if (threadIdx.x == 0) xchg = m;
        cluster_sync();                              // every CTA's partial is visible
        uint32_t all = 0;
        if (threadIdx.x < csize) all = ld_dsmem_u32(smem_u32(&xchg), threadIdx.x);
        am_bits = block_max(all, red);
        cluster_sync();                              // no CTA leaves while others read it
    } else {
        wait_prerequisite_grid();
        uint32_t m = 0;
        for (int i = threadIdx.x; i < n_partial; i += blockDim.x) m = max(m, partial[i]);
        am_bits = block_max(m, red);
    }
    const float amax = bf16_bits_to_f32(am_bits);
    const float gs = amax > 0.0f ? __fdiv_rn(gs_numerator(FMT), amax) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    const int lane = threadIdx.x & 31;
    const uint32_t nb = (uint32_t)(K / 32);
    const int64_t cpd4 = pad_to(nb, 4) / 4;
    const uint32_t nbp = (uint32_t)pad_to(nb, 4);
    const uint32_t total = (uint32_t)pad_to(M, 128) * nbp;
    const int64_t row_bytes = FMT == kE4M3 ? K : 3 * K / 4;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t gb = blockIdx.x * blockDim.x + threadIdx.x; gb < total; gb += stride) {
        const uint32_t r = gb / nbp, b = gb - r * nbp;
        const bool valid = r < M && b < nb;
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = valid ? act8<ACT>(x, r, 32 * (int64_t)b + 8 * i, M, K, err) : make_uint4(0, 0, 0, 0);
        if (act_out && valid && BSQ_IN_BUFFER(err, kChkQuantAct, (int64_t)r * K + 32 * (int64_t)b, 32, M * K)) {
            uint4* dst = reinterpret_cast<uint4*>(act_out + (int64_t)r * K + 32 * (int64_t)b);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = v[i];
        }
        uint32_t ue;
        float inv;
        mx_block_scale<FMT>(absmax32_bits(v), gs, ue, inv);
        uint32_t w[8];
        mx_encode_words<FMT>(v, inv, w);
        constexpr int kBlockBytes = FMT == kE4M3 ? 32 : 24;
        if (valid && BSQ_IN_BUFFER(err, kChkQuantCodes, (int64_t)r * row_bytes + kBlockBytes * (int64_t)b, kBlockBytes,
                                   M * row_bytes))
            mx_store_words<FMT>(codes + (int64_t)r * row_bytes + kBlockBytes * (int64_t)b, w);
        const uint32_t s4 = ue | (__shfl_down_sync(0xFFFFFFFFu, ue, 1) << 8) |
                            (__shfl_down_sync(0xFFFFFFFFu, ue, 2) << 16) | (__shfl_down_sync(0xFFFFFFFFu, ue, 3) << 24);
        if ((lane & 3) == 0 && BSQ_IN_BUFFER(err, kChkQuantScales, swz_offset(r, b, cpd4), 4, (int64_t)total))
            *reinterpret_cast<uint32_t*>(scales + swz_offset(r, b, cpd4)) = s4;
    }
}

// ------------------------------------------------------------- grouped ----
// Grouped (MoE) MX quantizer (b12x _lib/fp6.py quantize_grouped_mxfp6_torch):
// x [G, R, C]; group g's first row_counts[g] rows are quantized with the
// caller's global scale gs[g] (no amax pass: the scale is given), the other
// rows get zero codes and zero scales.  Codes are group-major [G, R, row_bytes]
// and every group has its own swizzled scale buffer of pad128(R) x pad4(C/32)
// bytes, so each group is an operand the (grouped) GEMM reads in place.  One
// lane per 32-value block slot over all groups' padded grids.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
quant_grouped_mx_kernel(const uint16_t* __restrict__ x, int64_t G, int64_t R, int64_t C,
                        const int32_t* __restrict__ row_counts, const float* __restrict__ gs_in,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ s_global,
                        uint32_t* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = C / 32, nbp = pad_to(nb, 4), cpd4 = nbp / 4;
    const int64_t per_group = pad_to(R, 128) * nbp;           // = the group's scale bytes
    const int64_t row_bytes = FMT == kE4M3 ? C : 3 * C / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t gb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gb < G * per_group; gb += stride) {
        const int64_t g = gb / per_group, rem = gb - g * per_group;
        const int64_t r = rem / nbp, b = rem - r * nbp;
        int64_t rc = __ldg(row_counts + g);
        rc = rc < 0 ? 0 : (rc > R ? R : rc);
        const float gs = __ldg(gs_in + g);
        if (rem == 0) s_global[g] = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;
        const bool live = r < rc && b < nb;
        uint4 v[4];
        if (live && BSQ_IN_BUFFER(err, kChkQuantX, (g * R + r) * C + 32 * b, 32, G * R * C)) {
            const uint4* src = reinterpret_cast<const uint4*>(x + ((g * R + r) * C + 32 * b));
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
        }
        uint32_t ue;
        float inv;
        mx_block_scale<FMT>(absmax32_bits(v), gs, ue, inv);
        if (!live) { ue = 0; inv = 0.0f; }
        uint32_t w[8];
        mx_encode_words<FMT>(v, inv, w);
        constexpr int kBlockBytes = FMT == kE4M3 ? 32 : 24;
        if (r < R && b < nb &&
            BSQ_IN_BUFFER(err, kChkQuantCodes, (g * R + r) * row_bytes + kBlockBytes * b, kBlockBytes, G * R * row_bytes))
            mx_store_words<FMT>(codes + (g * R + r) * row_bytes + kBlockBytes * b, w);
        const uint32_t s4 = ue | (__shfl_down_sync(0xFFFFFFFFu, ue, 1) << 8) |
                            (__shfl_down_sync(0xFFFFFFFFu, ue, 2) << 16) | (__shfl_down_sync(0xFFFFFFFFu, ue, 3) << 24);
        if ((lane & 3) == 0 &&
            BSQ_IN_BUFFER(err, kChkQuantScales, g * per_group + swz_offset(r, b, cpd4), 4, G * per_group))
            *reinterpret_cast<uint32_t*>(scales + g * per_group + swz_offset(r, b, cpd4)) = s4;
    }
}

// ------------------------------------------------------------ launching ----
// One cluster of kFusedCluster CTAs (16 needs the non-portable opt-in; a
// device that refuses it gets 8).
template <typename KernelT, typename... Args>
cudaError_t launch_cluster(KernelT kernel, cudaStream_t s, Args... args) {
    int csize = kFusedCluster;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        (void)cudaGetLastError();
        csize = 8;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    for (;; csize = 8) {
        cfg.gridDim = dim3(csize, 1, 1);
        attr[0].val.clusterDim.x = csize;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
        if (e == cudaSuccess || csize == 8) return e;
        (void)cudaGetLastError();
    }
}

// The encode pass, launched so that it may start while the amax pass runs; it
// waits (griddepcontrol.wait) for the amax pass before reading the partials.
template <typename KernelT, typename... Args>
cudaError_t launch_dependent_n(KernelT kernel, int grid, int threads, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
template <typename KernelT, typename... Args>
cudaError_t launch_dependent(KernelT kernel, int grid, cudaStream_t s, Args... args) {
    return launch_dependent_n(kernel, grid, kEncThreads, s, args...);
}

// The amax pass runs at full occupancy (8 x 256 threads per SM, <= 32
// registers) with eight loads in flight per thread; the encode pass runs one
// 1024-thread CTA per SM (a short launch ramp) walking whole blocks.
constexpr int kAmaxPerSm = 8;

int encode_grid(const DeviceInfo* info, int64_t M, int64_t K) {
    const int64_t slots = pad_to(M, 128) * pad_to(K / 32, 4);      // lanes needed (MX; nvfp4 pairs: the same)
    int64_t g = (slots + kEncThreads - 1) / kEncThreads;
    const int64_t cap = (int64_t)info->num_sms;
    return (int)(g < cap ? g : cap);
}

int amax_grid(const DeviceInfo* info, int64_t n) {
    int64_t g = (n / 8 + 8 * kThreads - 1) / (8 * kThreads);       // up to eight loads per thread
    int64_t cap = (int64_t)info->num_sms * kAmaxPerSm;
    if (cap > kMaxPartials) cap = kMaxPartials;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}


// The one-pass launch for a batch of tensors, when every CTA's slice fits its
// SM's shared memory.  CTAs are dealt to the tensors one at a time, each to the
// tensor whose CTAs currently carry the most slots.  Returns false (nothing
// launched) when the batch does not fit one launch.
template <int FMT>
bool onepass_batch(const DeviceInfo* info, const QTensor* ts, int n, uint32_t* ws, size_t ws_bytes, cudaStream_t s,
                   bsq_status* st) {
    const int G = info->num_sms;
    if (n < 1 || n > kMaxBatch || n > G || !ws || G > kOneThreads) return false;
    if ((size_t)(kCtlWord + 4) * sizeof(uint32_t) > ws_bytes || G + 1 > kCtlWord) return false;
    int64_t slots[kMaxBatch], spr[kMaxBatch];
    int cnt[kMaxBatch];
    bool transpose = true;                 // every row a whole number of 4-slot groups
    for (int i = 0; i < n; ++i) {
        if (ts[i].K % 32 != 0) return false;
        spr[i] = FMT == kNvfp4 ? pad_to(ts[i].K / 16, 4) / 2 : pad_to(ts[i].K / 32, 4);
        transpose = transpose && spr[i] == ts[i].K / 32;
        slots[i] = pad_to(ts[i].M, 128) * spr[i];
        if (slots[i] >= (int64_t(1) << 31)) return false;
        cnt[i] = 1;
    }
    for (int extra = G - n; extra > 0; --extra) {
        int best = 0;
        for (int i = 1; i < n; ++i)
            if (slots[i] * cnt[best] > slots[best] * cnt[i]) best = i;   // slots/cnt, compared exactly
        ++cnt[best];
    }
    int64_t slice_max = (int64_t)info->max_smem_optin - 1024;
    if (slice_max > (int64_t)kMaxChunks * kChunkBytes) slice_max = (int64_t)kMaxChunks * kChunkBytes;
    OnePassArgs a;
    int64_t per_max = 0;
    uint32_t first = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t per = pad_to((slots[i] + cnt[i] - 1) / cnt[i], 4);
        if (per * 64 > slice_max || per > (int64_t)kOneIters * kOneThreads) return false;
        per_max = per > per_max ? per : per_max;
        OneTensor& t = a.t[i];
        t.x = ts[i].x; t.M = ts[i].M; t.K = ts[i].K; t.codes = ts[i].codes; t.scales = ts[i].scales;
        t.s_global = ts[i].s_global; t.slots_per_row = (uint32_t)spr[i]; t.slots_per_cta = (uint32_t)per;
        a.first_cta[i] = first;
        first += (uint32_t)cnt[i];
    }
    for (int i = n; i <= kMaxBatch; ++i) a.first_cta[i] = first;
    for (int i = n; i < kMaxBatch; ++i) a.t[i] = a.t[0];
    a.n = n; a.ws = ws; a.err = info->err;
    // the piece-major rewrite works on whole 32-unit groups
    const size_t smem = (size_t)(transpose ? pad_to(per_max * 64, 2048) : per_max * 64);
    if ((int64_t)smem > slice_max) return false;
    static std::once_flag once[64];
    static bool ok_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::call_once(once[dev], [&] {
        ok_dev[dev] = cudaFuncSetAttribute(quant_onepass_kernel<FMT, false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           info->max_smem_optin - 1024) == cudaSuccess &&
                      cudaFuncSetAttribute(quant_onepass_kernel<FMT, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           info->max_smem_optin - 1024) == cudaSuccess;
    });
    if (!ok_dev[dev]) { (void)cudaGetLastError(); return false; }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(first, 1, 1);
    cfg.blockDim = dim3(kOneThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once: the grid barrier can complete
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = transpose ? cudaLaunchKernelEx(&cfg, quant_onepass_kernel<FMT, true>, a)
                                    : cudaLaunchKernelEx(&cfg, quant_onepass_kernel<FMT, false>, a);
    if (e != cudaSuccess) { (void)cudaGetLastError(); *st = BSQ_ERR_CUDA; return true; }
    count_launch(FMT == kNvfp4 ? BSQ_KERNEL_QUANT_NVFP4 : BSQ_KERNEL_QUANT_MX);
    *st = BSQ_OK;
    return true;
}

template <int FMT>
bool onepass_try(const DeviceInfo* info, const uint16_t* x, int64_t M, int64_t K, void* codes, uint8_t* scales,
                 float* s_global, uint32_t* ws, size_t ws_bytes, cudaStream_t s, bsq_status* st) {
    const QTensor t = {x, M, K, codes, scales, s_global};
    return onepass_batch<FMT>(info, &t, 1, ws, ws_bytes, s, st);
}
}  // namespace

size_t quantize_batch_workspace_bytes() { return (size_t)(kMaxPartials + kCtlWords) * sizeof(uint32_t); }

bsq_status quantize_batch_launch(const QTensor* ts, int n, int fmt, void* ws, size_t ws_bytes, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    if (!ws || ws_bytes < quantize_batch_workspace_bytes()) return BSQ_ERR_WORKSPACE;
    if (!aligned16(ws)) return BSQ_ERR_MISALIGNED;
    uint32_t* partial = static_cast<uint32_t*>(ws);
    bool done = false;
    switch (fmt) {
    case kE3M2: done = onepass_batch<kE3M2>(info, ts, n, partial, ws_bytes, s, &st); break;
    case kE2M3: done = onepass_batch<kE2M3>(info, ts, n, partial, ws_bytes, s, &st); break;
    case kE4M3: done = onepass_batch<kE4M3>(info, ts, n, partial, ws_bytes, s, &st); break;
    default: done = onepass_batch<kNvfp4>(info, ts, n, partial, ws_bytes, s, &st); break;
    }
    if (done) return st;
    // too large for one launch: the tensors one after another on the stream
    for (int i = 0; i < n; ++i) {
        const QTensor& t = ts[i];
        st = fmt == kNvfp4 ? quantize_nvfp4_launch(t.x, t.M, t.K, static_cast<uint32_t*>(t.codes), t.scales,
                                                   t.s_global, ws, ws_bytes, s)
                           : quantize_mx_launch(t.x, t.M, t.K, fmt, static_cast<uint8_t*>(t.codes), t.scales,
                                                t.s_global, ws, ws_bytes, s);
        if (st != BSQ_OK) return st;
    }
    return BSQ_OK;
}

int amax_partials_launch(const uint16_t* x, int64_t n, uint32_t* partial, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return -1;
    const int n_partial = amax_grid(info, n);
    amax_partial_kernel<<<n_partial, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), n / 8, partial);
    count_launch(BSQ_KERNEL_AMAX);
    return launch_status() == BSQ_OK ? n_partial : -1;
}

size_t quantize_workspace_bytes(int64_t M, int64_t K) {
    if (M * K <= kFusedMaxElems) return 0;
    return (size_t)(kMaxPartials + kCtlWords) * sizeof(uint32_t);
}

bsq_status quantize_mx_launch(const uint16_t* x, int64_t M, int64_t K, int fmt, uint8_t* codes,
                              uint8_t* scales, float* s_global, void* ws, size_t ws_bytes, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const bool fused = M * K <= kFusedMaxElems;
    uint32_t* partial = static_cast<uint32_t*>(ws);
    int n_partial = 0;
    if (!fused) {
        if (!ws || ws_bytes < quantize_workspace_bytes(M, K)) return BSQ_ERR_WORKSPACE;
        if (!aligned16(ws)) return BSQ_ERR_MISALIGNED;
        bool done = false;
        switch (fmt) {
        case kE3M2: done = onepass_try<kE3M2>(info, x, M, K, codes, scales, s_global, partial, ws_bytes, s, &st); break;
        case kE2M3: done = onepass_try<kE2M3>(info, x, M, K, codes, scales, s_global, partial, ws_bytes, s, &st); break;
        default: done = onepass_try<kE4M3>(info, x, M, K, codes, scales, s_global, partial, ws_bytes, s, &st); break;
        }
        if (done) return st;
        n_partial = amax_grid(info, M * K);
        amax_partial_kernel<<<n_partial, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), M * K / 8, partial);
        count_launch(BSQ_KERNEL_AMAX);
        if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    const int grid = encode_grid(info, M, K);
#define BSQ_QMX(F)                                                                                          \
    if (fused)                                                                                              \
        e = launch_cluster(quant_mx_kernel<F, true>, s, x, M, K, (const uint32_t*)nullptr, 0, codes, scales, \
                           s_global, info->err);                                                            \
    else                                                                                                    \
        e = launch_dependent(quant_mx_kernel<F, false>, grid, s, x, M, K, (const uint32_t*)partial, n_partial,   \
                             codes, scales, s_global, info->err);
    switch (fmt) {
    case kE3M2: BSQ_QMX(kE3M2); break;
    case kE2M3: BSQ_QMX(kE2M3); break;
    default: BSQ_QMX(kE4M3); break;
    }
#undef BSQ_QMX
    count_launch(fused ? BSQ_KERNEL_QUANT_SMALL : BSQ_KERNEL_QUANT_MX);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    return launch_status();
}


template <int FMT, int ACT>
bsq_status quantize_mx_act_fmt(const DeviceInfo* info, const uint16_t* x, int64_t M, int64_t K, uint8_t* codes,
                               uint8_t* scales, float* s_global, uint16_t* act_out, uint32_t* partial,
                               cudaStream_t s) {
    // The activation (an expf and a division per value for SiLU) dominates these
    // passes, so both spread it thinly: about one 8-value unit (amax pass) or
    // one 32-value block (encode pass) per thread, up to 4 x 256-thread CTAs per SM.
    const bool fused = M * K <= kFusedMaxElems;
    int n_partial = 0;
    const int64_t cap = (int64_t)info->num_sms * 4;
    if (!fused) {
        const int64_t units = M * K / 8;
        int64_t g = (units + kThreads - 1) / kThreads;
        if (g > cap) g = cap;
        if (g > kMaxPartials) g = kMaxPartials;
        n_partial = (int)g;
        act_amax_partial_kernel<ACT><<<n_partial, kThreads, 0, s>>>(x, M, K, partial, info->err);
        count_launch(BSQ_KERNEL_AMAX);
        if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    }
    cudaError_t e;
    if (fused) {
        e = launch_cluster(quant_mx_act_kernel<FMT, true, ACT>, s, x, M, K, (const uint32_t*)nullptr, 0, codes,
                           scales, s_global, act_out, info->err);
    } else {
        const int64_t slots = pad_to(M, 128) * pad_to(K / 32, 4);
        int64_t g = (slots + kThreads - 1) / kThreads;
        if (g > cap) g = cap;
        e = launch_dependent_n(quant_mx_act_kernel<FMT, false, ACT>, (int)g, kThreads, s, x, M, K,
                               (const uint32_t*)partial, n_partial, codes, scales, s_global, act_out, info->err);
    }
    count_launch(fused ? BSQ_KERNEL_QUANT_SMALL : BSQ_KERNEL_QUANT_MX);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    return launch_status();
}

bsq_status quantize_mx_act_launch(const uint16_t* x, int64_t M, int64_t K, int act, int fmt, uint8_t* codes,
                                  uint8_t* scales, float* s_global, uint16_t* act_out, void* ws, size_t ws_bytes,
                                  cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    uint32_t* partial = static_cast<uint32_t*>(ws);
    if (M * K > kFusedMaxElems) {
        if (!ws || ws_bytes < quantize_workspace_bytes(M, K)) return BSQ_ERR_WORKSPACE;
        if (!aligned16(ws)) return BSQ_ERR_MISALIGNED;
    }
#define BSQ_QACT(F)                                                                                           \
    return act == kActRelu2 ? quantize_mx_act_fmt<F, kActRelu2>(info, x, M, K, codes, scales, s_global, act_out, \
                                                                 partial, s)                                  \
                            : quantize_mx_act_fmt<F, kActSiluMul>(info, x, M, K, codes, scales, s_global, act_out, \
                                                                   partial, s);
    switch (fmt) {
    case kE3M2: BSQ_QACT(kE3M2);
    case kE2M3: BSQ_QACT(kE2M3);
    default: BSQ_QACT(kE4M3);
    }
#undef BSQ_QACT
}

// fp6 codes one per byte: the cluster launch for small tensors, else the amax
// pass and the encode pass (the one-pass kernel writes packed codes only).
bsq_status quantize_mx_containers_launch(const uint16_t* x, int64_t M, int64_t K, int fmt, uint8_t* codes,
                                         uint8_t* scales, float* s_global, void* ws, size_t ws_bytes,
                                         cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const bool fused = M * K <= kFusedMaxElems;
    uint32_t* partial = static_cast<uint32_t*>(ws);
    int n_partial = 0;
    if (!fused) {
        if (!ws || ws_bytes < quantize_workspace_bytes(M, K)) return BSQ_ERR_WORKSPACE;
        if (!aligned16(ws)) return BSQ_ERR_MISALIGNED;
        n_partial = amax_grid(info, M * K);
        amax_partial_kernel<<<n_partial, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), M * K / 8, partial);
        count_launch(BSQ_KERNEL_AMAX);
        if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    }
    cudaError_t e;
    const int grid = encode_grid(info, M, K);
#define BSQ_QCONT(F)                                                                                            \
    if (fused)                                                                                                  \
        e = launch_cluster(quant_mx_kernel<F, true, true>, s, x, M, K, (const uint32_t*)nullptr, 0, codes, scales, \
                           s_global, info->err);                                                                \
    else                                                                                                        \
        e = launch_dependent(quant_mx_kernel<F, false, true>, grid, s, x, M, K, (const uint32_t*)partial,      \
                             n_partial, codes, scales, s_global, info->err);
    if (fmt == kE3M2) { BSQ_QCONT(kE3M2); } else { BSQ_QCONT(kE2M3); }
#undef BSQ_QCONT
    count_launch(fused ? BSQ_KERNEL_QUANT_SMALL : BSQ_KERNEL_QUANT_MX);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    return launch_status();
}

bsq_status quantize_grouped_mx_launch(const uint16_t* x, int64_t G, int64_t R, int64_t C, const int32_t* row_counts,
                                      const float* gs, int fmt, uint8_t* codes, uint8_t* scales, float* s_global,
                                      cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const int64_t slots = G * pad_to(R, 128) * pad_to(C / 32, 4);
    int64_t grid = (slots + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)info->num_sms * 8;
    if (grid > cap) grid = cap;
    if (fmt == kE3M2)
        quant_grouped_mx_kernel<kE3M2><<<(unsigned)grid, kThreads, 0, s>>>(x, G, R, C, row_counts, gs, codes, scales, s_global,
                                                                        info->err);
    else if (fmt == kE2M3)
        quant_grouped_mx_kernel<kE2M3><<<(unsigned)grid, kThreads, 0, s>>>(x, G, R, C, row_counts, gs, codes, scales, s_global,
                                                                        info->err);
    else
        quant_grouped_mx_kernel<kE4M3><<<(unsigned)grid, kThreads, 0, s>>>(x, G, R, C, row_counts, gs, codes, scales, s_global,
                                                                        info->err);
    count_launch(BSQ_KERNEL_QUANT_MX);
    return launch_status();
}

bsq_status quantize_nvfp4_launch(const uint16_t* x, int64_t M, int64_t K, uint32_t* codes, uint8_t* scales,
                                 float* s_global, void* ws, size_t ws_bytes, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    const bool fused = M * K <= kFusedMaxElems;
    uint32_t* partial = static_cast<uint32_t*>(ws);
    int n_partial = 0;
    if (!fused) {
        if (!ws || ws_bytes < quantize_workspace_bytes(M, K)) return BSQ_ERR_WORKSPACE;
        if (!aligned16(ws)) return BSQ_ERR_MISALIGNED;
        if (onepass_try<kNvfp4>(info, x, M, K, codes, scales, s_global, partial, ws_bytes, s, &st)) return st;
        n_partial = amax_grid(info, M * K);
        amax_partial_kernel<<<n_partial, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), M * K / 8, partial);
        count_launch(BSQ_KERNEL_AMAX);
        if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    if (fused)
        e = launch_cluster(quant_nvfp4_kernel<true>, s, x, M, K, (const uint32_t*)nullptr, 0, codes, scales,
                           s_global, info->err);
    else
        e = launch_dependent(quant_nvfp4_kernel<false>, encode_grid(info, M, K), s, x, M, K,
                             (const uint32_t*)partial, n_partial, codes, scales, s_global, info->err);
    count_launch(fused ? BSQ_KERNEL_QUANT_SMALL : BSQ_KERNEL_QUANT_NVFP4);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    return launch_status();
}

}  // namespace bsq

// ---------------------------------------------------------------------------
// Allocation-free variant of bsq_quantize_mxfp6.
//
// Some callers cannot allocate device memory on this path: a plugin whose host
// framework owns all device memory and forbids cudaMalloc while it executes, or
// a latency-critical loop where an allocation (and the synchronization it
// implies) is not acceptable.  This entry point keeps the large-tensor path's
// scratch -- the per-CTA partial maxima of the amax pass -- in a file-scope
// device array instead of a caller-provided workspace.
//
// The array (kMaxPartials words, 8 KiB) lives on every GPU that loads the
// library until the process exits.  Its device address is looked up once per
// device, with that device current, by the first call on that device (host
// code cannot use the array's name as a device address).  Every call shares
// the array: the amax pass rewrites each slot the encode pass reads, so nothing
// needs clearing, but two calls whose kernels overlap on the GPU (for example
// on two streams) race on it.
// ---------------------------------------------------------------------------
namespace bsq {
namespace {

static __device__ __align__(256) uint32_t g_noalloc_partials[kMaxPartials];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
std::atomic<uint32_t*> g_noalloc_ptr[kNoallocMaxDevices];

// Device address of the scratch array on the current device (nullptr on error).
// Only a successful lookup is kept: a lookup that failed (for instance one
// attempted during a stream capture) is tried again by the next call.
uint32_t* noalloc_scratch() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return nullptr;
    uint32_t* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_noalloc_partials) == cudaSuccess) {
            p = static_cast<uint32_t*>(q);
            g_noalloc_ptr[dev].store(p, std::memory_order_release);
        } else {
            (void)cudaGetLastError();
        }
    }
    return p;
}

}  // namespace
}  // namespace bsq

extern "C" BSQ_API bsq_status bsq_quantize_mxfp6_noalloc(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt,
                                                        uint8_t* codes, uint8_t* scales, float* s_global,
                                                        cudaStream_t stream) {
    using namespace bsq;
    if (!x || !codes || !scales || !s_global || (fmt != BSQ_E3M2 && fmt != BSQ_E2M3 && fmt != BSQ_E4M3))
        return BSQ_ERR_INVALID_ARG;
    if (M < 1 || K < 32 || K % 32 || M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return BSQ_ERR_MISALIGNED;
    if (M * K <= kFusedMaxElems)    // the single cluster launch needs no scratch
        return quantize_mx_launch(x, M, K, fmt, codes, scales, s_global, nullptr, 0, stream);
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    uint32_t* scratch = noalloc_scratch();
    if (!scratch) return BSQ_ERR_CUDA;
    const int n_partial = amax_grid(info, M * K);
    if (n_partial > kMaxPartials) return BSQ_ERR_UNSUPPORTED;   // more partial maxima than the array holds
    amax_partial_kernel<<<n_partial, kThreads, 0, stream>>>(reinterpret_cast<const uint4*>(x), M * K / 8, scratch);
    count_launch(BSQ_KERNEL_AMAX);
    if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    const int grid = encode_grid(info, M, K);
    switch (fmt) {
    case BSQ_E3M2:
        quant_mx_kernel<kE3M2, false><<<grid, kEncThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global,
                                                                         info->err);
        break;
    case BSQ_E2M3:
        quant_mx_kernel<kE2M3, false><<<grid, kEncThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global,
                                                                         info->err);
        break;
    default:
        quant_mx_kernel<kE4M3, false><<<grid, kEncThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global,
                                                                         info->err);
        break;
    }
    count_launch(BSQ_KERNEL_QUANT_MX);
    return launch_status();
}
