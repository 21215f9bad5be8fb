// bsq_device.cuh -- device-side building blocks shared by the libbsq kernels:
// format constants, IEEE-exact scale steps, the hardware minifloat conversions,
// and thin inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsq {

// ---------------------------------------------------------------- constants --
// Largest finite magnitudes (b12x _lib/fp6.py constants; e2m1's is 6).
constexpr float kMaxE3M2 = 28.0f;
constexpr float kMaxE2M3 = 7.5f;
constexpr float kMaxE4M3 = 448.0f;
constexpr float kMaxE2M1 = 6.0f;

enum Fmt : int { kE3M2 = 0, kE2M3 = 1, kE4M3 = 2 };

__host__ __device__ constexpr float fmt_max(int fmt) {
    return fmt == kE3M2 ? kMaxE3M2 : fmt == kE2M3 ? kMaxE2M3 : kMaxE4M3;
}
// mx_gs_numerator: 448 * fmt_max (exact in f32).
__host__ __device__ constexpr float gs_numerator(int fmt) { return kMaxE4M3 * fmt_max(fmt); }

__host__ __device__ inline int64_t pad_to(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Byte offset of the scale of (row, block) in the swizzled block-scale buffer
// (b12x _lib/fp6.py, mxfp6_swizzled_scale_offset).
__host__ __device__ inline int64_t swz_offset(int64_t row, int64_t block, int64_t cpd4) {
    return ((((row >> 7) * cpd4 + (block >> 2)) * 32 + (row & 31)) * 4 + ((row >> 5) & 3)) * 4 + (block & 3);
}

// ------------------------------------------------------------- error word ---
// Site ids written into the device error word by bounded waits.
enum ErrorSite : uint32_t {
    kErrNone = 0,
    kErrGemmProducer = 0x101,
    kErrGemmMma = 0x102,
    kErrGemmEpilogue = 0x103,
    kErrGemmDrain = 0x104,
    kErrGemvProducer = 0x201,
    kErrGemvConsumer = 0x202,
    kErrQuantLoad = 0x301,
    kErrQuantBarrier = 0x302,
};

// ------------------------------------------------------ device bounds checks --
// A build with -DBSQ_DEVICE_CHECKS checks every global store of these kernels,
// and every global load addressed from a row and a column (TMA tensor-map
// loads are bounded by their maps, the amax passes' linear loads by the element
// count of their loop), against the extent of its buffer as the call's sizes
// give it.  An access that leaves the buffer is skipped; the first one is
// recorded in the error word as kCheckFlag | site << 24 | (its offset & 0xFFFFFF),
// the offset in the buffer's own units.  Timeout sites never have bit 31 set.
// Without the flag BSQ_IN_BUFFER is the constant true and nothing is compiled.
constexpr uint32_t kCheckFlag = 0x80000000u;
enum CheckSite : uint32_t {
    kChkQuantX = 0x01,        // quantizer: load of x
    kChkQuantCodes = 0x02,    // quantizer: store of codes
    kChkQuantScales = 0x03,   // quantizer: store of block scales
    kChkQuantAct = 0x04,      // fused activation quantizer: store of the activation
    kChkGemmY = 0x11,         // GEMM: store of Y
    kChkGemvX = 0x21,         // GEMV: load of x
    kChkGemvW = 0x22,         // GEMV: load of weight codes
    kChkGemvScales = 0x23,    // GEMV: load of weight block scales
    kChkGemvY = 0x24,         // GEMV: store of y
    kChkDequantIn = 0x31,     // dequantizer: load of codes or scales
    kChkDequantOut = 0x32,    // dequantizer: store of the output
};

#ifdef BSQ_DEVICE_CHECKS
// A test build may tighten one site's extent by one unit (BSQ_TEST_CHECK_TIGHT_SITE):
// the last in-bounds access of that site is then recorded and skipped.
#ifdef BSQ_TEST_CHECK_TIGHT_SITE
constexpr uint32_t kTightSite = BSQ_TEST_CHECK_TIGHT_SITE;
#else
constexpr uint32_t kTightSite = 0;
#endif
// [off, off + n) inside [0, size)?  Records the first failure (see above).
__device__ __forceinline__ bool in_buffer(uint32_t* err, uint32_t site, int64_t off, int64_t n, int64_t size) {
    if (site == kTightSite) size -= 1;
    if (off >= 0 && n >= 0 && off + n <= size) return true;
    atomicCAS(err, 0u, kCheckFlag | (site << 24) | ((uint32_t)off & 0xFFFFFFu));
    return false;
}
#define BSQ_IN_BUFFER(err, site, off, n, size) ::bsq::in_buffer((err), (site), (off), (n), (size))
#else
#define BSQ_IN_BUFFER(err, site, off, n, size) true
#endif

// Wall-clock bound of every spin-wait in these kernels (ns).  A test build
// may set a shorter one (BSQ_WAIT_LIMIT_NS) to make a wait run out quickly.
#ifndef BSQ_WAIT_LIMIT_NS
#define BSQ_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitLimitNs = BSQ_WAIT_LIMIT_NS;

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------- scale arithmetic -----
// fp6_block_ue8m0_exact (b12x _lib/fp6.py): ratio = fl(fl(amax_b*gs)/fmt_max);
// byte = exponent field + (mantissa != 0), clamped to [0, 255]; 0 if ratio <= 0.
__device__ __forceinline__ uint32_t ue8m0_from_block_max(float amax_b, float gs, float fmax) {
    float t = __fmul_rn(amax_b, gs);
    float ratio = __fdiv_rn(t, fmax);
    uint32_t b = __float_as_uint(ratio);
    int32_t r = (int32_t)((b >> 23) & 0xFF) + ((b & 0x7FFFFF) != 0 ? 1 : 0);
    r = r < 0 ? 0 : (r > 255 ? 255 : r);
    return ratio <= 0.0f ? 0u : (uint32_t)r;
}

// ue8m0_output_scale_exact: gs * 2^(127-ue), the power built from its bits
// (exponent field 254-ue); 0 when ue == 0.
__device__ __forceinline__ float ue8m0_output_scale(uint32_t ue, float gs) {
    float p = __uint_as_float((uint32_t)(254 - (int32_t)ue) << 23);
    float r = __fmul_rn(p, gs);
    return ue == 0 ? 0.0f : r;
}

// ------------------------------------------------ hardware conversions -----
// cvt.rn.satfinite.<fmt>x2.f32 d, hi, lo: RNE with saturation to the largest
// finite value; `lo` lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == kE3M2)
        asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else if constexpr (FMT == kE2M3)
        asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e2m1 codes (lo in bits 0..3, hi in bits 4..7).
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Exact decode of an e4m3 byte (low byte of c) to f32, via the hardware's
// e4m3x2 -> f16x2 conversion (exact) and f16 -> f32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(c & 0xFF)));
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((uint16_t)(h2 & 0xFFFF)));
    return f;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// f32 -> bf16 round to nearest even, NaN kept a NaN (hardware cvt).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// One 32-byte global store (a full sector; sm_100's 256-bit vector
// store); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7) : "memory");
}

// two values, round to nearest even: lo in bits 0-15, hi in bits 16-31
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------ addresses ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// --------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  On timeout
// records `site` in *err (first writer wins), sets *abort and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicCAS(err, 0u, site);
            *abort = 1;
            return false;
        }
    }
}

// -------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(map) : "memory");
}

// ---------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
// Copy one 32-row x 16-byte block-scale group from shared memory into four
// TMEM columns, replicated to all four lane quarters.
__device__ __forceinline__ void tc_cp_scales(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p; }"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf4nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p; }"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
// ---- CTA pair (cta_group::2): the two CTAs of a cluster whose ranks differ in
// bit 0.  Established on GB300 against a CPU product: the allocation is
// collective (one warp of each CTA issues it and both receive the same
// columns); rank 0 issues the MMA, which reads A's 128 rows and B's N half
// from each CTA's shared memory at the same offsets and writes each CTA's
// 128 accumulator rows into its own TMEM; each CTA's TMEM holds A's scale
// factors for its own rows and B's for all N rows of the MMA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
// Arrive on the barrier at the same offset in both CTAs of the pair once this
// thread's earlier pair MMAs have completed.
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(bar), "h"((uint16_t)3) : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8f6f4_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                     uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p; }"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf4nvf4_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                     uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p; }"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
// Arrive on a barrier given by its shared::cluster address, e.g. the peer
// CTA's copy of a barrier (mapa).  Default semantics (release at CTA scope):
// a cluster-scope release would make the arriving warp wait for the SM's
// outstanding memory operations, serializing a pipeline's relay.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Registers r[0..N) -> TMEM columns [col, col + N) of the warp's 32 lanes
// (lane l of the warp writes its own TMEM lane); N a multiple of 4.
template <int N>
__device__ __forceinline__ void tc_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N % 4 == 0, "columns in groups of four");
    if constexpr (N % 16 == 0) {
#pragma unroll
        for (int c = 0; c < N; c += 16)
            asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                         "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                         :: "r"(taddr + c), "r"(r[c]), "r"(r[c + 1]), "r"(r[c + 2]), "r"(r[c + 3]), "r"(r[c + 4]),
                            "r"(r[c + 5]), "r"(r[c + 6]), "r"(r[c + 7]), "r"(r[c + 8]), "r"(r[c + 9]),
                            "r"(r[c + 10]), "r"(r[c + 11]), "r"(r[c + 12]), "r"(r[c + 13]), "r"(r[c + 14]),
                            "r"(r[c + 15]) : "memory");
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 4)
            asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                         :: "r"(taddr + c), "r"(r[c]), "r"(r[c + 1]), "r"(r[c + 2]), "r"(r[c + 3]) : "memory");
    }
}

// 32 lanes x 32 columns of 32-bit words: thread i of the warp gets its lane's
// 32 consecutive columns.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and stride
// byte offsets (>> 4), the fixed version bit 46, and the layout (swizzle) mode
// in bits 61..63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

}  // namespace bsq
