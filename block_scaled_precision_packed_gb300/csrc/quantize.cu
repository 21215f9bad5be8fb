// quantize.cu -- bf16 -> MX (e3m2 / e2m3 / e4m3, UE8M0 per 32) and
// bf16 -> nvfp4 (e2m1, ue4m3 per 16) block quantizers.
//
// Recipe: b12x _lib/fp6.py, quantize_grouped_mxfp6_torch with the exact scale
// steps of fp6_block_ue8m0_exact / ue8m0_output_scale_exact and the per-block
// quantizers quantize_block_fp6_*_fast (the nvfp4 variant is the same recipe
// with e2m1's maximum and a round-to-nearest e4m3 block scale).
//
// Two launch shapes:
//  * small tensors (M*K <= kFusedMaxElems): ONE launch of a thread-block
//    cluster.  Each CTA reduces the amax of its slice, the cluster exchanges
//    the partial maxima through distributed shared memory, and every CTA then
//    encodes its share of the blocks.  No workspace, no grid-wide wait.
//  * large tensors: an amax pass writes per-CTA partial maxima to the caller's
//    workspace; the encode pass reduces them (a few hundred words) in every
//    CTA and encodes.  The second read of x is normally an L2 hit.
//
// Encode mapping: one warp per (row, 1024-element chunk).  Lane l loads 16
// contiguous bytes (8 values) per step j (0..3) at element 256*j + 8*l, so a
// warp's load is 512 contiguous bytes.  A 32-value MX block is four lanes (a
// quad), a 16-value nvfp4 block two lanes; the block amax is a shuffle.
#include <cstdio>
#include <mutex>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPartials = 1024;
constexpr int64_t kFusedMaxElems = 262144;   // 512 KB of bf16
constexpr int kFusedCluster = 8;

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
    v = lane < kWarps ? red[lane] : 0u;
    return warp_max(v);
}

__global__ void __launch_bounds__(kThreads) amax_partial_kernel(const uint4* __restrict__ x, int64_t n8,
                                                                uint32_t* __restrict__ partial) {
    __shared__ uint32_t red[32];
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n8; i += (int64_t)gridDim.x * kThreads)
        m = max(m, absmax8_bits(__ldg(x + i)));
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
        for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) m = max(m, absmax8_bits(__ldg(x4 + i)));
        m = block_max(m, red);
        if (threadIdx.x == 0) *xchg = m;
        cluster_sync();                              // every CTA's partial is visible
        uint32_t all = 0;
        if (threadIdx.x < csize) all = ld_dsmem_u32(smem_u32(xchg), threadIdx.x);
        all = block_max(all, red);
        cluster_sync();                              // no CTA leaves while others read it
        return all;
    } else {
        uint32_t m = 0;
        for (int i = threadIdx.x; i < n_partial; i += kThreads) m = max(m, __ldg(partial + i));
        return block_max(m, red);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------------ MX ----
template <int FMT, bool FUSED>
__global__ void __launch_bounds__(kThreads)
quant_mx_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, const uint32_t* __restrict__ partial,
                int n_partial, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                float* __restrict__ s_global) {
    __shared__ uint32_t red[32];
    __shared__ uint32_t xchg;
    const uint32_t am_bits = tensor_amax_bits<FUSED>(x, M * K, partial, n_partial, red, &xchg);
    const float amax = bf16_bits_to_f32(am_bits);
    const float gs = amax > 0.0f ? __fdiv_rn(gs_numerator(FMT), amax) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    constexpr float fmax = fmt_max(FMT);
    const int lane = threadIdx.x & 31, q = lane & 3;
    const int64_t nb = K / 32, cpd4 = pad_to(nb, 4) / 4;
    const int64_t chunks = (K + 1023) / 1024, rows_pad = pad_to(M, 128);
    const int64_t n_tasks = rows_pad * chunks;
    const int64_t row_bytes = FMT == kE4M3 ? K : 3 * K / 4;
    const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;

    for (int64_t task = warp0; task < n_tasks; task += nwarps) {
        const int64_t r = task / chunks, c = task % chunks;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t e = c * 1024 + j * 256 + lane * 8;
            const bool valid = r < M && e < K;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) v = __ldg(reinterpret_cast<const uint4*>(x + r * K + e));
            uint32_t mb = absmax8_bits(v);
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            const float amax_b = bf16_bits_to_f32(mb);
            uint32_t ue = 0;
            float inv = 0.0f;
            if (gs != 0.0f) {
                ue = ue8m0_from_block_max(amax_b, gs, fmax);
                inv = ue8m0_output_scale(ue, gs);
            }
            // eight codes, one byte each (zero when inv == 0)
            uint32_t p0 = 0, p1 = 0, p2 = 0, p3 = 0;
            if (inv != 0.0f) {
                p0 = cvt_x2<FMT>(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv));
                p1 = cvt_x2<FMT>(__fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv));
                p2 = cvt_x2<FMT>(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv));
                p3 = cvt_x2<FMT>(__fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv));
            }
            if constexpr (FMT == kE4M3) {
                if (valid) {
                    const uint64_t w = (uint64_t)(p0 | (p1 << 16)) | ((uint64_t)(p2 | (p3 << 16)) << 32);
                    *reinterpret_cast<uint64_t*>(codes + r * row_bytes + e) = w;
                }
            } else {
                // 8 codes -> 48 bits, c_i at bit 6i (four-in-three rule, twice)
                const uint64_t v48 = (uint64_t)(p0 & 0x3F) | ((uint64_t)((p0 >> 8) & 0x3F) << 6) |
                                     ((uint64_t)(p1 & 0x3F) << 12) | ((uint64_t)((p1 >> 8) & 0x3F) << 18) |
                                     ((uint64_t)(p2 & 0x3F) << 24) | ((uint64_t)((p2 >> 8) & 0x3F) << 30) |
                                     ((uint64_t)(p3 & 0x3F) << 36) | ((uint64_t)((p3 >> 8) & 0x3F) << 42);
                const uint64_t nxt = __shfl_down_sync(0xFFFFFFFFu, v48, 1);
                // the quad's 24 bytes as three 8-byte words
                const uint64_t out = q == 0 ? (v48 | (nxt << 48))
                                   : q == 1 ? ((v48 >> 16) | (nxt << 32))
                                            : ((v48 >> 32) | (nxt << 16));
                if (valid && q < 3) {
                    const int64_t b = e / 32;
                    *reinterpret_cast<uint64_t*>(codes + r * row_bytes + b * 24 + q * 8) = out;
                }
            }
            // four consecutive blocks' scale bytes -> one 32-bit store
            const uint32_t s4 = ue | (__shfl_down_sync(0xFFFFFFFFu, ue, 4) << 8) |
                                (__shfl_down_sync(0xFFFFFFFFu, ue, 8) << 16) |
                                (__shfl_down_sync(0xFFFFFFFFu, ue, 12) << 24);
            const int64_t b0 = c * 32 + j * 8 + (lane >> 2);
            if ((lane & 15) == 0 && b0 < nb)
                *reinterpret_cast<uint32_t*>(scales + swz_offset(r, b0, cpd4)) = s4;
        }
    }
}

// --------------------------------------------------------------- nvfp4 ----
template <bool FUSED>
__global__ void __launch_bounds__(kThreads)
quant_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, const uint32_t* __restrict__ partial,
                   int n_partial, uint32_t* __restrict__ codes, uint8_t* __restrict__ scales,
                   float* __restrict__ s_global) {
    __shared__ uint32_t red[32];
    __shared__ uint32_t xchg;
    const uint32_t am_bits = tensor_amax_bits<FUSED>(x, M * K, partial, n_partial, red, &xchg);
    const float amax = bf16_bits_to_f32(am_bits);
    const float gs = amax > 0.0f ? __fdiv_rn(kMaxE4M3 * kMaxE2M1, amax) : 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = gs != 0.0f ? __fdiv_rn(1.0f, gs) : 0.0f;

    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 16, cpd4 = pad_to(nb, 4) / 4;
    const int64_t chunks = (K + 1023) / 1024, rows_pad = pad_to(M, 128);
    const int64_t n_tasks = rows_pad * chunks;
    const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;

    for (int64_t task = warp0; task < n_tasks; task += nwarps) {
        const int64_t r = task / chunks, c = task % chunks;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t e = c * 1024 + j * 256 + lane * 8;
            const bool valid = r < M && e < K;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) v = __ldg(reinterpret_cast<const uint4*>(x + r * K + e));
            uint32_t mb = absmax8_bits(v);
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            const float amax_b = bf16_bits_to_f32(mb);
            uint32_t sb = 0;
            float inv = 0.0f;
            if (gs != 0.0f) {
                const float t = __fmul_rn(amax_b, gs);
                const float ratio = __fdiv_rn(t, kMaxE2M1);
                sb = cvt_x2<kE4M3>(ratio, 0.0f) & 0xFFu;
                if (sb != 0) inv = __fdiv_rn(gs, e4m3_to_f32(sb));
            }
            uint32_t word = 0;
            if (inv != 0.0f) {
                word = cvt_e2m1x2(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv)) |
                       (cvt_e2m1x2(__fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv)) << 8) |
                       (cvt_e2m1x2(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv)) << 16) |
                       (cvt_e2m1x2(__fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv)) << 24);
            }
            if (valid) codes[r * (K / 8) + e / 8] = word;
            const uint32_t s4 = sb | (__shfl_down_sync(0xFFFFFFFFu, sb, 2) << 8) |
                                (__shfl_down_sync(0xFFFFFFFFu, sb, 4) << 16) |
                                (__shfl_down_sync(0xFFFFFFFFu, sb, 6) << 24);
            const int64_t b0 = c * 64 + j * 16 + (lane >> 1);
            if ((lane & 7) == 0 && b0 < nb)
                *reinterpret_cast<uint32_t*>(scales + swz_offset(r, b0, cpd4)) = s4;
        }
    }
}

// ------------------------------------------------------------ launching ----
template <typename KernelT, typename... Args>
cudaError_t launch_cluster(KernelT kernel, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kFusedCluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kFusedCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int encode_grid(const DeviceInfo* info, int64_t M, int64_t K) {
    const int64_t tasks = pad_to(M, 128) * ((K + 1023) / 1024);
    int64_t g = (tasks + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)info->num_sms * 8;
    return (int)(g < cap ? g : cap);
}

int amax_grid(const DeviceInfo* info, int64_t n) {
    int64_t g = (n / 8 + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)info->num_sms * 4;
    if (cap > kMaxPartials) cap = kMaxPartials;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

size_t quantize_workspace_bytes(int64_t M, int64_t K) {
    if (M * K <= kFusedMaxElems) return 0;
    return (size_t)kMaxPartials * sizeof(uint32_t);
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
                           s_global);                                                                       \
    else                                                                                                    \
        quant_mx_kernel<F, false><<<grid, kThreads, 0, s>>>(x, M, K, partial, n_partial, codes, scales, s_global);
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
        n_partial = amax_grid(info, M * K);
        amax_partial_kernel<<<n_partial, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), M * K / 8, partial);
        count_launch(BSQ_KERNEL_AMAX);
        if (launch_status() != BSQ_OK) return BSQ_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    if (fused)
        e = launch_cluster(quant_nvfp4_kernel<true>, s, x, M, K, (const uint32_t*)nullptr, 0, codes, scales,
                           s_global);
    else
        quant_nvfp4_kernel<false><<<encode_grid(info, M, K), kThreads, 0, s>>>(x, M, K, partial, n_partial, codes,
                                                                              scales, s_global);
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
// The array (kMaxPartials words, 4 KiB) lives on every GPU that loads the
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
std::once_flag g_noalloc_once[kNoallocMaxDevices];
uint32_t* g_noalloc_ptr[kNoallocMaxDevices];

// Device address of the scratch array on the current device (nullptr on error).
uint32_t* noalloc_scratch() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return nullptr;
    std::call_once(g_noalloc_once[dev], [dev] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) == cudaSuccess) g_noalloc_ptr[dev] = static_cast<uint32_t*>(p);
        else (void)cudaGetLastError();
    });
    return g_noalloc_ptr[dev];
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
        quant_mx_kernel<kE3M2, false><<<grid, kThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global);
        break;
    case BSQ_E2M3:
        quant_mx_kernel<kE2M3, false><<<grid, kThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global);
        break;
    default:
        quant_mx_kernel<kE4M3, false><<<grid, kThreads, 0, stream>>>(x, M, K, scratch, n_partial, codes, scales, s_global);
        break;
    }
    count_launch(BSQ_KERNEL_QUANT_MX);
    return launch_status();
}
