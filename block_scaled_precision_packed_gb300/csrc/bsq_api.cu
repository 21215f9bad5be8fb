// bsq_api.cu -- the C ABI of libbsq: argument validation, per-device set-up,
// the device error word, launch counters, and dispatch to the kernels.
#include <atomic>
#include <cstring>
#include <mutex>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {

// The device error word (one per device that loads the library).  Bounded
// waits that give up write their site id here; bsq_get_device_error reads it.
static __device__ uint32_t g_device_error;

namespace {

std::atomic<uint64_t> g_launches[BSQ_KERNEL_COUNT];

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];
bsq_status g_init_status[kMaxDevices];

}  // namespace

const DeviceInfo* device_info(bsq_status* st) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        *st = BSQ_ERR_CUDA;
        return nullptr;
    }
    std::call_once(g_once[dev], [dev] {
        DeviceInfo& d = g_info[dev];
        g_init_status[dev] = BSQ_ERR_CUDA;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return;
        if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return;
        if (major != 10 || minor != 3) { g_init_status[dev] = BSQ_ERR_UNSUPPORTED; return; }
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return;
        d.err = static_cast<uint32_t*>(p);
        g_init_status[dev] = BSQ_OK;
    });
    if (g_init_status[dev] != BSQ_OK) {
        (void)cudaGetLastError();
        *st = g_init_status[dev];
        return nullptr;
    }
    *st = BSQ_OK;
    return &g_info[dev];
}

void count_launch(int kernel_id) { g_launches[kernel_id].fetch_add(1, std::memory_order_relaxed); }

EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

}  // namespace bsq

using namespace bsq;

namespace {

bool valid_mx(int f) { return f == BSQ_E3M2 || f == BSQ_E2M3 || f == BSQ_E4M3; }
bool valid_out(int o) { return o == BSQ_OUT_F32 || o == BSQ_OUT_BF16; }
int64_t mx_row_bytes(int f, int64_t K) { return f == BSQ_E4M3 ? K : 3 * K / 4; }
// 16U6 TMA wants 32-byte aligned fp6 operands.
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
constexpr int64_t kMaxDim = int64_t(1) << 31;

}  // namespace

extern "C" {

const char* bsq_status_string(int status) {
    switch (status) {
    case BSQ_OK: return "BSQ_OK";
    case BSQ_ERR_INVALID_ARG: return "BSQ_ERR_INVALID_ARG";
    case BSQ_ERR_UNSUPPORTED: return "BSQ_ERR_UNSUPPORTED";
    case BSQ_ERR_MISALIGNED: return "BSQ_ERR_MISALIGNED";
    case BSQ_ERR_WORKSPACE: return "BSQ_ERR_WORKSPACE";
    case BSQ_ERR_CUDA: return "BSQ_ERR_CUDA";
    case BSQ_ERR_TIMEOUT: return "BSQ_ERR_TIMEOUT";
    case BSQ_ERR_DEVICE_CHECK: return "BSQ_ERR_DEVICE_CHECK";
    default: return "BSQ_ERR_UNKNOWN";
    }
}

int bsq_abi_version(void) { return BSQ_ABI_VERSION; }

size_t bsq_scale_bytes(int64_t rows, int64_t n_blocks) {
    if (rows < 0 || n_blocks < 0) return 0;
    return (size_t)(pad_to(rows, 128) * pad_to(n_blocks, 4));
}

size_t bsq_quantize_workspace_bytes(int64_t M, int64_t K) {
    if (M < 0 || K < 0) return 0;
    return quantize_workspace_bytes(M, K);
}

bsq_status bsq_quantize_mxfp6(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt, uint8_t* codes,
                              uint8_t* scales, float* s_global, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    if (!x || !codes || !scales || !s_global || !valid_mx(fmt)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || K < 32 || K % 32 || M >= kMaxDim || K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return BSQ_ERR_MISALIGNED;
    return quantize_mx_launch(x, M, K, fmt, codes, scales, s_global, workspace, workspace_bytes, stream);
}

bsq_status bsq_quantize_grouped_mxfp6(const uint16_t* x, int64_t G, int64_t R, int64_t C, const int32_t* row_counts,
                                      const float* gs, bsq_mxfmt fmt, uint8_t* codes, uint8_t* scales,
                                      float* s_global, cudaStream_t stream) {
    if (!x || !row_counts || !gs || !codes || !scales || !s_global || !valid_mx(fmt)) return BSQ_ERR_INVALID_ARG;
    if (G < 1 || R < 1 || C < 32 || C % 32 || G * R >= kMaxDim || C >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (reinterpret_cast<uintptr_t>(row_counts) & 3u) ||
        (reinterpret_cast<uintptr_t>(gs) & 3u) || (reinterpret_cast<uintptr_t>(s_global) & 3u))
        return BSQ_ERR_MISALIGNED;
    return quantize_grouped_mx_launch(x, G, R, C, row_counts, gs, fmt, codes, scales, s_global, stream);
}

bsq_status bsq_gemm_grouped_mxfp6(const uint8_t* A, bsq_mxfmt fa, const uint8_t* sA, const float* gA, const uint8_t* W,
                                  bsq_mxfmt fw, const uint8_t* sW, const float* gW, const int32_t* row_counts, void* Y,
                                  bsq_outtype out, int64_t G, int64_t R, int64_t N, int64_t K, cudaStream_t stream) {
    if (!A || !sA || !gA || !W || !sW || !gW || !row_counts || !Y || !valid_mx(fa) || !valid_mx(fw) || !valid_out(out))
        return BSQ_ERR_INVALID_ARG;
    if (G < 1 || G > 256 || R < 1 || N < 1 || K < 128 || K % 128 || G * R >= kMaxDim || G * N >= kMaxDim ||
        K >= kMaxDim)
        return BSQ_ERR_INVALID_ARG;
    if (!aligned16(sA) || !aligned16(sW) || !aligned16(Y)) return BSQ_ERR_MISALIGNED;
    if (!(fa == BSQ_E4M3 ? aligned16(A) : aligned32(A)) || !(fw == BSQ_E4M3 ? aligned16(W) : aligned32(W)))
        return BSQ_ERR_MISALIGNED;
    // every group's scale buffer (a multiple of 512 bytes) starts 16-byte aligned
    return gemm_grouped_launch(A, fa, sA, gA, W, fw, sW, gW, row_counts, Y, out, G, R, N, K, false, stream);
}

bsq_status bsq_quantize_mxfp6_containers(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt, uint8_t* codes,
                                         uint8_t* scales, float* s_global, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
    if (!x || !codes || !scales || !s_global || (fmt != BSQ_E3M2 && fmt != BSQ_E2M3)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || K < 32 || K % 32 || M >= kMaxDim || K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return BSQ_ERR_MISALIGNED;
    return quantize_mx_containers_launch(x, M, K, fmt, codes, scales, s_global, workspace, workspace_bytes, stream);
}

bsq_status bsq_quantize_mxfp6_act(const uint16_t* x, int64_t M, int64_t K, bsq_act act, bsq_mxfmt fmt,
                                  uint8_t* codes, uint8_t* scales, float* s_global, uint16_t* act_out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!x || !codes || !scales || !s_global || !valid_mx(fmt)) return BSQ_ERR_INVALID_ARG;
    if (act != BSQ_ACT_RELU2 && act != BSQ_ACT_SILU_MUL) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || K < 32 || K % 32 || M >= kMaxDim || 2 * K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (act_out && !aligned16(act_out)))
        return BSQ_ERR_MISALIGNED;
    return quantize_mx_act_launch(x, M, K, (int)act, fmt, codes, scales, s_global, act_out, workspace,
                                  workspace_bytes, stream);
}

size_t bsq_quantize_batch_workspace_bytes(void) { return quantize_batch_workspace_bytes(); }

static bsq_status quantize_batch(const bsq_qtensor* t, int n, int fmt, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!t || n < 1 || n > BSQ_MAX_BATCH) return BSQ_ERR_INVALID_ARG;
    QTensor q[BSQ_MAX_BATCH];
    const int64_t kmod = fmt == kNvfp4 ? 16 : 32;
    for (int i = 0; i < n; ++i) {
        if (!t[i].x || !t[i].codes || !t[i].scales || !t[i].s_global) return BSQ_ERR_INVALID_ARG;
        if (t[i].M < 1 || t[i].K < kmod || t[i].K % kmod || t[i].M >= kMaxDim || t[i].K >= kMaxDim)
            return BSQ_ERR_INVALID_ARG;
        if (!aligned16(t[i].x) || !aligned16(t[i].codes) || !aligned16(t[i].scales)) return BSQ_ERR_MISALIGNED;
        q[i] = QTensor{t[i].x, t[i].M, t[i].K, t[i].codes, t[i].scales, t[i].s_global};
    }
    return quantize_batch_launch(q, n, fmt, ws, ws_bytes, s);
}

bsq_status bsq_quantize_mxfp6_batch(const bsq_qtensor* tensors, int n, bsq_mxfmt fmt, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
    if (!valid_mx(fmt)) return BSQ_ERR_INVALID_ARG;
    return quantize_batch(tensors, n, fmt, workspace, workspace_bytes, stream);
}

bsq_status bsq_quantize_nvfp4_batch(const bsq_qtensor* tensors, int n, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    return quantize_batch(tensors, n, kNvfp4, workspace, workspace_bytes, stream);
}

bsq_status bsq_quantize_nvfp4(const uint16_t* x, int64_t M, int64_t K, uint32_t* codes, uint8_t* scales,
                              float* s_global, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!x || !codes || !scales || !s_global) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || K < 16 || K % 16 || M >= kMaxDim || K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return BSQ_ERR_MISALIGNED;
    return quantize_nvfp4_launch(x, M, K, codes, scales, s_global, workspace, workspace_bytes, stream);
}

bsq_status bsq_gemm_nvfp4(const uint32_t* A, const uint8_t* sA, const float* gA, const uint32_t* W,
                          const uint8_t* sW, const float* gW, void* Y, bsq_outtype out, int64_t M, int64_t N,
                          int64_t K, cudaStream_t stream) {
    if (!A || !sA || !W || !sW || !Y || !valid_out(out)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 64 || K % 64 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return BSQ_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W) || !aligned16(sA) || !aligned16(sW) || !aligned16(Y))
        return BSQ_ERR_MISALIGNED;
    return gemm_launch(A, kNvfp4, sA, gA, W, kNvfp4, sW, gW, Y, out, M, N, K, true, stream);
}

bsq_status bsq_gemm_mxfp6(const uint8_t* A, bsq_mxfmt fa, const uint8_t* sA, const float* gA, const uint8_t* W,
                          bsq_mxfmt fw, const uint8_t* sW, const float* gW, void* Y, bsq_outtype out, int64_t M,
                          int64_t N, int64_t K, cudaStream_t stream) {
    if (!A || !sA || !W || !sW || !Y || !valid_out(out) || !valid_mx(fa) || !valid_mx(fw))
        return BSQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 128 || K % 128 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return BSQ_ERR_INVALID_ARG;
    if (!aligned16(sA) || !aligned16(sW) || !aligned16(Y)) return BSQ_ERR_MISALIGNED;
    if (!(fa == BSQ_E4M3 ? aligned16(A) : aligned32(A)) || !(fw == BSQ_E4M3 ? aligned16(W) : aligned32(W)))
        return BSQ_ERR_MISALIGNED;
    (void)mx_row_bytes;
    return gemm_launch(A, fa, sA, gA, W, fw, sW, gW, Y, out, M, N, K, false, stream);
}

size_t bsq_gemm_quant_a_workspace_bytes(void) { return kAmaxPartialsBytes; }

bsq_status bsq_gemm_mxfp6_quant_a(const uint16_t* x, bsq_mxfmt fa, const uint8_t* W, bsq_mxfmt fw,
                                  const uint8_t* sW, const float* gW, void* Y, bsq_outtype out, float* s_global_a,
                                  int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    if (!x || !W || !sW || !Y || !valid_out(out) || !valid_mx(fa) || !valid_mx(fw)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 128 || K % 128 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return BSQ_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kAmaxPartialsBytes) return BSQ_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(sW) || !aligned16(Y) || !aligned16(workspace)) return BSQ_ERR_MISALIGNED;
    if (s_global_a && (reinterpret_cast<uintptr_t>(s_global_a) & 3u)) return BSQ_ERR_MISALIGNED;
    if (!(fw == BSQ_E4M3 ? aligned16(W) : aligned32(W))) return BSQ_ERR_MISALIGNED;
    return gemm_quant_a_launch(x, fa, W, fw, sW, gW, Y, out, s_global_a, M, N, K, static_cast<uint32_t*>(workspace),
                               stream);
}

bsq_status bsq_gemv_nvfp4(const uint16_t* x, const uint32_t* W, const uint8_t* sW, const float* gW, void* y,
                          bsq_outtype out, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    if (!x || !W || !sW || !y || !valid_out(out)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || M > 32 || N < 1 || K < 64 || K % 64 || N >= kMaxDim || K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(sW)) return BSQ_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(y) & 3u) return BSQ_ERR_MISALIGNED;
    return gemv_launch(x, W, kNvfp4, sW, gW, y, out, M, N, K, true, stream);
}

bsq_status bsq_gemv_mxfp6(const uint16_t* x, const uint8_t* W, bsq_mxfmt fw, const uint8_t* sW, const float* gW,
                          void* y, bsq_outtype out, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    if (!x || !W || !sW || !y || !valid_out(out) || !valid_mx(fw)) return BSQ_ERR_INVALID_ARG;
    if (M < 1 || M > 32 || N < 1 || K < 128 || K % 128 || N >= kMaxDim || K >= kMaxDim) return BSQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(sW)) return BSQ_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(y) & 3u) return BSQ_ERR_MISALIGNED;
    return gemv_launch(x, W, fw, sW, gW, y, out, M, N, K, false, stream);
}

bsq_status bsq_dequant_nvfp4(const uint32_t* codes, const uint8_t* scales, const float* g, float* out, int64_t R,
                             int64_t K, cudaStream_t stream) {
    if (!codes || !scales || !out || R < 1 || K < 16 || K % 16) return BSQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(codes) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u) ||
        (g && (reinterpret_cast<uintptr_t>(g) & 3u)))
        return BSQ_ERR_MISALIGNED;
    return dequant_launch(codes, kNvfp4, scales, g, out, R, K, true, stream);
}

bsq_status bsq_dequant_mxfp6(const uint8_t* codes, bsq_mxfmt fmt, const uint8_t* scales, const float* g, float* out,
                             int64_t R, int64_t K, cudaStream_t stream) {
    if (!codes || !scales || !out || !valid_mx(fmt) || R < 1 || K < 32 || K % 32) return BSQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) || (g && (reinterpret_cast<uintptr_t>(g) & 3u)))
        return BSQ_ERR_MISALIGNED;
    return dequant_launch(codes, fmt, scales, g, out, R, K, false, stream);
}

bsq_status bsq_get_device_error(cudaStream_t stream, uint32_t* code_out) {
    if (!code_out) return BSQ_ERR_INVALID_ARG;
    bsq_status st;
    if (!device_info(&st)) return st;
    // the work enqueued on `stream` has finished, then the word is read (and
    // cleared if set) in stream order; other streams are not waited for
    uint32_t v = 0;
    static const uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof v, 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return BSQ_ERR_CUDA;
    }
    if (v != 0 && (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream) !=
                       cudaSuccess ||
                   cudaStreamSynchronize(stream) != cudaSuccess)) {
        (void)cudaGetLastError();
        return BSQ_ERR_CUDA;
    }
    *code_out = v;
    if (v == 0) return BSQ_OK;
    return (v & kCheckFlag) ? BSQ_ERR_DEVICE_CHECK : BSQ_ERR_TIMEOUT;
}

uint64_t bsq_launch_count(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= BSQ_KERNEL_COUNT) return 0;
    return g_launches[kernel_id].load(std::memory_order_relaxed);
}

void bsq_reset_launch_counts(void) {
    for (auto& c : g_launches) c.store(0, std::memory_order_relaxed);
}

}  // extern "C"
