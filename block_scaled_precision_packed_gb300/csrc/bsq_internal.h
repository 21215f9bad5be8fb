// bsq_internal.h -- host-side plumbing shared by the libbsq translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsq.h"

namespace bsq {

// Per-device state, set up by the first call on a device (with that device
// current): the device error word's address and the SM count.
struct DeviceInfo {
    uint32_t* err = nullptr;   // device address of the error word
    int num_sms = 0;
    int max_smem_optin = 0;
};

// Returns nullptr (and sets *st) if the current device cannot be set up.
const DeviceInfo* device_info(bsq_status* st);

void count_launch(int kernel_id);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The launch status of the kernel just enqueued.
inline bsq_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

// cuTensorMapEncodeTiled, resolved through the runtime (no -lcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// One tensor of a quantizer batch.
struct QTensor {
    const uint16_t* x;
    int64_t M, K;
    void* codes;
    uint8_t* scales;
    float* s_global;
};

// Entry points implemented per translation unit.
bsq_status quantize_mx_launch(const uint16_t* x, int64_t M, int64_t K, int fmt, uint8_t* codes,
                              uint8_t* scales, float* s_global, void* ws, size_t ws_bytes, cudaStream_t s);
// act: 1 = ReLU^2, 2 = SiLU(gate) * up (x rows of 2K); act_out optional
bsq_status quantize_mx_act_launch(const uint16_t* x, int64_t M, int64_t K, int act, int fmt, uint8_t* codes,
                                  uint8_t* scales, float* s_global, uint16_t* act_out, void* ws, size_t ws_bytes,
                                  cudaStream_t s);
bsq_status quantize_mx_containers_launch(const uint16_t* x, int64_t M, int64_t K, int fmt, uint8_t* codes,
                                         uint8_t* scales, float* s_global, void* ws, size_t ws_bytes,
                                         cudaStream_t s);
bsq_status quantize_grouped_mx_launch(const uint16_t* x, int64_t G, int64_t R, int64_t C, const int32_t* row_counts,
                                      const float* gs, int fmt, uint8_t* codes, uint8_t* scales, float* s_global,
                                      cudaStream_t s);
bsq_status quantize_nvfp4_launch(const uint16_t* x, int64_t M, int64_t K, uint32_t* codes, uint8_t* scales,
                                 float* s_global, void* ws, size_t ws_bytes, cudaStream_t s);
size_t quantize_workspace_bytes(int64_t M, int64_t K);
// The amax pass alone: per-CTA maxima of |x| (bf16 magnitude bits) over x [n]
// into partial (at most kAmaxPartialsBytes); returns how many, or -1.
constexpr size_t kAmaxPartialsBytes = 2048 * sizeof(uint32_t);
int amax_partials_launch(const uint16_t* x, int64_t n, uint32_t* partial, cudaStream_t s);
size_t quantize_batch_workspace_bytes();
// fmt: a bsq_mxfmt, or kNvfp4
bsq_status quantize_batch_launch(const QTensor* ts, int n, int fmt, void* ws, size_t ws_bytes, cudaStream_t s);

bsq_status gemm_launch(const void* A, int fa, const uint8_t* sA, const float* gA, const void* W, int fw,
                       const uint8_t* sW, const float* gW, void* Y, int out, int64_t M, int64_t N,
                       int64_t K, bool nvfp4, cudaStream_t s);

// GEMM whose bf16 activations are MX-quantized in the kernel (the amax pass,
// then the GEMM); partial: kAmaxPartialsBytes of device scratch.
bsq_status gemm_quant_a_launch(const uint16_t* x, int fa, const void* W, int fw, const uint8_t* sW, const float* gW,
                               void* Y, int out, float* s_global_a, int64_t M, int64_t N, int64_t K, uint32_t* partial,
                               cudaStream_t s);

bsq_status gemm_grouped_launch(const void* A, int fa, const uint8_t* sA, const float* gA, const void* W, int fw,
                               const uint8_t* sW, const float* gW, const int32_t* row_counts, void* Y, int out,
                               int64_t G, int64_t R, int64_t N, int64_t K, bool nvf4, cudaStream_t s);

bsq_status gemv_launch(const uint16_t* x, const void* W, int fw, const uint8_t* sW, const float* gW, void* y,
                       int out, int64_t M, int64_t N, int64_t K, bool nvfp4, cudaStream_t s);

bsq_status dequant_launch(const void* codes, int fmt, const uint8_t* scales, const float* g, float* out,
                          int64_t R, int64_t K, bool nvfp4, cudaStream_t s);

// Format id for nvfp4 in the internal launchers (the MX ids are bsq_mxfmt).
constexpr int kNvfp4 = 3;

}  // namespace bsq
