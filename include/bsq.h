/*
 * bsq.h -- C ABI of libbsq: block-scaled packed-precision matrix products and
 * their quantizers on one GB300 (sm_103a).
 *
 * The operation (cubecl-tile tests/tile/packed.rs, nvfp4_shaped_matmul and
 * packed_matmul_rhs): c = (w (x) s_block (x) s_global) . x, written here as
 *     Y[m, n] = gA * gW * sum_k A[m, k] * W[n, k]          (Y = A W^T)
 * where each packed operand's element is decode(code) * block_scale.
 *
 * Formats (all little-endian):
 *   nvfp4  e2m1 codes, eight per uint32 word, element 0 in bits 0..3 ("low field
 *          first", cubecl-tile packed.rs module doc); rows of K/8 words.  One
 *          ue4m3 scale byte per 16 elements of a row; one fp32 tensor factor.
 *   MX     e3m2 / e2m3 codes packed four in three bytes,
 *          bits = c0 | c1<<6 | c2<<12 | c3<<18 (b12x _lib/fp6.py,
 *          pack_4_fp6_codes); rows of 3K/4 bytes.  e4m3 codes one byte each,
 *          rows of K bytes.  One UE8M0 byte (2^(e-127)) per 32 elements.
 *   block scales   a buffer of pad128(rows) * pad4(blocks) bytes, the scale of
 *          (row r, block b) at
 *          ((((r/128)*(pad4(blocks)/4) + b/4)*32 + r%32)*4 + (r%128)/32)*4 + b%4
 *          (b12x _lib/fp6.py, mxfp6_swizzled_scale_offset); padding bytes zero.
 *   tensor factor  s_global: the dequantization multiplier, a device float.
 *          The quantizers write 1/gs (gs = 448*fmt_max/amax; 0 if amax == 0).
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     never frees them, never keeps them after the call returns, and never
 *     modifies an input.
 *   - Work is enqueued on `stream` (0 = the legacy default stream); nothing
 *     synchronizes and nothing allocates on these call paths, so the calls can
 *     be captured in a CUDA graph.  The first call on a device loads its
 *     kernels; make one call before capturing.
 *   - Arguments are validated on the host before any launch; a failed check
 *     returns a status and launches nothing.
 *   - Launch failures return BSQ_ERR_CUDA.  Device-side timeouts of bounded
 *     waits are recorded in a device error word; read it with
 *     bsq_get_device_error.
 *   - Y / y are row-major [M, N], bf16 or fp32 as `out` says.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BSQ_ABI_VERSION 2

#if defined(__GNUC__)
#define BSQ_API __attribute__((visibility("default")))
#else
#define BSQ_API
#endif

typedef enum bsq_status {
    BSQ_OK = 0,
    BSQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum */
    BSQ_ERR_UNSUPPORTED = 2,   /* shape outside what a kernel supports */
    BSQ_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    BSQ_ERR_WORKSPACE = 4,     /* workspace missing or too small */
    BSQ_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    BSQ_ERR_TIMEOUT = 6,       /* a device-side bounded wait gave up */
    BSQ_ERR_DEVICE_CHECK = 7   /* a device-side check failed */
} bsq_status;

typedef enum bsq_mxfmt { BSQ_E3M2 = 0, BSQ_E2M3 = 1, BSQ_E4M3 = 2 } bsq_mxfmt;
typedef enum bsq_outtype { BSQ_OUT_F32 = 0, BSQ_OUT_BF16 = 1 } bsq_outtype;

/* Human-readable name of a status code (static storage; never NULL). */
BSQ_API const char* bsq_status_string(int status);

/* BSQ_ABI_VERSION of the loaded library. */
BSQ_API int bsq_abi_version(void);

/* Bytes of a block-scale buffer: pad128(rows) * pad4(n_blocks). */
BSQ_API size_t bsq_scale_bytes(int64_t rows, int64_t n_blocks);

/* Workspace the quantizers need for an [M, K] input; 0 when M*K is small
 * enough for the single-cluster path.  It holds the per-CTA partial maxima of
 * the tensor amax and, at its end, a small control block for the grid-wide
 * wait of the one-pass path.  Any initial contents are accepted: a call that
 * does not find the block's 64-bit marker initializes it, every call leaves it
 * ready for the next, and a call that reports a device error clears the marker
 * so the next call starts afresh.  (Contents that happen to hold the exact
 * marker with inconsistent counters -- odds 2^-64 for random bytes -- are not
 * detected.)  A call owns its workspace until its kernels finish: two calls
 * whose kernels may overlap on the GPU need two workspaces.  Always 256-byte
 * aligned sizes. */
BSQ_API size_t bsq_quantize_workspace_bytes(int64_t M, int64_t K);

/*
 * bsq_quantize_mxfp6 -- bf16 [M, K] -> MX codes + UE8M0 block scales + s_global.
 * b12x _lib/fp6.py: quantize_grouped_mxfp6_torch (one group) with the exact
 * scale steps of fp6_block_ue8m0_exact and ue8m0_output_scale_exact:
 *   amax = max|x|; gs = 448*fmt_max / amax (0 if amax == 0);
 *   per 32-block: ue = ceil(log2(fl(fl(amax_b*gs)/fmt_max))) + 127 (exact, by
 *   the f32 exponent field + (mantissa != 0)), clamped to [0, 255];
 *   inv = gs * 2^(127-ue) (0 if ue == 0);
 *   code = cvt.rn.satfinite(fl(x * inv)) (0 if inv == 0);
 *   *s_global = fl(1/gs) (0 if gs == 0).
 *   x        [M, K] bf16 bits, 16-byte aligned.  K % 32 == 0, M >= 1.
 *   fmt      BSQ_E3M2 / BSQ_E2M3 (fp6, codes [M, 3K/4] bytes) or BSQ_E4M3
 *            (codes [M, K] bytes).
 *   scales   bsq_scale_bytes(M, K/32) bytes, written whole (padding = 0).
 *   s_global one device float.
 *   workspace/workspace_bytes  >= bsq_quantize_workspace_bytes(M, K) bytes of
 *            device memory, 16-byte aligned (may be NULL when that is 0).
 * Results are bit-identical to the CPU oracle.
 */
BSQ_API bsq_status bsq_quantize_mxfp6(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt,
                              uint8_t* codes, uint8_t* scales, float* s_global,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bsq_quantize_grouped_mxfp6 -- grouped (MoE) MX quantize.
 * b12x _lib/fp6.py quantize_grouped_mxfp6_torch and as_grouped_mxfp6_scale_view:
 * group g's first row_counts[g] rows are quantized with the caller's global
 * scale gs[g] (not derived from an amax: the page takes it as an argument):
 * per 32-block ue = exact ceil of log2(fl(fl(amax_b*gs[g])/fmt_max)) + 127,
 * inv = gs[g] * 2^(127-ue), code = cvt.rn.satfinite(fl(x * inv)); rows past
 * row_counts[g] get zero codes and zero scales.
 *   x          [G, R, C] bf16 (16-byte aligned), C % 32 == 0.
 *   row_counts [G] int32 (device); values clamp to [0, R].
 *   gs         [G] float (device): each group's global scale (codes ~ x*gs/scale).
 *   codes      [G, R, row_bytes] bytes, group-major (row_bytes = 3C/4, or C for
 *              e4m3).  The page's [R, 3C/4, G] order is codes transposed.
 *   scales     G consecutive swizzled buffers of bsq_scale_bytes(R, C/32) bytes
 *              (the storage under the page's 6-D grouped scale view).
 *   s_global   [G] float (device): 1/gs[g] (0 if gs[g] == 0), the factor the
 *              products multiply by.
 * One launch, no workspace.  Results are bit-identical to the CPU oracle.
 */
BSQ_API bsq_status bsq_quantize_grouped_mxfp6(const uint16_t* x, int64_t G, int64_t R, int64_t C,
                                              const int32_t* row_counts, const float* gs, bsq_mxfmt fmt,
                                              uint8_t* codes, uint8_t* scales, float* s_global,
                                              cudaStream_t stream);

/*
 * bsq_gemm_grouped_mxfp6 -- grouped block-scaled GEMM over experts: for every
 * group g and row r < row_counts[g],
 *   Y[g, r, n] = gA[g] * gW[g] * sum_k A[g, r, k] * W[g, n, k]
 * with A and W in the grouped layouts of bsq_quantize_grouped_mxfp6 (A [G, R,
 * K], W [G, N, K], each group its own swizzled scale buffer and factor); rows
 * r >= row_counts[g] of Y are not written.  tcgen05 block-scaled MMA, one
 * persistent launch over every group's tiles (the row counts are read on the
 * device, so a routing step can produce them without a host round trip).
 *   fa, fw     MX formats of A and W; K % 128 == 0; G <= 256.
 *   gA, gW     [G] floats (device), e.g. the quantizers' s_global arrays.
 *   Y          [G, R, N] fp32 or bf16.
 * Tolerances as bsq_gemm_mxfp6 (fp32: 1e-5 * sum|a*w| per output).
 */
BSQ_API bsq_status bsq_gemm_grouped_mxfp6(const uint8_t* A, bsq_mxfmt fa, const uint8_t* sA, const float* gA,
                                          const uint8_t* W, bsq_mxfmt fw, const uint8_t* sW, const float* gW,
                                          const int32_t* row_counts, void* Y, bsq_outtype out, int64_t G,
                                          int64_t R, int64_t N, int64_t K, cudaStream_t stream);

/*
 * bsq_quantize_mxfp6_containers -- bsq_quantize_mxfp6 with fp6 byte-container
 * output: b12x _lib/fp6.py quantize_block_fp6_e3m2_bytes / _e2m3_bytes with
 * pack_32_byte_containers_to_4xu64 -- identical quantization, each 6-bit code
 * in its own byte (bits [5:0], bits [7:6] zero), K order, instead of four codes
 * in three bytes (the layout warp-level fp6 MMAs read without an expansion).
 *   fmt      BSQ_E3M2 or BSQ_E2M3 only.
 *   codes    [M, K] bytes; x, scales, s_global, workspace as bsq_quantize_mxfp6.
 * Results are bit-identical to the CPU oracle.
 */
BSQ_API bsq_status bsq_quantize_mxfp6_containers(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt,
                                                 uint8_t* codes, uint8_t* scales, float* s_global,
                                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bsq_quantize_mxfp6_act -- fused activation + MX quantize.
 * b12x _lib/fp6.py: relu2_quantize_grouped_mxfp6_torch and
 * silu_mul_quantize_grouped_mxfp6_torch (one group): the activation is
 * evaluated in f32 and rounded to bf16 (the input dtype), and that [M, K]
 * tensor is quantized exactly as by bsq_quantize_mxfp6 (amax recipe, exact
 * ceil UE8M0).  The activated tensor is not stored unless asked for.
 *   act = BSQ_ACT_RELU2:    a = max(x, 0)^2;             x [M, K] bf16.
 *   act = BSQ_ACT_SILU_MUL: a = fl(fl(g / fl(1 + exp(-g))) * u), g = x[m, k],
 *                           u = x[m, K + k];             x [M, 2K] bf16.
 *   act_out  NULL, or [M, K] bf16 (16-byte aligned): the activated tensor.
 *   codes, scales, s_global, workspace: as bsq_quantize_mxfp6 for this M, K
 *            (bsq_quantize_workspace_bytes(M, K)).
 * ReLU^2 results are bit-identical to the CPU oracle.  SiLU uses CUDA's expf,
 * whose last-place rounding can differ from a C library's, so an activated
 * value may sit one bf16 ulp from the oracle's; codes, scales and s_global are
 * bit-identical to the MX quantizer applied to act_out.
 * Errors: BSQ_ERR_INVALID_ARG (null pointer, act or fmt out of range, M < 1,
 * K % 32), BSQ_ERR_MISALIGNED, BSQ_ERR_WORKSPACE, BSQ_ERR_CUDA.
 */
typedef enum bsq_act { BSQ_ACT_RELU2 = 1, BSQ_ACT_SILU_MUL = 2 } bsq_act;
BSQ_API bsq_status bsq_quantize_mxfp6_act(const uint16_t* x, int64_t M, int64_t K, bsq_act act, bsq_mxfmt fmt,
                                          uint8_t* codes, uint8_t* scales, float* s_global, uint16_t* act_out,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bsq_quantize_mxfp6_noalloc -- bsq_quantize_mxfp6 for callers that cannot
 * allocate device memory on this path (no counterpart on the pages; this is a
 * library convenience).  Same arguments, results and validation minus the
 * workspace: the large-tensor path keeps its scratch (the amax pass's partial
 * maxima) in an 8 KiB device array owned by the library, present on every GPU
 * that loads it until the process exits.  The array holds 2048 partial maxima;
 * the amax pass never launches more CTAs than that, so every size the checks
 * above accept fits, and a call that would need more returns
 * BSQ_ERR_UNSUPPORTED.  The first call on a device looks up the array's device
 * address (make it before any stream capture); a lookup that fails returns
 * BSQ_ERR_CUDA and is tried again by the next call.  Calls share the array:
 * two calls whose kernels overlap on the GPU race on it.  Calls no allocator.
 */
BSQ_API bsq_status bsq_quantize_mxfp6_noalloc(const uint16_t* x, int64_t M, int64_t K, bsq_mxfmt fmt,
                                      uint8_t* codes, uint8_t* scales, float* s_global,
                                      cudaStream_t stream);

/*
 * bsq_quantize_nvfp4 -- bf16 [M, K] -> e2m1 words + ue4m3 block scales + s_global.
 * The pages give no nvfp4 recipe; this applies the MX recipe above with
 * e2m1's maximum 6 and a round-to-nearest e4m3 block scale:
 *   gs = 2688 / amax; s_b = e4m3_rn_satfinite(fl(fl(amax_b*gs)/6));
 *   inv = fl(gs / s_b) (0 if s_b == 0); code = e2m1_rn_satfinite(fl(x*inv)).
 *   codes  [M, K/8] uint32 words, low nibble first.  K % 16 == 0.
 *   scales bsq_scale_bytes(M, K/16) bytes.
 */
BSQ_API bsq_status bsq_quantize_nvfp4(const uint16_t* x, int64_t M, int64_t K,
                              uint32_t* codes, uint8_t* scales, float* s_global,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Batched quantizers -- up to BSQ_MAX_BATCH independent tensors (for example
 * a layer's activation and its weight) in one launch.  Each tensor is
 * quantized exactly as the single-tensor entry point above would (its own
 * amax, block scales and s_global; bit-identical results); the batch shares
 * one launch and one grid-wide wait instead of paying them per tensor.  The
 * b12x pages quantize "grouped" tensors (several experts' rows with
 * per-group global scales, _lib/fp6.py quantize_grouped_mxfp6_torch); this is
 * that idea for tensors of different shapes, not the pages' interleaved
 * grouped code layout.
 *   tensors[i]  as the single-tensor arguments: x [M, K] bf16 bits; codes as
 *               bsq_quantize_mxfp6 / bsq_quantize_nvfp4 lay them out; scales
 *               bsq_scale_bytes(M, K/32) (MX) or bsq_scale_bytes(M, K/16)
 *               (nvfp4); s_global one device float.  The tensors' outputs must
 *               not overlap one another or any input.
 *   n           1 .. BSQ_MAX_BATCH.
 *   workspace   >= bsq_quantize_batch_workspace_bytes() bytes of device
 *               memory, 16-byte aligned, owned by the call until its kernels
 *               finish.
 * A batch too large for one launch (more shared memory than the GPU has) runs
 * its tensors one after another on the stream, with the same results.
 */
#define BSQ_MAX_BATCH 8
typedef struct {
    const uint16_t* x;
    int64_t M, K;
    void* codes;
    uint8_t* scales;
    float* s_global;
} bsq_qtensor;

BSQ_API size_t bsq_quantize_batch_workspace_bytes(void);
BSQ_API bsq_status bsq_quantize_mxfp6_batch(const bsq_qtensor* tensors, int n, bsq_mxfmt fmt,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);
BSQ_API bsq_status bsq_quantize_nvfp4_batch(const bsq_qtensor* tensors, int n,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bsq_gemm_nvfp4 -- Y = gA*gW * A W^T with both operands nvfp4, on the 5th-gen
 * tensor cores (tcgen05.mma kind::mxf4nvf4, ue4m3 scale per 16).
 *   A [M, K/8] words + sA (bsq_scale_bytes(M, K/16)); W [N, K/8] + sW.
 *   gA, gW  device floats (NULL = 1).  K % 64 == 0; M, N >= 1.
 *   Y       [M, N] bf16 or fp32.
 * fp32 accumulation; |Y - Y_exact| <= 1e-5 * sum_k |a_k w_k| (fp32 out).
 */
BSQ_API bsq_status bsq_gemm_nvfp4(const uint32_t* A, const uint8_t* sA, const float* gA,
                          const uint32_t* W, const uint8_t* sW, const float* gW,
                          void* Y, bsq_outtype out, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream);

/*
 * bsq_gemm_mxfp6 -- Y = gA*gW * A W^T with MX operands (tcgen05.mma
 * kind::mxf8f6f4, UE8M0 per 32).  Each side is e3m2, e2m3 (4-in-3 packed) or
 * e4m3 (one byte per code), e.g. W6A6 e3m2 x e3m2 or W6A8 e4m3 x e2m3.
 *   A [M, K*bits/8] bytes + sA (bsq_scale_bytes(M, K/32)); W [N, ...] + sW.
 *   K % 128 == 0 (the packed-fp6 TMA unit); M, N >= 1.
 */
BSQ_API bsq_status bsq_gemm_mxfp6(const uint8_t* A, bsq_mxfmt fa, const uint8_t* sA, const float* gA,
                          const uint8_t* W, bsq_mxfmt fw, const uint8_t* sW, const float* gW,
                          void* Y, bsq_outtype out, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream);

/*
 * bsq_gemm_mxfp6_quant_a -- the MX product with the activation quantizer fused
 * into the GEMM (b12x fp6.py, the _containers quantize-then-MMA variants:
 * bf16 activations quantized in the kernel straight into the operand layout).
 * Two launches on `stream`: an amax pass over x (per-CTA maxima into the
 * workspace), then the GEMM, which reduces those maxima to A's global scale
 * gs = 448 * fmt_max / amax and, per 128 x 128 stage of A, computes the UE8M0
 * block scales and codes exactly as bsq_quantize_mxfp6 does and writes them
 * into shared memory for the tensor cores; A's codes never reach global memory.
 * Y equals, bit for bit, bsq_quantize_mxfp6(x, fa) followed by bsq_gemm_mxfp6
 * whenever that GEMM also runs 128-wide tiles (M*N small enough that 256-wide
 * tiles would not give every SM one).
 *   x          [M, K] bf16 activations, 16-byte aligned; fa e3m2, e2m3 or e4m3.
 *   W, fw, sW, gW  as for bsq_gemm_mxfp6.
 *   s_global_a device float receiving A's s_global = 1/gs (NULL: not stored).
 *   workspace  >= bsq_gemm_quant_a_workspace_bytes() bytes, 16-byte aligned,
 *              caller-owned scratch (contents on entry do not matter).
 *   K % 128 == 0; M, N >= 1.  Errors: BSQ_ERR_INVALID_ARG, BSQ_ERR_MISALIGNED,
 *   BSQ_ERR_WORKSPACE, BSQ_ERR_CUDA.
 */
BSQ_API size_t bsq_gemm_quant_a_workspace_bytes(void);
BSQ_API bsq_status bsq_gemm_mxfp6_quant_a(const uint16_t* x, bsq_mxfmt fa, const uint8_t* W, bsq_mxfmt fw,
                          const uint8_t* sW, const float* gW, void* Y, bsq_outtype out, float* s_global_a,
                          int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * bsq_gemv_nvfp4 -- decode product y = gW * x W^T with bf16 activations and an
 * nvfp4 weight (cubecl-tile packed.rs, packed_one_row_product: one activation
 * row, or a few, against packed weights streamed from HBM).
 *   x [M, K] bf16, 1 <= M <= 32; W [N, K/8] words + sW; gW device float
 *   (NULL = 1); K % 64 == 0; y [M, N] bf16 or fp32.
 */
BSQ_API bsq_status bsq_gemv_nvfp4(const uint16_t* x, const uint32_t* W, const uint8_t* sW, const float* gW,
                          void* y, bsq_outtype out, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream);

/*
 * bsq_gemv_mxfp6 -- the same decode product with an MX weight (e3m2 / e2m3
 * 4-in-3 packed, or e4m3).  K % 128 == 0; 1 <= M <= 32.  Every UE8M0 byte
 * 0..254 is applied exactly (byte 0 as 2^-127): each 32-code block's products
 * are summed in fp32 and scaled by the block's power of two before they are
 * added up.  |y - y_exact| <= 1e-5 * sum_k |x_k w_k| (fp32 out) while the
 * result and the fp32 partial sums stay in fp32's normal range.
 */
BSQ_API bsq_status bsq_gemv_mxfp6(const uint16_t* x, const uint8_t* W, bsq_mxfmt fw, const uint8_t* sW,
                          const float* gW, void* y, bsq_outtype out, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream);

/*
 * Dequantization (test and debugging aid; cubecl-tile packed.rs
 * packed_scaled_copy, b12x _lib/fp6.py dequant_mxfp6_torch):
 *   out[r, k] = decode(code) * scale(r, k/blk) * g   (fp32, [R, K])
 * g: device float (NULL = 1).  UE8M0 byte 0 decodes as 2^-127.
 * nvfp4 codes, out and g must be 4-byte aligned (BSQ_ERR_MISALIGNED).
 */
BSQ_API bsq_status bsq_dequant_nvfp4(const uint32_t* codes, const uint8_t* scales, const float* g,
                             float* out, int64_t R, int64_t K, cudaStream_t stream);
BSQ_API bsq_status bsq_dequant_mxfp6(const uint8_t* codes, bsq_mxfmt fmt, const uint8_t* scales,
                             const float* g, float* out, int64_t R, int64_t K, cudaStream_t stream);

/*
 * Reads and clears the device error word of the current device (a bounded
 * wait that timed out, or a device-side check).  Waits for the work enqueued
 * on `stream` (0 = the legacy default stream) to finish, then reads the word
 * and, if it is set, clears it, in stream order; work on other streams is not
 * waited for (the word is shared by every stream of the device).
 * *code_out = 0 when nothing was recorded; otherwise the first code written:
 *   - a bounded wait gave up: a site id 0x101..0x3FF (bit 31 clear), returned
 *     as BSQ_ERR_TIMEOUT;
 *   - a device bounds check failed (only in a library built with
 *     -DBSQ_DEVICE_CHECKS, which checks every global store and every global
 *     load addressed from a row and a column against its buffer's extent and
 *     skips the access when it leaves the buffer):
 *     0x80000000 | site << 24 | (offset & 0xFFFFFF), the
 *     offset of the access in its buffer's units, returned as
 *     BSQ_ERR_DEVICE_CHECK.  Sites: 0x01 quantizer x load, 0x02 codes store,
 *     0x03 scales store, 0x04 activation store; 0x11 GEMM Y store; 0x21 GEMV
 *     x load, 0x22 codes load, 0x23 scales load, 0x24 y store; 0x31
 *     dequantizer load, 0x32 dequantizer store.
 * Returns BSQ_ERR_CUDA if the stream reported an error.
 */
BSQ_API bsq_status bsq_get_device_error(cudaStream_t stream, uint32_t* code_out);

/* Launch counters (host side), one per kernel family, for dispatch tests and
 * for counting launches in a timed region.  ids: see BSQ_KERNEL_*. */
enum {
    BSQ_KERNEL_AMAX = 0,
    BSQ_KERNEL_QUANT_MX = 1,
    BSQ_KERNEL_QUANT_NVFP4 = 2,
    BSQ_KERNEL_QUANT_SMALL = 3,
    BSQ_KERNEL_GEMM_NVFP4 = 4,
    BSQ_KERNEL_GEMM_MX = 5,
    BSQ_KERNEL_GEMV_NVFP4 = 6,
    BSQ_KERNEL_GEMV_MX = 7,
    BSQ_KERNEL_DEQUANT = 8,
    BSQ_KERNEL_COUNT = 9
};
BSQ_API uint64_t bsq_launch_count(int kernel_id);
BSQ_API void bsq_reset_launch_counts(void);

#ifdef __cplusplus
}
#endif
#endif /* BSQ_H */
