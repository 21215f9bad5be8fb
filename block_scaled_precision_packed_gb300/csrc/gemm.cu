// gemm.cu -- block-scaled GEMM on the 5th-generation tensor cores (sm_103a):
//     Y[m, n] = gA * gW * sum_k A[m, k] * W[n, k]
// with both operands packed minifloats and per-block scales
// (cubecl-tile tests/tile/packed.rs, nvfp4_shaped_matmul: the block level,
// then the tensor factor).
//
//   nvfp4  tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X: e2m1 x e2m1,
//          ue4m3 scale per 16, K = 64 per instruction (32 packed bytes).
//   MX     tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X: e3m2 / e2m3 /
//          e4m3 on either side, UE8M0 per 32, K = 32 per instruction.
//          The MMA reads a 6-bit operand from shared memory as 16 codes packed
//          in 12 bytes (the four-in-three rule) followed by 4 unused bytes;
//          the TMA unit produces exactly that from the packed rows
//          (CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B), counting the 96 packed
//          bytes of a 128-code row toward the stage's transaction.
//
// One persistent CTA per SM, warp-specialised (448 threads):
//   warp 0      TMA producer: A / W tiles (128-byte swizzle) and the scale
//               atoms (plain bulk copies) into an S-stage shared-memory ring.
//   warp 1      owns the TMEM allocation; one lane issues tcgen05.mma and
//               commits each stage back to the producer and each finished
//               tile to the epilogue.
//   warps 2-9   epilogue (two warps per TMEM lane quarter, one per column
//               half): tcgen05.ld the 128 x BN fp32 accumulator, scale by
//               gA*gW, convert; for bf16 output the whole tile is held in
//               registers so TMEM is released before the stores start.
//   warps 10-13 scale factors: one warp per TMEM lane quarter moves each
//               stage's scale atoms, as soon as they land (they are copied
//               ahead of the operand tiles, on a barrier of their own), from
//               shared memory into the stage's TMEM scale columns with
//               tcgen05.st (every quarter gets the same 32 x 16-byte rows,
//               the replicated layout the block-scaled MMA reads); once the
//               stage's operand tiles have landed too, one arrival per warp
//               releases it to the MMA thread, which so waits on a single
//               barrier per stage (each wait is a fixed cost in the one
//               thread that feeds the tensor pipe).  A tcgen05.cp of an atom
//               occupies the tensor pipe for about as long as a 128x256 MMA;
//               these stores do not.
// GROUPED (MoE experts, b12x fp6.py's grouped layout): A holds G groups of R
// rows ([G*R, K]), W holds G weights of N rows ([G*N, K]), each with its own
// swizzled scale buffer and global factor; group g contributes the first
// row_counts[g] rows of its A.  The persistent CTAs walk the tiles of every
// group (the per-group row-block counts, read from the device row counts, are
// prefix-summed in shared memory at the start) and store only valid rows.
// Every wait is bounded (2 s); a timeout records its site in the device error
// word, drains the copies in flight, frees TMEM and returns.
//
// The block-scale buffers are consumed in place: their layout (128 rows x 4
// blocks per 512-byte atom) is the one tcgen05.cp .32x128b.warpx4 moves into
// four TMEM columns, so a stage's scales are whole atoms.
#include <cstdio>
#include <mutex>

#include "bsq_device.cuh"
#include "bsq_internal.h"
#include "mx_encode.cuh"

namespace bsq {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 448;     // producer warp, MMA warp, 8 epilogue warps, 4 scale-factor warps
constexpr int kSfWarp0 = 10;      // first scale-factor warp
constexpr int kEpiThreads = 256;
constexpr int kAtom = 512;          // bytes of one 128-row x 4-block scale atom
constexpr uint32_t kTmemCols = 512;

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

template <bool NVF4, int BN, bool QX = false, bool PAIR = false>
struct Cfg {
    // QX: the stage also holds A's bf16 tile (128 x 128), quantized in the CTA.
    // PAIR: a CTA pair computes a 256 x BN tile; each CTA stages its own 128 A
    // rows and its own BN/2 W rows, and B's scale atoms for all BN rows.
    static constexpr int kStages = QX ? 3 : PAIR ? (NVF4 ? 5 : 6) : BN == 256 ? 4 : 6;
    static constexpr int kStageK = NVF4 ? 256 : 128;             // elements of K per stage
    static constexpr int kAtomsPerStage = NVF4 ? 4 : 1;          // scale atoms along K per 128 rows
    static constexpr int kRowTilesB = BN / 128;
    static constexpr int kRowsB = PAIR ? BN / 2 : BN;            // W rows in this CTA's B tile
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;          // output rows per tile
    static constexpr int kABytes = kBM * 128;
    static constexpr int kBBytes = kRowsB * 128;
    static constexpr int kSfaBytes = kAtomsPerStage * kAtom;
    static constexpr int kSfbBytes = kRowTilesB * kAtomsPerStage * kAtom;
    static constexpr int kXBytes = QX ? kBM * 128 * 2 : 0;         // two {64, 128} bf16 boxes
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes + kXBytes;
    // TMEM: accumulator columns [0, BN), then per stage SFA then SFB columns.
    static constexpr int kSfaCols = kAtomsPerStage * 4;
    static constexpr int kSfbCols = kRowTilesB * kAtomsPerStage * 4;
    static constexpr int kSfColsPerStage = kSfaCols + kSfbCols;
    static_assert(BN + kStages * kSfColsPerStage <= (int)kTmemCols, "TMEM budget");
    static_assert(!PAIR || (BN == 256 && !QX), "pair tiles: 256 x 256, operands from memory");
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 512 /*barriers*/;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    // barriers: full, empty, sf_full, sf_land, a_ready per stage; acc_full,
    // acc_empty, drain; the TMEM base and abort flag (one slot)
    static_assert((5 * kStages + 4) * 8 <= 512, "barrier slots");
};

constexpr int kMaxGroups = 256;

struct GemmArgs {
    const float* gA;           // grouped: [G]
    const float* gW;           // grouped: [G]
    void* Y;
    int64_t M, N, K;           // grouped: M = R, the rows per group of A
    const int32_t* row_counts; // grouped: [G] valid A rows per group
    int64_t G;                 // groups (1 when not grouped)
    int out_bf16;
    uint32_t idesc;        // instruction descriptor without the scale-id fields
    uint32_t tx_ab;        // TMA transaction bytes of one stage's A and W tiles (W only when A is quantized here)
    uint32_t* err;
    // A quantized in the kernel (QA >= 0): bf16 activations [M, K], the amax
    // pass's partial maxima, and where to put A's s_global (may be null)
    const uint16_t* qx;
    const uint32_t* qpartial;
    int qn_partial;
    float* qs_global;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Programmatic dependent launch: the next kernel on the stream may start its
// prologue; this kernel waits for the previous one's results before reading them.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The shared::cluster address of `local_addr` in the CTA of cluster rank `rank`
// (a CTA's window is contiguous, so offsets add to the mapped base).
__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" :: "r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(cluster_addr));
    return v;
}

// SPLIT == 1: persistent, one CTA per SM, tiles strided over the grid.
// SPLIT  > 1: split-K; a cluster of SPLIT CTAs owns one output tile, CTA rank r
//            runs K stages [r*S/SPLIT, (r+1)*S/SPLIT), and the fp32 partial
//            tiles are summed (rank order, deterministic) through distributed
//            shared memory -- no workspace, no atomics.
template <bool NVF4, int BN, int SPLIT, bool GROUPED = false, int QA = -1, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
            const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSW, const GemmArgs args) {
    using C = Cfg<NVF4, BN, (QA >= 0), PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA_st = smem;
    uint8_t* sB_st = sA_st + C::kStages * C::kABytes;
    uint8_t* sSfa = sB_st + C::kStages * C::kBBytes;
    uint8_t* sSfb = sSfa + C::kStages * C::kSfaBytes;
    uint8_t* sX = sSfb + C::kStages * C::kSfbBytes;                // QA: [kStages] bf16 A tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sX + C::kStages * C::kXBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::kStages;
    uint64_t* acc_full = bars + 2 * C::kStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_full + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(acc_full + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);
    uint64_t* sf_full = acc_full + 4;                 // [kStages]: scales in TMEM and operands landed
    uint64_t* sf_land = sf_full + C::kStages;         // [kStages]: the stage's scale atoms are in smem
    uint64_t* a_ready = sf_land + C::kStages;         // [kStages] (QA): the stage's A tile and SFA atom are made

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t num_mb = (M + C::kTileM - 1) / C::kTileM, num_nb = (N + BN - 1) / BN;
    const int64_t num_tiles = num_mb * num_nb;
    const int64_t nks_all = (K + C::kStageK - 1) / C::kStageK;
    const int64_t rt_total = pad_to(N, 128) / 128;   // 128-row scale tiles of W
    const int64_t rt_total_a = pad_to(M, 128) / 128; // ... and of A
    const uint32_t krank = SPLIT > 1 ? cluster_rank() : 0u;
    // PAIR: rank 0 of the pair issues the MMAs; rank 1 stages the other half
    const uint32_t prank = PAIR ? cluster_rank() : 0u;
    const int64_t ks_begin = nks_all * krank / SPLIT, ks_end = nks_all * (krank + 1) / SPLIT;
    const int64_t tile_first = PAIR ? (int64_t)(blockIdx.x / 2)
                                    : SPLIT > 1 ? (int64_t)(blockIdx.x / SPLIT) : (int64_t)blockIdx.x;
    const int64_t tile_step = PAIR ? (int64_t)(gridDim.x / 2) : SPLIT > 1 ? num_tiles : (int64_t)gridDim.x;
    static_assert(!GROUPED || SPLIT == 1, "grouped products are persistent, not split-K");
    static_assert(!PAIR || (SPLIT == 1 && !GROUPED && QA < 0), "pair tiles: persistent, ungrouped, quantized operands");
    static_assert(QA < 0 || (!NVF4 && BN == 128 && !GROUPED), "in-kernel A quantization: MX, 128-wide tiles");
    __shared__ uint32_t qa_red[QA >= 0 ? kThreads / 32 : 1];
    // grouped: mb_first[g] = row blocks of the groups before g (prefix sums)
    __shared__ int32_t mb_first[GROUPED ? kMaxGroups + 1 : 1];
    int64_t n_units = num_tiles, n_mt = num_mb;      // units: tiles; row-block count of the unit space

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(sf_full + s), PAIR ? 8 : 4);     // PAIR: both CTAs' scale-factor warps
            mbar_init(smem_u32(sf_land + s), 1);
            mbar_init(smem_u32(a_ready + s), kEpiThreads / 32);
        }
        mbar_init(smem_u32(acc_full), 1);
        mbar_init(smem_u32(acc_empty), PAIR ? 2 * (kEpiThreads / 32) : kEpiThreads);   // PAIR: one per warp
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmW);
        if constexpr (QA < 0) prefetch_tmap(&tmSA);
        prefetch_tmap(&tmSW);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_base_s), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_base_s), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // both CTAs' barriers exist before either signals the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    // the setup above overlaps the previous kernel; its outputs (A, W, their
    // scales and global factors) are read only after this
    pdl_wait();
    if constexpr (GROUPED) {
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int64_t g = 0; g < args.G; ++g) {
                mb_first[g] = acc;
                int64_t rc = args.row_counts[g];
                rc = rc < 0 ? 0 : (rc > M ? M : rc);
                acc += (int32_t)((rc + kBM - 1) / kBM);
            }
            mb_first[args.G] = acc;
        }
        __syncthreads();
        n_mt = mb_first[args.G];
        n_units = n_mt * num_nb;
    }
    // A quantized here: the tensor amax from the amax pass's partial maxima (every
    // thread), then gs = 448 * fmt_max / amax and s_global = fl(1/gs), exactly as
    // the quantizer computes them.
    float gs_a = 0.0f, sg_a = 0.0f;
    if constexpr (QA >= 0) {
        uint32_t m = 0;
        for (int i = threadIdx.x; i < args.qn_partial; i += kThreads) m = max(m, args.qpartial[i]);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) qa_red[warp] = m;
        __syncthreads();
        m = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) m = max(m, qa_red[w]);
        const float amax = bf16_bits_to_f32(m);
        gs_a = amax > 0.0f ? __fdiv_rn(gs_numerator(QA), amax) : 0.0f;
        sg_a = gs_a != 0.0f ? __fdiv_rn(1.0f, gs_a) : 0.0f;
        if (blockIdx.x == 0 && threadIdx.x == 0 && args.qs_global) *args.qs_global = sg_a;
    }
    // unit -> (group, row block within the group, column block)
    auto unit_at = [&](int64_t u, int64_t& g, int64_t& mb, int64_t& nb) {
        nb = u / n_mt;
        const int64_t mt = u - nb * n_mt;
        g = 0;
        if constexpr (GROUPED) {
            int64_t lo = 0, hi = args.G - 1;                 // the last g with mb_first[g] <= mt
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (mb_first[mid] <= mt) lo = mid; else hi = mid - 1;
            }
            g = lo;
            mb = mt - mb_first[g];
        } else {
            mb = mt;
        }
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer --
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_parity = 0, issued_any = 0;   // bit s: stage s's last parity / ever issued
            bool ok = true;
            for (int64_t tile = tile_first; tile < n_units && ok; tile += tile_step) {
                int64_t grp, mb, nb;
                unit_at(tile, grp, mb, nb);
                const int64_t a_row0 = grp * M + mb * C::kTileM + prank * kBM;
                const int64_t w_row0 = grp * N + nb * BN + prank * C::kRowsB;
                // this CTA's 128-row scale tile of A (past M: zeros)
                const int64_t a_rt = mb * (C::kTileM / kBM) + prank;
                for (int64_t ks = ks_begin; ks < ks_end; ++ks) {
                    if (!mbar_wait(smem_u32(empty + stage), phase ^ 1, args.err, abort_flag, kErrGemmProducer)) {
                        ok = false;
                        break;
                    }
                    const int64_t kg = ks * C::kAtomsPerStage;             // first scale atom along K
                    // The scale atoms go first, on their own barrier: the
                    // scale-factor warps move them into TMEM while the
                    // operand tiles are still in flight.  One tensor-map load
                    // per operand ({128 words, atoms, row tiles} of the
                    // atom-contiguous scale buffer); atoms past K and row tiles
                    // past the operand's rows read as zeros.
                    const uint32_t lb = smem_u32(sf_land + stage);
                    mbar_arrive_expect_tx(lb, (uint32_t)((QA >= 0 ? 0 : C::kSfaBytes) + C::kSfbBytes));
                    if constexpr (QA < 0)          // else the epilogue warps make A and its scale atom
                        tma_load_3d(smem_u32(sSfa + stage * C::kSfaBytes), &tmSA, lb, 0, (int32_t)kg,
                                    (int32_t)(grp * rt_total_a + a_rt));
                    tma_load_3d(smem_u32(sSfb + stage * C::kSfbBytes), &tmSW, lb, 0, (int32_t)kg,
                                (int32_t)(grp * rt_total + nb * C::kRowTilesB));
                    const uint32_t fb = smem_u32(full + stage);
                    mbar_arrive_expect_tx(fb, args.tx_ab);
                    const int32_t kx = (int32_t)(ks * (NVF4 ? 128 : C::kStageK));   // bytes (nvfp4) / elements
                    if constexpr (QA < 0) {
                        tma_load_2d(smem_u32(sA_st + stage * C::kABytes), &tmA, fb, kx, (int32_t)a_row0);
                    } else {                   // tmA maps the bf16 activations: two 64-value boxes
                        tma_load_2d(smem_u32(sX + stage * C::kXBytes), &tmA, fb, kx, (int32_t)a_row0);
                        tma_load_2d(smem_u32(sX + stage * C::kXBytes + C::kXBytes / 2), &tmA, fb, kx + 64,
                                    (int32_t)a_row0);
                    }
                    tma_load_2d(smem_u32(sB_st + stage * C::kBBytes), &tmW, fb, kx, (int32_t)w_row0);
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    issued_any |= 1u << stage;
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
            if (*abort_flag) {
                // drain: every copy issued must land before the CTA retires
                for (int s = 0; s < C::kStages; ++s) {
                    if (!((issued_any >> s) & 1u)) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(full + s), (issued_parity >> s) & 1u) && globaltimer() - t0 < kWaitLimitNs) {
                    }
                    while (!mbar_try_wait(smem_u32(sf_land + s), (issued_parity >> s) & 1u) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (NVF4 && PAIR && warp == 1) {
        if (prank == 0) {
            // ------------------------------------ MMA issue, nvfp4 CTA pairs --
            // The single thread that feeds the tensor pipe is the limit here (a
            // stage of four 256x256x64 MMAs is 512 cycles of tensor work; every
            // instruction the issuing thread spends between them shows up as
            // idle pipe), so this loop is kept lean: the whole warp runs it
            // (warp-uniform control flow) and lane 0 issues; the ring is walked
            // kStages slots per outer iteration, so each slot's barrier,
            // descriptor and TMEM column offsets are immediates added to
            // 32-bit bases.
            const bool leader = lane == 0;
            const uint64_t dA0 = smem_desc(smem_u32(sA_st), 16, 1024, 2);
            const uint64_t dB0 = smem_desc(smem_u32(sB_st), 16, 1024, 2);
            const uint32_t d_hi = (uint32_t)(dA0 >> 32);            // equal for A and B
            uint32_t a_lo = (uint32_t)dA0, b_lo = (uint32_t)dB0, sf_base = tmem + (uint32_t)BN;
            const uint32_t sf_full_b = smem_u32(sf_full), empty_b = smem_u32(empty);
            const int64_t nks = ks_end - ks_begin;
            const int64_t my_tiles = n_units > tile_first ? (n_units - tile_first + tile_step - 1) / tile_step : 0;
            const int64_t total = my_tiles * nks;
            // the stage cut by K (K % 256 != 0): its index within a tile and its MMA count
            const int64_t ks_cut = (K % C::kStageK) != 0 ? nks - 1 : -1;
            const int n_cut = (int)((K % C::kStageK) / 64);
            int64_t ks = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t g = 0; g < total && ok; g += C::kStages) {
                // opaque to the compiler, so the per-slot operands are formed here
                // by a few adds rather than all held in registers across the loop
                asm volatile("" : "+r"(a_lo), "+r"(b_lo), "+r"(sf_base));
#pragma unroll
                for (int j = 0; j < C::kStages; ++j) {
                    if (g + j < total && ok) {
                        if (ks == 0) {
                            ok = mbar_wait(smem_u32(acc_empty), acc_phase ^ 1, args.err, abort_flag, kErrGemmMma);
                            tc_fence_after();
                        }
                        // the slot's scales are in TMEM and both CTAs' tiles have landed
                        if (ok) ok = mbar_wait(sf_full_b + 8 * j, phase, args.err, abort_flag, kErrGemmMma);
                        if (ok) {
                            tc_fence_after();
                            if (leader) {
                                const uint32_t sfc = sf_base + (uint32_t)(j * C::kSfColsPerStage);
                                const uint32_t al = a_lo + (uint32_t)(j * (C::kABytes >> 4));
                                const uint32_t bl = b_lo + (uint32_t)(j * (C::kBBytes >> 4));
                                // K step kk: +32 bytes in both operands, scale atom kk
                                auto issue = [&](int kk, uint32_t acc) {
                                    tc_mma_mxf4nvf4_pair(tmem, ((uint64_t)d_hi << 32) | (al + 2u * kk),
                                                         ((uint64_t)d_hi << 32) | (bl + 2u * kk), args.idesc, sfc + 4 * kk,
                                                         sfc + C::kSfaCols + kk * C::kRowTilesB * 4, acc);
                                };
                                const uint32_t acc0 = ks != 0 ? 1u : 0u;
                                if (ks != ks_cut) {
                                    issue(0, acc0);
                                    issue(1, 1u);
                                    issue(2, 1u);
                                    issue(3, 1u);
                                } else {
                                    for (int kk = 0; kk < n_cut; ++kk) issue(kk, kk > 0 ? 1u : acc0);
                                }
                                // the slot is free again in both CTAs once these MMAs complete
                                tc_commit_pair_both(empty_b + 8 * j);
                            }
                            if (++ks == nks) {
                                if (leader) tc_commit_pair_both(smem_u32(acc_full));
                                ks = 0;
                                acc_phase ^= 1;
                            }
                        }
                    }
                }
                phase ^= 1;
            }
            if (leader) {
                // every MMA issued has completed before TMEM is released
                tc_commit_pair_local(smem_u32(drain));
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(drain), 0)) {
                    if (globaltimer() - t0 > kWaitLimitNs) { atomicCAS(args.err, 0u, (uint32_t)kErrGemmDrain); break; }
                }
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        if (lane == 0 && prank == 0) {
            // --------------------------------------------------- MMA issue --
            // Descriptors of stage 0's tiles; a stage or K step is an offset in
            // the 16-byte-unit address field (smem < 256 KB), so the single
            // issuing thread spends one add per tcgen05 instruction.
            const uint64_t dA0 = smem_desc(smem_u32(sA_st), 16, 1024, 2);
            const uint64_t dB0 = smem_desc(smem_u32(sB_st), 16, 1024, 2);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t tile = tile_first; tile < n_units && ok; tile += tile_step) {
                if (!mbar_wait(smem_u32(acc_empty), acc_phase ^ 1, args.err, abort_flag, kErrGemmMma))
                    break;
                tc_fence_after();
                for (int64_t ks = ks_begin; ks < ks_end; ++ks) {
                    // the stage's operands have landed and its scales are in TMEM
                    // one wait per stage: the scale-factor warps release the
                    // stage once its scales are in TMEM and its tiles landed
                    if (!mbar_wait(smem_u32(sf_full + stage), phase, args.err, abort_flag, kErrGemmMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_col = (uint32_t)(BN + stage * C::kSfColsPerStage);
                    const uint64_t a_st = dA0 + (uint64_t)(stage * (C::kABytes >> 4));
                    const uint64_t b_st = dB0 + (uint64_t)(stage * (C::kBBytes >> 4));
                    // MX: the stage's one atom per operand serves all 4 K steps;
                    // nvfp4: K step kk reads atom kk
                    auto issue = [&](int kk) {
                        const uint64_t ad = a_st + (uint64_t)(2 * kk);          // +32 bytes per K step
                        const uint64_t bd = b_st + (uint64_t)(2 * kk);
                        const uint32_t acc = (ks > ks_begin || kk > 0) ? 1u : 0u;
                        if constexpr (NVF4 && PAIR) {
                            tc_mma_mxf4nvf4_pair(tmem, ad, bd, args.idesc, tmem + sf_col + 4 * kk,
                                                 tmem + sf_col + C::kSfaCols + kk * C::kRowTilesB * 4, acc);
                        } else if constexpr (NVF4) {
                            tc_mma_mxf4nvf4(tmem, ad, bd, args.idesc, tmem + sf_col + 4 * kk,
                                            tmem + sf_col + C::kSfaCols + kk * C::kRowTilesB * 4, acc);
                        } else {
                            const uint32_t id = args.idesc | ((uint32_t)kk << 29) | ((uint32_t)kk << 4);
                            if constexpr (PAIR)
                                tc_mma_mxf8f6f4_pair(tmem, ad, bd, id, tmem + sf_col, tmem + sf_col + C::kSfaCols, acc);
                            else
                                tc_mma_mxf8f6f4(tmem, ad, bd, id, tmem + sf_col, tmem + sf_col + C::kSfaCols, acc);
                        }
                    };
                    // A whole stage issues its four MMAs back to back, with no branch
                    // between them; only an nvfp4 stage cut by K (K % 256 != 0) checks.
                    if (!NVF4 || (ks + 1) * C::kStageK <= K) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) issue(kk);
                    } else {
                        const int n_mma = (int)((K - ks * C::kStageK) / 64);
                        for (int kk = 0; kk < n_mma; ++kk) issue(kk);
                    }
                    // the stage is free again in both CTAs of a pair once these MMAs complete
                    if constexpr (PAIR) tc_commit_pair_both(smem_u32(empty + stage));
                    else tc_commit(smem_u32(empty + stage));
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if constexpr (PAIR) tc_commit_pair_both(smem_u32(acc_full));
                else tc_commit(smem_u32(acc_full));
                acc_phase ^= 1;
            }
            // every MMA issued has completed before TMEM is released
            if constexpr (PAIR) tc_commit_pair_local(smem_u32(drain));
            else tc_commit(smem_u32(drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(drain), 0)) {
                if (globaltimer() - t0 > kWaitLimitNs) { atomicCAS(args.err, 0u, (uint32_t)kErrGemmDrain); break; }
            }
        }
    } else if (warp >= kSfWarp0) {
        // -------------------------------------------------- scale factors --
        // Lane l of the warp for lane quarter q writes TMEM lane 32q + l: row l
        // (16 bytes = 4 columns) of every atom of the stage.
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t tile = tile_first; tile < n_units && ok; tile += tile_step) {
            for (int64_t ks = ks_begin; ks < ks_end; ++ks) {
                if (!mbar_wait(smem_u32(sf_land + stage), phase, args.err, abort_flag, kErrGemmMma) ||
                    (QA >= 0 && !mbar_wait(smem_u32(a_ready + stage), phase, args.err, abort_flag, kErrGemmMma))) {
                    ok = false;
                    break;
                }
                const uint32_t sf_col = (uint32_t)(BN + stage * C::kSfColsPerStage);
                const uint8_t* sa = sSfa + stage * C::kSfaBytes + 16 * lane;
                const uint8_t* sb = sSfb + stage * C::kSfbBytes + 16 * lane;
                uint32_t ra[4 * C::kAtomsPerStage];
                uint32_t rb[4 * C::kAtomsPerStage * C::kRowTilesB];
#pragma unroll
                for (int a = 0; a < C::kAtomsPerStage; ++a) {
                    const uint4 v = *reinterpret_cast<const uint4*>(sa + a * kAtom);
                    ra[4 * a] = v.x; ra[4 * a + 1] = v.y; ra[4 * a + 2] = v.z; ra[4 * a + 3] = v.w;
#pragma unroll
                    for (int rt = 0; rt < C::kRowTilesB; ++rt) {
                        const uint4 w = *reinterpret_cast<const uint4*>(sb + (rt * C::kAtomsPerStage + a) * kAtom);
                        const int j = 4 * (a * C::kRowTilesB + rt);
                        rb[j] = w.x; rb[j + 1] = w.y; rb[j + 2] = w.z; rb[j + 3] = w.w;
                    }
                }
                tc_st_cols(lane_base + sf_col, ra);
                tc_st_cols(lane_base + sf_col + C::kSfaCols, rb);
                tc_wait_st();
                tc_fence_before();
                // relay the operand tiles' landing, so that the MMA thread
                // waits on one barrier per stage
                if (!mbar_wait(smem_u32(full + stage), phase, args.err, abort_flag, kErrGemmMma)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (lane == 0) {
                    // a pair's MMA thread (rank 0) waits for both CTAs' warps
                    if (PAIR && prank != 0) mbar_arrive_cluster(map_rank(smem_u32(sf_full + stage), 0));
                    else mbar_arrive(smem_u32(sf_full + stage));
                }
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue --
        if constexpr (QA >= 0) {
            // First the A operand: the producer loads each stage's 128 x 128 bf16
            // tile of A beside the W tile (two {64, 128} boxes, 128-byte swizzle,
            // zeros past M and K); these warps quantize it (the quantizer's block
            // scale and encode) straight into the layout the tensor map would have
            // produced for the codes -- row r's 16-code chunk c at (c ^ (r & 7)) *
            // 16, an fp6 chunk as its 12 packed bytes and 4 zero bytes, an e4m3
            // chunk as 16 bytes -- and its UE8M0 bytes into the stage's scale
            // atom.  Thread (r, h) takes values [64h, 64h + 64) of row r of the
            // stage: blocks 2h and 2h + 1.  Zero values give zero codes and zero
            // scales, as the quantizer writes them.  One tile per CTA (the host
            // launches no persistence).
            const int et = (int)threadIdx.x - 64;
            const int qr = et >> 1, qh = et & 1;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t tile = tile_first; tile < n_units && ok; tile += tile_step) {
                int64_t grp, mb, nb;
                unit_at(tile, grp, mb, nb);
                (void)mb;
                for (int64_t ks = ks_begin; ks < ks_end; ++ks) {
                    // the stage's W tile and bf16 A tile have landed (the producer refilled
                    // the stage only after the MMAs that read it before completed)
                    if (!mbar_wait(smem_u32(full + stage), phase, args.err, abort_flag, kErrGemmEpilogue)) {
                        ok = false;
                        break;
                    }
                    // this thread's 64 values: box qh, row qr (128-byte swizzle: 16-byte
                    // piece c at (c ^ (qr & 7)) * 16); rows >= M and values past K are zero
                    uint4 xv[2][4];
                    const uint32_t xb = smem_u32(sX + stage * C::kXBytes + qh * (C::kXBytes / 2)) + (uint32_t)qr * 128u;
#pragma unroll
                    for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            xv[bl][j] = lds_v4(xb + ((((uint32_t)(4 * bl + j)) ^ (uint32_t)(qr & 7)) << 4));
                    const uint32_t a_row = smem_u32(sA_st + stage * C::kABytes) + (uint32_t)qr * 128u;
                    uint32_t ue2 = 0;
#pragma unroll
                    for (int bl = 0; bl < 2; ++bl) {
                        uint32_t ue, w[8];
                        float inv;
                        mx_block_scale<QA>(absmax32_bits(xv[bl]), gs_a, ue, inv);
                        mx_encode_words<QA>(xv[bl], inv, w);
                        ue2 |= ue << (8 * bl);
                        const uint32_t c = (uint32_t)(4 * qh + 2 * bl);       // first 16-code chunk of the block
                        const uint32_t p0 = a_row + ((c ^ (uint32_t)(qr & 7)) << 4);
                        const uint32_t p1 = a_row + (((c + 1) ^ (uint32_t)(qr & 7)) << 4);
                        if constexpr (QA == kE4M3) {
                            sts_v4(p0, w[0], w[1], w[2], w[3]);
                            sts_v4(p1, w[4], w[5], w[6], w[7]);
                        } else {
                            sts_v4(p0, w[0], w[1], w[2], 0u);
                            sts_v4(p1, w[3], w[4], w[5], 0u);
                        }
                    }
                    sts_u16(smem_u32(sSfa + stage * C::kSfaBytes) + (uint32_t)((qr & 31) * 16 + ((qr >> 5) & 3) * 4 + 2 * qh),
                            (uint16_t)ue2);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the MMA reads A via the async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(a_ready + stage));
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
        }
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;             // which half of the tile's columns
        constexpr int kHalf = BN / 2;
        const float f = __fmul_rn(QA >= 0 ? sg_a : (args.gA ? __ldg(args.gA) : 1.0f), args.gW ? __ldg(args.gW) : 1.0f);
        uint32_t acc_phase = 0;
        // hand the accumulator back to the MMA thread: every thread (count 256),
        // or for a pair one arrival per warp of either CTA on rank 0's barrier
        auto release_acc = [&]() {
            if constexpr (PAIR) {
                __syncwarp();
                if (lane == 0) {
                    if (prank != 0) mbar_arrive_cluster(map_rank(smem_u32(acc_empty), 0));
                    else mbar_arrive(smem_u32(acc_empty));
                }
            } else {
                mbar_arrive(smem_u32(acc_empty));
            }
        };
        const bool vec = args.out_bf16 ? (N % 8 == 0) : (N % 4 == 0);
        // Each thread writes one output row: 32-byte stores (whole sectors)
        // halve the memory requests of 16-byte ones.
        const bool vec32 = (N % (args.out_bf16 ? 16 : 8) == 0) && ((reinterpret_cast<uintptr_t>(args.Y) & 31) == 0);
        if constexpr (SPLIT > 1) {
            // Partial tile -> this CTA's shared memory (the operand ring is idle:
            // the single tile's last MMA has completed), then sum across the
            // cluster, each CTA finishing kBM/SPLIT rows.
            float* part = reinterpret_cast<float*>(smem);               // [kBM][BN + 4] fp32
            constexpr int kPitch = BN + 4;
            const bool have = mbar_wait(smem_u32(acc_full), 0, args.err, abort_flag, kErrGemmEpilogue);
            if (have) {
                tc_fence_after();
                const int lrow = 32 * q + lane;
#pragma unroll 1
                for (int c = 0; c < kHalf / 32; ++c) {
                    uint32_t r[32];
                    tc_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kHalf * half + 32 * c), r);
                    tc_wait_ld();
                    float4* dst = reinterpret_cast<float4*>(part + lrow * kPitch + kHalf * half + 32 * c);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                             __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                }
                tc_fence_before();
            }
        }
        for (int64_t tile = tile_first; tile < n_units && SPLIT == 1; tile += tile_step) {
            int64_t grp, mb, nb;
            unit_at(tile, grp, mb, nb);
            if (!mbar_wait(smem_u32(acc_full), acc_phase, args.err, abort_flag, kErrGemmEpilogue))
                break;
            tc_fence_after();
            const int64_t row_base = mb * C::kTileM + prank * kBM;     // this CTA's first row of the tile
            const int64_t lrow = row_base + 32 * q + lane;              // row within the group
            int64_t rows_valid = M;
            float fg = f;
            if constexpr (GROUPED) {
                const int64_t rc = args.row_counts[grp];
                rows_valid = rc < 0 ? 0 : (rc > M ? M : rc);
                fg = __fmul_rn(__ldg(args.gA + grp), __ldg(args.gW + grp));
            }
            const bool row_ok = lrow < rows_valid;
            const int64_t row = grp * M + lrow;                         // output row
            if (args.out_bf16) {
                // Drain the whole accumulator row into registers as bf16 pairs,
                // hand TMEM back to the MMA warp, then store: the next tile's
                // MMAs overlap these stores.
                // (16 columns per TMEM load keeps the 256-wide tile's drain
                // within the register budget)
                uint32_t packed[kHalf / 2];
#pragma unroll
                for (int c = 0; c < kHalf / 16; ++c) {
                    uint32_t r0[16];
                    tc_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kHalf * half + 16 * c), r0);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        packed[8 * c + e] = f32x2_to_bf16x2_bits(__fmul_rn(__uint_as_float(r0[2 * e]), fg),
                                                                __fmul_rn(__uint_as_float(r0[2 * e + 1]), fg));
                }
                tc_fence_before();
                release_acc();
                acc_phase ^= 1;
                if (vec32) {
                    // Whole 128-byte lines: within each group of four lanes
                    // (four consecutive rows) the 32-byte chunks are
                    // transposed with two butterfly exchanges, so that lane i
                    // of the group holds chunk i of 64 columns of each of the
                    // four rows; one store then writes 8 rows x 128 bytes.
                    const int gi = lane & 3;
                    const int64_t lrow0 = row_base + 32 * q + (lane & ~3);  // the group's first row (within the group)
                    uint16_t* ybase = static_cast<uint16_t*>(args.Y) + (grp * M + lrow0) * N + nb * BN + kHalf * half;
#pragma unroll
                    for (int h = 0; h < kHalf / 64; ++h) {
                        uint32_t* x = packed + 32 * h;                        // chunk j: x[8j .. 8j+7]
#pragma unroll
                        for (int j = 0; j < 4; j += 2) {                      // exchange with lane ^ 1
#pragma unroll
                            for (int w = 0; w < 8; ++w) {
                                const uint32_t send = (gi & 1) ? x[8 * j + w] : x[8 * (j + 1) + w];
                                const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
                                if (gi & 1) x[8 * j + w] = recv; else x[8 * (j + 1) + w] = recv;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {                         // exchange with lane ^ 2
#pragma unroll
                            for (int w = 0; w < 8; ++w) {
                                const uint32_t send = (gi & 2) ? x[8 * j + w] : x[8 * (j + 2) + w];
                                const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 2);
                                if (gi & 2) x[8 * j + w] = recv; else x[8 * (j + 2) + w] = recv;
                            }
                        }
                        const int64_t col = nb * BN + kHalf * half + 64 * h + 16 * gi;
#pragma unroll
                        for (int j = 0; j < 4; ++j)                           // row lrow0 + j, columns col .. col+15
                            if (lrow0 + j < rows_valid && col + 16 <= N &&
                                BSQ_IN_BUFFER(args.err, kChkGemmY, (grp * M + lrow0 + j) * N + col, 16, args.G * M * N))
                                st_global_v8(ybase + j * N + 64 * h + 16 * gi, x[8 * j], x[8 * j + 1], x[8 * j + 2],
                                             x[8 * j + 3], x[8 * j + 4], x[8 * j + 5], x[8 * j + 6], x[8 * j + 7]);
                    }
                } else if (row_ok) {
                    uint16_t* yr = static_cast<uint16_t*>(args.Y) + row * N + nb * BN + kHalf * half;
#pragma unroll
                    for (int c = 0; c < kHalf / 32; ++c) {
                        const int64_t col0 = nb * BN + kHalf * half + 32 * c;
                        if (col0 < N && !BSQ_IN_BUFFER(args.err, kChkGemmY, row * N + col0, N - col0 < 32 ? N - col0 : 32,
                                                       args.G * M * N))
                            continue;
                        if (vec && col0 + 32 <= N) {
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                *reinterpret_cast<uint4*>(yr + 32 * c + 8 * v) =
                                    make_uint4(packed[16 * c + 4 * v], packed[16 * c + 4 * v + 1],
                                               packed[16 * c + 4 * v + 2], packed[16 * c + 4 * v + 3]);
                        } else {
                            // ragged columns: constant register indices only
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const uint32_t two = packed[16 * c + e];
                                if (col0 + 2 * e < N) yr[32 * c + 2 * e] = (uint16_t)(two & 0xFFFFu);
                                if (col0 + 2 * e + 1 < N) yr[32 * c + 2 * e + 1] = (uint16_t)(two >> 16);
                            }
                        }
                    }
                }
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t r[32];
                tc_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kHalf * half + 32 * c), r);
                tc_wait_ld();
                const int64_t col0 = nb * BN + kHalf * half + 32 * c;
                if (row_ok && col0 < N &&
                    BSQ_IN_BUFFER(args.err, kChkGemmY, row * N + col0, N - col0 < 32 ? N - col0 : 32, args.G * M * N)) {
                    // fp32 output (the bf16 case returned above)
                    float* yr = static_cast<float*>(args.Y) + row * N + col0;
                    float o[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __fmul_rn(__uint_as_float(r[e]), fg);
                    if (vec32 && col0 + 32 <= N) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            st_global_v8(yr + 8 * v, __float_as_uint(o[8 * v]), __float_as_uint(o[8 * v + 1]),
                                         __float_as_uint(o[8 * v + 2]), __float_as_uint(o[8 * v + 3]),
                                         __float_as_uint(o[8 * v + 4]), __float_as_uint(o[8 * v + 5]),
                                         __float_as_uint(o[8 * v + 6]), __float_as_uint(o[8 * v + 7]));
                    } else if (vec && col0 + 32 <= N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *reinterpret_cast<float4*>(yr + 4 * v) = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (col0 + e < N) yr[e] = o[e];
                    }
                }
            }
            tc_fence_before();
            release_acc();
            acc_phase ^= 1;
        }
    }

    if constexpr (SPLIT > 1) {
        __syncwarp();                                     // reconverge the role warps first
        cluster_sync();                                   // every rank's partial tile is in its smem
        const int64_t tile = tile_first;
        const int64_t mb = tile % num_mb, nb = tile / num_mb;
        constexpr int kPitch = BN + 4;
        constexpr int kRows = kBM / SPLIT;
        const float f = __fmul_rn(QA >= 0 ? sg_a : (args.gA ? __ldg(args.gA) : 1.0f), args.gW ? __ldg(args.gW) : 1.0f);
        // Each thread owns up to kPer float4 groups of this rank's rows; every
        // rank's copy of all of them is requested before the first sum, so the
        // distributed-shared-memory latency is paid once.
        constexpr int kItems = kRows * (BN / 4);
        constexpr int kPer = (kItems + kThreads - 1) / kThreads;
        uint32_t base[SPLIT];
#pragma unroll
        for (int rk = 0; rk < SPLIT; ++rk) base[rk] = map_rank(smem_u32(smem), (uint32_t)rk);
        float4 v[kPer][SPLIT];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int it = (int)threadIdx.x + j * kThreads;
            if (it >= kItems) break;
            const int lr = (int)krank * kRows + it / (BN / 4), cg = it % (BN / 4);
            const uint32_t off = (uint32_t)((lr * kPitch + 4 * cg) * 4);
#pragma unroll
            for (int rk = 0; rk < SPLIT; ++rk) v[j][rk] = ld_cluster_f4(base[rk] + off);
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int it = (int)threadIdx.x + j * kThreads;
            if (it >= kItems) break;
            const int lr = (int)krank * kRows + it / (BN / 4), cg = it % (BN / 4);
            float4 acc = v[j][0];                          // rank order: deterministic
#pragma unroll
            for (int rk = 1; rk < SPLIT; ++rk) {
                acc.x += v[j][rk].x; acc.y += v[j][rk].y; acc.z += v[j][rk].z; acc.w += v[j][rk].w;
            }
            const int64_t row = mb * kBM + lr, col = nb * BN + 4 * cg;
            if (row >= M || col >= N) continue;
            if (!BSQ_IN_BUFFER(args.err, kChkGemmY, row * N + col, N - col < 4 ? N - col : 4, args.G * M * N)) continue;
            const float o[4] = {__fmul_rn(acc.x, f), __fmul_rn(acc.y, f), __fmul_rn(acc.z, f), __fmul_rn(acc.w, f)};
            if (args.out_bf16) {
                uint16_t* y = static_cast<uint16_t*>(args.Y) + row * N + col;
                if (col + 4 <= N && (N % 4) == 0) {
                    *reinterpret_cast<uint2*>(y) =
                        make_uint2(f32x2_to_bf16x2_bits(o[0], o[1]), f32x2_to_bf16x2_bits(o[2], o[3]));
                } else {
                    for (int e = 0; e < 4 && col + e < N; ++e) y[e] = f32_to_bf16_bits(o[e]);
                }
            } else {
                float* y = static_cast<float*>(args.Y) + row * N + col;
                if (col + 4 <= N && (N % 4) == 0) *reinterpret_cast<float4*>(y) = make_float4(o[0], o[1], o[2], o[3]);
                else for (int e = 0; e < 4 && col + e < N; ++e) y[e] = o[e];
            }
        }
        cluster_sync();                                   // no rank leaves while others read its smem
    }
    pdl_launch_dependents();
    tc_fence_before();
    if constexpr (PAIR) {
        // neither CTA releases TMEM or its shared memory before the pair's
        // last MMA (which reads both) has completed: rank 0's MMA thread waited
        // for it above
        __syncwarp();
        cluster_sync();
    } else {
        __syncthreads();
    }
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host ----
// Instruction descriptor (kind::mxf8f6f4 / kind::mxf4nvf4, dense, K-major):
// bits 7-9 A format, 10-12 B format, 17-22 N>>3, 23 scale type (1 = UE8M0),
// 24-28 M>>4; the scale-factor ids (bits 4-5 B, 29-30 A) are set per MMA.
uint32_t make_idesc(bool nvf4, int fa, int fw, int bn, int bm = kBM) {
    auto code = [](int f) -> uint32_t { return f == kE4M3 ? 0u : f == kE2M3 ? 3u : 4u; };
    uint32_t d = 0;
    if (nvf4) {
        d |= 1u << 7;            // e2m1
        d |= 1u << 10;
    } else {
        d |= code(fa) << 7;
        d |= code(fw) << 10;
        d |= 1u << 23;           // UE8M0 scales
    }
    d |= (uint32_t)(bn >> 3) << 17;
    d |= (uint32_t)(bm >> 4) << 24;        // a pair's MMA spans both CTAs' rows: M = 256
    return d;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over a block-scale buffer as 32-bit words: {128 words of a
// 512-byte atom, atoms along K (cpd4), 128-row tiles}; one load of box
// {128, box_atoms, box_tiles} brings a stage's atoms of one or two row tiles
// into shared memory in [tile][atom][512 B] order, zeros past either end.
bool scale_map(CUtensorMap* map, const uint8_t* base, int64_t row_tiles, int64_t cpd4, uint32_t box_atoms,
               uint32_t box_tiles) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)cpd4, (cuuint64_t)row_tiles};
    const cuuint64_t strides[2] = {(cuuint64_t)kAtom, (cuuint64_t)(cpd4 * kAtom)};
    const cuuint32_t box[3] = {128, box_atoms, box_tiles};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four tensor maps of a launch: operands A and W, their scale buffers.
struct Maps {
    CUtensorMap a, w, sa, sw;
};

// Tensor map of one operand: nvfp4 as raw bytes (K/2 per row), fp6 through
// the 16U6_ALIGN16B unpacking type (K codes per row), e4m3 as bytes.
bool operand_map(CUtensorMap* map, const void* p, int fmt, bool nvf4, int64_t rows, int64_t K, uint32_t box_rows) {
    if (nvf4) return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, p, (uint64_t)(K / 2), (uint64_t)rows,
                                (uint64_t)(K / 2), 128, box_rows);
    if (fmt == kE4M3) return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, p, (uint64_t)K, (uint64_t)rows,
                                        (uint64_t)K, 128, box_rows);
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B, p, (uint64_t)K, (uint64_t)rows,
                      (uint64_t)(3 * K / 4), 128, box_rows);
}

template <bool NVF4, int BN, int SPLIT, bool GROUPED = false, int QA = -1, bool PAIR = false>
bsq_status launch_gemm(const DeviceInfo* info, const Maps& mp, const GemmArgs& a, cudaStream_t s) {
    using C = Cfg<NVF4, BN, (QA >= 0), PAIR>;
    auto kernel = gemm_kernel<NVF4, BN, SPLIT, GROUPED, QA, PAIR>;
    static std::once_flag flags[64];
    static bool ok_dev[64];
    static int pairs_dev[64];          // PAIR: how many CTA pairs fit on the device at once
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSQ_ERR_CUDA;
    std::call_once(flags[dev], [&] {
        ok_dev[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) ==
                      cudaSuccess;
        if (PAIR && ok_dev[dev]) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3((unsigned)(2 * (info->num_sms / 2)), 1, 1);
            q.blockDim = dim3(kThreads, 1, 1);
            q.dynamicSmemBytes = C::kSmemBytes;
            cudaLaunchAttribute ca;
            ca.id = cudaLaunchAttributeClusterDimension;
            ca.val.clusterDim.x = 2;
            ca.val.clusterDim.y = 1;
            ca.val.clusterDim.z = 1;
            q.attrs = &ca;
            q.numAttrs = 1;
            int n = 0;
            ok_dev[dev] = cudaOccupancyMaxActiveClusters(&n, kernel, &q) == cudaSuccess && n > 0;
            pairs_dev[dev] = n;
        }
    });
    if (!ok_dev[dev]) { (void)cudaGetLastError(); return BSQ_ERR_CUDA; }
    const int64_t tiles = ((a.M + C::kTileM - 1) / C::kTileM) * ((a.N + BN - 1) / BN);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    // programmatic dependent launch: the prologue may overlap the previous kernel
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if constexpr (PAIR) {
        // persistent CTA pairs, no more than can be resident together (a pair
        // that had to wait for another to finish would serialize its tiles)
        cfg.gridDim = dim3((unsigned)(2 * imin64(tiles, pairs_dev[dev])), 1, 1);
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    } else if constexpr (GROUPED) {
        // the tile count depends on the device row counts: one persistent CTA per SM
        cfg.gridDim = dim3((unsigned)imin64(a.G * tiles, info->num_sms), 1, 1);
    } else if constexpr (SPLIT == 1) {
        // in-kernel A quantization runs one tile per CTA (no persistence)
        cfg.gridDim = dim3((unsigned)(QA >= 0 ? tiles : imin64(tiles, info->num_sms)), 1, 1);
    } else {
        cfg.gridDim = dim3((unsigned)(tiles * SPLIT), 1, 1);
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = SPLIT;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kernel, mp.a, mp.w, mp.sa, mp.sw, a) != cudaSuccess) {
        (void)cudaGetLastError();
        return BSQ_ERR_CUDA;
    }
    return BSQ_OK;
}

}  // namespace

bsq_status gemm_launch(const void* A, int fa, const uint8_t* sA, const float* gA, const void* W, int fw,
                       const uint8_t* sW, const float* gW, void* Y, int out, int64_t M, int64_t N, int64_t K,
                       bool nvf4, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    // BN = 256 when that still gives every SM a tile, else 128; when even the
    // 128-wide tiles leave most SMs idle, split K across a cluster.
    const int64_t tiles256 = ((M + kBM - 1) / kBM) * ((N + 255) / 256);
    const int64_t tiles128 = ((M + kBM - 1) / kBM) * ((N + 127) / 128);
    const int64_t pair_tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + 255) / 256);
    const int bn = tiles256 >= info->num_sms ? 256 : 128;
    // 256 x 256 tiles on CTA pairs when A has more than one 128-row block and
    // the pair tiles still give every pair of SMs one: each SM then stages half
    // of B, halving the shared-memory traffic of the B operand per MMA
    const bool pair = bn == 256 && M > kBM && pair_tiles >= info->num_sms / 2;
    const int64_t nks = (K + (nvf4 ? 255 : 127)) / (nvf4 ? 256 : 128);
    int split = 1;
    if (bn == 128)
        for (int sp = 8; sp >= 2; sp /= 2)
            if (tiles128 * sp <= info->num_sms && nks >= sp) { split = sp; break; }
    const uint32_t rows_b = pair ? 128u : (uint32_t)bn;     // W rows one CTA stages per tile
    const int64_t cpd4 = pad_to(K / (nvf4 ? 16 : 32), 4) / 4;
    const uint32_t stage_atoms = nvf4 ? 4u : 1u;
    Maps mp;
    if (!operand_map(&mp.a, A, fa, nvf4, M, K, kBM) || !operand_map(&mp.w, W, fw, nvf4, N, K, rows_b) ||
        !scale_map(&mp.sa, sA, pad_to(M, 128) / 128, cpd4, stage_atoms, 1) ||
        !scale_map(&mp.sw, sW, pad_to(N, 128) / 128, cpd4, stage_atoms, (uint32_t)(bn / 128)))
        return BSQ_ERR_CUDA;
    GemmArgs a;
    a.gA = gA; a.gW = gW; a.Y = Y;
    a.M = M; a.N = N; a.K = K;
    a.row_counts = nullptr; a.G = 1;
    a.qx = nullptr; a.qpartial = nullptr; a.qn_partial = 0; a.qs_global = nullptr;
    a.out_bf16 = out == BSQ_OUT_BF16;
    a.idesc = make_idesc(nvf4, fa, fw, bn, pair ? 2 * kBM : kBM);
    a.err = info->err;
    // A 16U6_ALIGN16B load lands 128 bytes per 128-code row in shared memory but
    // counts the 96 packed bytes it read toward the transaction.
    auto row_tx = [&](int f) { return (uint32_t)(nvf4 || f == kE4M3 ? 128 : 96); };
    a.tx_ab = kBM * row_tx(fa) + rows_b * row_tx(fw);
    bsq_status r;
    if (pair) {
        if (nvf4) r = launch_gemm<true, 256, 1, false, -1, true>(info, mp, a, s);
        else r = launch_gemm<false, 256, 1, false, -1, true>(info, mp, a, s);
    } else if (nvf4) {
        if (bn == 256) r = launch_gemm<true, 256, 1>(info, mp, a, s);
        else if (split == 8) r = launch_gemm<true, 128, 8>(info, mp, a, s);
        else if (split == 4) r = launch_gemm<true, 128, 4>(info, mp, a, s);
        else if (split == 2) r = launch_gemm<true, 128, 2>(info, mp, a, s);
        else r = launch_gemm<true, 128, 1>(info, mp, a, s);
    } else {
        if (bn == 256) r = launch_gemm<false, 256, 1>(info, mp, a, s);
        else if (split == 8) r = launch_gemm<false, 128, 8>(info, mp, a, s);
        else if (split == 4) r = launch_gemm<false, 128, 4>(info, mp, a, s);
        else if (split == 2) r = launch_gemm<false, 128, 2>(info, mp, a, s);
        else r = launch_gemm<false, 128, 1>(info, mp, a, s);
    }
    count_launch(nvf4 ? BSQ_KERNEL_GEMM_NVFP4 : BSQ_KERNEL_GEMM_MX);
    return r;
}


bsq_status gemm_grouped_launch(const void* A, int fa, const uint8_t* sA, const float* gA, const void* W, int fw,
                               const uint8_t* sW, const float* gW, const int32_t* row_counts, void* Y, int out,
                               int64_t G, int64_t R, int64_t N, int64_t K, bool nvf4, cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    // 256-wide W tiles when the groups' full row blocks would still give every SM one
    const int64_t full256 = G * ((R + kBM - 1) / kBM) * ((N + 255) / 256);
    const int bn = full256 >= info->num_sms ? 256 : 128;
    const int64_t nblk = K / (nvf4 ? 16 : 32);
    const int64_t cpd4 = pad_to(nblk, 4) / 4;
    Maps mp;
    if (!operand_map(&mp.a, A, fa, nvf4, G * R, K, kBM) || !operand_map(&mp.w, W, fw, nvf4, G * N, K, (uint32_t)bn) ||
        !scale_map(&mp.sa, sA, G * (pad_to(R, 128) / 128), cpd4, nvf4 ? 4u : 1u, 1) ||
        !scale_map(&mp.sw, sW, G * (pad_to(N, 128) / 128), cpd4, nvf4 ? 4u : 1u, (uint32_t)(bn / 128)))
        return BSQ_ERR_CUDA;
    GemmArgs a;
    a.gA = gA; a.gW = gW; a.Y = Y;
    a.M = R; a.N = N; a.K = K;
    a.row_counts = row_counts; a.G = G;
    a.qx = nullptr; a.qpartial = nullptr; a.qn_partial = 0; a.qs_global = nullptr;
    a.out_bf16 = out == BSQ_OUT_BF16;
    a.idesc = make_idesc(nvf4, fa, fw, bn);
    a.err = info->err;
    auto row_tx = [&](int f) { return (uint32_t)(nvf4 || f == kE4M3 ? 128 : 96); };
    a.tx_ab = kBM * row_tx(fa) + (uint32_t)bn * row_tx(fw);
    bsq_status r;
    if (nvf4) r = bn == 256 ? launch_gemm<true, 256, 1, true>(info, mp, a, s) : launch_gemm<true, 128, 1, true>(info, mp, a, s);
    else r = bn == 256 ? launch_gemm<false, 256, 1, true>(info, mp, a, s) : launch_gemm<false, 128, 1, true>(info, mp, a, s);
    count_launch(nvf4 ? BSQ_KERNEL_GEMM_NVFP4 : BSQ_KERNEL_GEMM_MX);
    return r;
}


bsq_status gemm_quant_a_launch(const uint16_t* x, int fa, const void* W, int fw, const uint8_t* sW, const float* gW,
                               void* Y, int out, float* s_global_a, int64_t M, int64_t N, int64_t K, uint32_t* partial,
                               cudaStream_t s) {
    bsq_status st;
    const DeviceInfo* info = device_info(&st);
    if (!info) return st;
    // the amax pass over x, then the GEMM (a programmatic dependent launch that
    // reduces the partial maxima before it quantizes A)
    const int n_partial = amax_partials_launch(x, M * K, partial, s);
    if (n_partial < 0) return BSQ_ERR_CUDA;
    const int64_t tiles128 = ((M + kBM - 1) / kBM) * ((N + 127) / 128);
    const int64_t nks = (K + 127) / 128;
    int split = 1;
    for (int sp = 8; sp >= 2; sp /= 2)
        if (tiles128 * sp <= info->num_sms && nks >= sp) { split = sp; break; }
    Maps mp;
    if (!operand_map(&mp.w, W, fw, false, N, K, 128u) ||
        !scale_map(&mp.sw, sW, pad_to(N, 128) / 128, pad_to(K / 32, 4) / 4, 1, 1))
        return BSQ_ERR_CUDA;
    mp.sa = mp.sw;        // A's scales are made in the kernel; this map is never read
    // x [M, K] bf16 as 64-value boxes of 128 rows (128-byte swizzle, zeros past M and K)
    if (!encode_map(&mp.a, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, (uint64_t)K, (uint64_t)M, (uint64_t)(K * 2), 64, 128))
        return BSQ_ERR_CUDA;
    GemmArgs a;
    a.gA = nullptr; a.gW = gW; a.Y = Y;
    a.M = M; a.N = N; a.K = K;
    a.row_counts = nullptr; a.G = 1;
    a.qx = x; a.qpartial = partial; a.qn_partial = n_partial; a.qs_global = s_global_a;
    a.out_bf16 = out == BSQ_OUT_BF16;
    a.idesc = make_idesc(false, fa, fw, 128);
    a.err = info->err;
    a.tx_ab = 128u * (fw == kE4M3 ? 128u : 96u) + (uint32_t)(kBM * 128 * 2);   // the W tile and A's bf16 tile
    bsq_status r;
#define BSQ_QA_SPLITS(F)                                                            \
    if (split == 8) r = launch_gemm<false, 128, 8, false, F>(info, mp, a, s);   \
    else if (split == 4) r = launch_gemm<false, 128, 4, false, F>(info, mp, a, s); \
    else if (split == 2) r = launch_gemm<false, 128, 2, false, F>(info, mp, a, s); \
    else r = launch_gemm<false, 128, 1, false, F>(info, mp, a, s);
    switch (fa) {
    case kE3M2: BSQ_QA_SPLITS(kE3M2); break;
    case kE2M3: BSQ_QA_SPLITS(kE2M3); break;
    default: BSQ_QA_SPLITS(kE4M3); break;
    }
#undef BSQ_QA_SPLITS
    count_launch(BSQ_KERNEL_GEMM_MX);
    return r;
}

}  // namespace bsq
