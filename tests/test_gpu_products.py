"""GPU products against the oracle, output by output: the nvfp4 and MX
decode GEMVs (mma.sync path) and the tcgen05 block-scaled GEMMs, on shapes that
span several tiles and ragged tails in M, N and K, with fp32 and bf16 output."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import check_products, dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

# ue4m3 block scales spread over 2^-6 .. 2^7 with all mantissas
UE4M3_CODES = list(range(0x08, 0x68))
MX = {"e3m2": O.E3M2, "e2m3": O.E2M3, "e4m3": O.E4M3}


def nvfp4_operand(R, K, seed):
    W = S.random_words((R, K // 8), seed)
    sc = S.choice_bytes(O.scale_bytes(R, K // 16), seed + 1, UE4M3_CODES)
    return W, sc


def mx_operand(R, K, fmt_name, seed):
    """Quantized from bf16 by the oracle (the codes and scales a quantizer makes)."""
    x = S.normal_bf16((R, K), 0.02, seed, outlier_frac=0.01)
    return O.quantize_mx(x, MX[fmt_name])


@pytest.mark.parametrize("M", [1, 2, 5, 8, 13, 17, 32])
@pytest.mark.parametrize("N,K", [(256, 256), (300, 320), (129, 1024), (1, 64), (200, 4160), (1000, 2048)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_gemv_nvfp4(bsq, M, N, K, out):
    x = S.normal_bf16((M, K), 1.0, 7 + M)
    W, sc = nvfp4_operand(N, K, 31 + N + K)
    g = torch.tensor([0.375], device="cuda")
    y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), g, K, out_dtype=out)
    want, s = O.gemv_nvfp4(x, W, sc, 0.375, M, N, K)
    check_products(y, want, s, f"gemv_nvfp4 M{M} N{N} K{K}")


def test_gemv_nvfp4_every_code_and_subnormal_scales(bsq):
    """Every e2m1 code (both zeros, the 0.5 subnormal) against ue4m3 scales that
    include e4m3 subnormals, so the exact in-register decode is exercised end to end."""
    M, N, K = 3, 128, 512
    x = S.normal_bf16((M, K), 1.0, 9)
    codes = (np.arange(N * K) % 16).astype(np.uint32).reshape(N, K)
    W = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        W |= codes[:, j::8] << np.uint32(4 * j)
    sc = S.choice_bytes(O.scale_bytes(N, K // 16), 3, list(range(0x01, 0x7F)))
    y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), None, K, out_dtype=torch.float32)
    want, s = O.gemv_nvfp4(x, W, sc, 1.0, M, N, K)
    check_products(y, want, s, "gemv_nvfp4 all codes")


@pytest.mark.parametrize("M", [1, 2, 8, 17, 32])
def test_gemv_nvfp4_activations_outside_f16(bsq, M):
    """Activations that f16 cannot hold exactly (huge, tiny, bf16 subnormal) in
    some 256-wide K chunks and not in others: those chunks take the bf16 decode,
    the rest the f16 one, in the same call and the same outputs.  Columns 300 and
    1200 put such values in the first and in the second 128-wide half of a stage
    (the tensor-core kernel's granules; 1152..1279 is bf16 while 1024..1151 stays f16)."""
    N, K = 300, 1536
    x = S.normal_bf16((M, K), 1.0, 40 + M)
    x[:, 300] = 0x4B80          # 1.68e7  (> f16 max)
    x[:, 1200] = 0x4B80
    x[:, 777] = 0x3380          # 5.96e-8 (below the f16 normal range)
    x[0, 1300] = 0x0005         # bf16 subnormal
    x[-1, 1301] = 0xC780        # -65536 (just beyond f16)
    W, sc = nvfp4_operand(N, K, 44)
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), None, K, out_dtype=out)
        want, s = O.gemv_nvfp4(x, W, sc, 1.0, M, N, K)
        check_products(y, want, s, f"gemv_nvfp4 mixed chunks M{M}")


@pytest.mark.parametrize("M", [1, 8, 32])
def test_gemv_nvfp4_activations_on_f16_subnormals(bsq, M):
    """A whole activation row of values in [2^-17, 2^-14): bf16 values with
    exponent field 110..112 are exact f16 subnormals, so they take the f16 path;
    were subnormal operands flushed, that row's outputs would be lost entirely
    (its sum_k |x_k w_k| is of the same tiny size).  Values of field 109 and below
    elsewhere still take the exact bf16 path."""
    N, K = 300, 1024
    g = np.random.default_rng(70 + M)
    x = S.normal_bf16((M, K), 1.0, 71 + M)
    field = g.integers(110, 113, K).astype(np.uint16)
    x[0] = (g.integers(0, 2, K).astype(np.uint16) << 15) | (field << 7) | g.integers(0, 128, K).astype(np.uint16)
    if M > 1:
        x[1, ::97] = 0x3480                     # 2^-22: below the f16-exact range (a bf16 stage)
    W, sc = nvfp4_operand(N, K, 72)
    want, s = O.gemv_nvfp4(x, W, sc, 1.0, M, N, K)
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), None, K, out_dtype=out)
        check_products(y, want, s, f"gemv_nvfp4 f16-subnormal activations M{M}")


# bf16 magnitudes at the edges of "exactly an f16 value": exponent fields 109
# (not exact: an f16 subnormal cannot hold 8 significant bits there), 110 and
# 112 (exact f16 subnormals), 113 (smallest f16 normal binade), 142 (largest
# f16 binade) and 143 (beyond f16), each with mantissas 0, 1 and 127.
F16_EDGE_BITS = [(e << 7) | m for e in (109, 110, 112, 113, 142, 143) for m in (0, 1, 127)]


@pytest.mark.parametrize("M", [1, 8, 32])
def test_gemv_nvfp4_activations_at_the_f16_edges(bsq, M):
    """Each activation row made of one edge magnitude (random signs), so that a
    wrong f16 decision shows in every output: a value taken as exact in f16
    when it is not is rounded by ~2^-7 relative (or overflows), far beyond
    the tolerance for outputs made only of such values."""
    N, K = 96, 512
    W, sc = nvfp4_operand(N, K, 80 + M)
    g = np.random.default_rng(81 + M)
    for bits in F16_EDGE_BITS:
        sign = g.integers(0, 2, (M, K)).astype(np.uint16) << 15
        x = (sign | np.uint16(bits)).astype(np.uint16)
        want, s = O.gemv_nvfp4(x, W, sc, 1.0, M, N, K)
        y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), None, K, out_dtype=torch.float32)
        check_products(y, want, s, f"gemv_nvfp4 M{M} activations 0x{bits:04x}")


@pytest.mark.parametrize("M", [17, 32])
def test_gemv_nvfp4_tensor_core_many_tiles(bsq, M):
    """The tensor-core decode product with more 192-row CTAs than SMs (a second
    wave) and a ragged last CTA whose second 128-row tile is partly past N;
    activations outside f16 in one 256-wide K chunk take the bf16 decode in
    the same call."""
    N, K = 2 * 152 * 128 + 100, 512
    x = S.normal_bf16((M, K), 1.0, 50 + M)
    x[:, 300] = 0x4B80          # > f16 max: that 256-wide chunk takes the bf16 decode
    W, sc = nvfp4_operand(N, K, 52)
    g = torch.tensor([0.625], device="cuda")
    want, s = O.gemv_nvfp4(x, W, sc, 0.625, M, N, K)
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(W), dev_tensor(sc), g, K, out_dtype=out)
        check_products(y, want, s, f"gemv_nvfp4 many tiles M{M}")


@pytest.mark.parametrize("fmt", ["e3m2", "e2m3", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (8, 300, 512), (32, 129, 384)])
def test_gemv_mx(bsq, fmt, M, N, K):
    x = S.normal_bf16((M, K), 1.0, 17 + M)
    codes, sc, g = mx_operand(N, K, fmt, 41 + N)
    gt = torch.tensor([g], device="cuda")
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemv_mxfp6(dev_tensor(x), dev_tensor(codes), fmt, dev_tensor(sc), gt, K, out_dtype=out)
        want, s = O.gemv_mx(x, codes, MX[fmt], sc, g, M, N, K)
        check_products(y, want, s, f"gemv_{fmt} M{M} N{N} K{K}")


def swizzle_plain(plain):
    """Row-major [rows, blocks] scale bytes -> the swizzled buffer (the oracle's offset rule)."""
    rows, blocks = plain.shape
    buf = np.zeros(O.scale_bytes(rows, blocks), dtype=np.uint8)
    for r in range(rows):
        for b in range(blocks):
            buf[O.swz_offset(r, b, blocks)] = plain[r, b]
    return buf


@pytest.mark.parametrize("fmt", ["e3m2", "e2m3", "e4m3"])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_gemv_mx_every_ue8m0_byte(bsq, fmt, M):
    """Block scales covering every UE8M0 byte 0..254 (2^-127 .. 2^127; byte 0
    read as 2^-127).  Two bands keep every output finite in fp32: bytes 0..140
    with N(0,1) activations, bytes 115..254 with activations scaled by 2^-24;
    within a row the blocks' scales are mixed across the whole band."""
    N, K = 300, 512
    nb = K // 32
    g = np.random.default_rng(2000 + M)
    rb = K if fmt == "e4m3" else 3 * K // 4
    codes = g.integers(0, 256, size=(N, rb), dtype=np.uint8)
    if fmt == "e4m3":
        codes[(codes & 0x7F) == 0x7F] &= 0xFE            # no NaN codes
    for lo, hi, xstd in ((0, 140, 1.0), (115, 254, 2.0 ** -24)):
        plain = g.integers(lo, hi + 1, size=(N, nb)).astype(np.uint8)
        plain.ravel()[:hi - lo + 1] = np.arange(lo, hi + 1, dtype=np.uint8)   # every byte of the band occurs
        sc = swizzle_plain(plain)
        x = S.normal_bf16((M, K), xstd, 2100 + M + lo)
        want, s = O.gemv_mx(x, codes, MX[fmt], sc, 1.0, M, N, K)
        assert np.isfinite(want).all()
        for out in (torch.float32, torch.bfloat16):
            y = bsq.gemv_mxfp6(dev_tensor(x), dev_tensor(codes), fmt, dev_tensor(sc), None, K, out_dtype=out)
            check_products(y, want, s, f"gemv_{fmt} M{M} UE8M0 bytes {lo}..{hi}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (200, 333, 320), (1, 256, 64), (256, 512, 1024),
                                   (384, 1024, 512), (130, 4096, 256), (200, 336, 256)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_gemm_nvfp4(bsq, M, N, K, out):
    A, sA = nvfp4_operand(M, K, 51 + M)
    W, sW = nvfp4_operand(N, K, 61 + N)
    gA = torch.tensor([0.5], device="cuda")
    gW = torch.tensor([0.25], device="cuda")
    y = bsq.gemm_nvfp4(dev_tensor(A), dev_tensor(sA), gA, dev_tensor(W), dev_tensor(sW), gW, K, out_dtype=out)
    want, s = O.gemm_nvfp4(A, sA, 0.5, W, sW, 0.25, M, N, K)
    check_products(y, want, s, f"gemm_nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("fa,fw", [(a, w) for a in ("e3m2", "e2m3", "e4m3") for w in ("e3m2", "e2m3", "e4m3")])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 333, 384), (256, 1024, 1024), (1, 300, 256)])
def test_gemm_mx(bsq, fa, fw, M, N, K):
    A, sA, gA = mx_operand(M, K, fa, 71 + M)
    W, sW, gW = mx_operand(N, K, fw, 81 + N)
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemm_mxfp6(dev_tensor(A), fa, dev_tensor(sA), torch.tensor([gA], device="cuda"),
                           dev_tensor(W), fw, dev_tensor(sW), torch.tensor([gW], device="cuda"), K, out_dtype=out)
        want, s = O.gemm_mx(A, MX[fa], sA, gA, W, MX[fw], sW, gW, M, N, K)
        check_products(y, want, s, f"gemm_{fa}x{fw} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1100, 4315, 256), (1024, 9728, 128), (1100, 4400, 128)])
def test_gemm_nvfp4_many_tiles(bsq, M, N, K):
    """More 256 x 256 tiles than pairs of SMs (the persistent CTA-pair path)
    with several row blocks, an odd row-block count with a ragged last block,
    and a ragged N edge; every output checked."""
    A, sA = nvfp4_operand(M, K, 91 + M)
    W, sW = nvfp4_operand(N, K, 93 + N)
    gA = torch.tensor([0.5], device="cuda")
    gW = torch.tensor([0.75], device="cuda")
    y = bsq.gemm_nvfp4(dev_tensor(A), dev_tensor(sA), gA, dev_tensor(W), dev_tensor(sW), gW, K,
                       out_dtype=torch.bfloat16)
    want, s = O.gemm_nvfp4(A, sA, 0.5, W, sW, 0.75, M, N, K)
    check_products(y, want, s, f"gemm_nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(300, 9800, 320), (2048, 4864, 512)])
def test_gemm_nvfp4_pair_tiles(bsq, M, N, K):
    """256 x 256 tiles on CTA pairs: rank 0 issues MMAs over both CTAs' A rows
    and W halves.  300 rows leave the second pair tile's rank 1 entirely past M
    (zero-filled rows, clamped scale tile) and rank 0 ragged; N = 9800 leaves the
    last W tile's second half past N; K = 320 ends in a one-MMA stage."""
    A, sA = nvfp4_operand(M, K, 101 + M)
    W, sW = nvfp4_operand(N, K, 103 + N)
    gA = torch.tensor([0.5], device="cuda")
    gW = torch.tensor([1.5], device="cuda")
    want, s = O.gemm_nvfp4(A, sA, 0.5, W, sW, 1.5, M, N, K)
    for out in (torch.float32, torch.bfloat16):
        y = bsq.gemm_nvfp4(dev_tensor(A), dev_tensor(sA), gA, dev_tensor(W), dev_tensor(sW), gW, K, out_dtype=out)
        check_products(y, want, s, f"gemm_nvfp4 pair {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["nvfp4", "e4m3xe2m3"])
def test_gemm_single_cta_256_wide(bsq, kind):
    """One 128-row block of A and more 256-wide W tiles than SMs: the product
    stays on single-CTA 128 x 256 tiles (a CTA pair would idle its second half)."""
    M, N, K = 100, 152 * 256 + 40, 128
    if kind == "nvfp4":
        A, sA = nvfp4_operand(M, K, 105)
        W, sW = nvfp4_operand(N, K, 106)
        y = bsq.gemm_nvfp4(dev_tensor(A), dev_tensor(sA), None, dev_tensor(W), dev_tensor(sW), None, K,
                           out_dtype=torch.bfloat16)
        want, s = O.gemm_nvfp4(A, sA, 1.0, W, sW, 1.0, M, N, K)
    else:
        A, sA, gA = mx_operand(M, K, "e4m3", 107)
        W, sW, gW = mx_operand(N, K, "e2m3", 108)
        y = bsq.gemm_mxfp6(dev_tensor(A), "e4m3", dev_tensor(sA), torch.tensor([gA], device="cuda"),
                           dev_tensor(W), "e2m3", dev_tensor(sW), torch.tensor([gW], device="cuda"), K,
                           out_dtype=torch.bfloat16)
        want, s = O.gemm_mx(A, O.E4M3, sA, gA, W, O.E2M3, sW, gW, M, N, K)
    check_products(y, want, s, f"gemm {kind} {M}x{N}x{K}")


@pytest.mark.parametrize("fa,fw,N,out", [("e4m3", "e2m3", 4315, torch.float32), ("e3m2", "e3m2", 4315, torch.float32),
                                         ("e4m3", "e2m3", 4400, torch.bfloat16), ("e3m2", "e3m2", 4315, torch.bfloat16)])
def test_gemm_mx_many_tiles(bsq, fa, fw, N, out):
    """The persistent 256 x 256 CTA-pair path for MX operands (fp6 W included)
    on a ragged shape with more tiles than pairs of SMs; every output checked.  N = 4400 (a
    multiple of 16, not of the tile) takes the whole-line bf16 stores up to a
    ragged column edge."""
    M, K = 1100, 256
    A, sA, gA = mx_operand(M, K, fa, 95)
    W, sW, gW = mx_operand(N, K, fw, 97)
    y = bsq.gemm_mxfp6(dev_tensor(A), fa, dev_tensor(sA), torch.tensor([gA], device="cuda"),
                       dev_tensor(W), fw, dev_tensor(sW), torch.tensor([gW], device="cuda"), K,
                       out_dtype=out)
    want, s = O.gemm_mx(A, MX[fa], sA, gA, W, MX[fw], sW, gW, M, N, K)
    check_products(y, want, s, f"gemm_{fa}x{fw} {M}x{N}x{K}")


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_gemm_output_16_byte_aligned_only(bsq, out):
    """Y 16-byte but not 32-byte aligned: the epilogue falls back from
    32-byte stores to 16-byte ones; the words around Y are not touched."""
    M, N, K = 1100, 4400, 128
    A, sA = nvfp4_operand(M, K, 99)
    W, sW = nvfp4_operand(N, K, 98)
    gA = torch.tensor([0.5], device="cuda")
    gW = torch.tensor([0.75], device="cuda")
    pad = 16 // torch.tensor([], dtype=out).element_size()
    buf = torch.full((M * N + 2 * pad,), 7.0, dtype=out, device="cuda")
    Y = buf[pad:pad + M * N].view(M, N)
    assert Y.data_ptr() % 32 == 16
    bsq.gemm_nvfp4_(dev_tensor(A), dev_tensor(sA), gA, dev_tensor(W), dev_tensor(sW), gW, Y, M, N, K)
    torch.cuda.synchronize()
    want, s = O.gemm_nvfp4(A, sA, 0.5, W, sW, 0.75, M, N, K)
    check_products(Y, want, s, f"gemm_nvfp4 {M}x{N}x{K}, Y at 16 mod 32")
    assert (buf[:pad] == 7.0).all() and (buf[pad + M * N:] == 7.0).all()
