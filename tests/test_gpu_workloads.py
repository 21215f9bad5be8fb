"""The five workloads at full size, in the launch configuration the benchmark
times.

Quantizers: the oracle quantizes the whole tensor from the same bf16 input and
every byte of the GPU's codes and scale buffer, and s_global, must equal it.

Products: the expected values come only from the oracle's own quantized
operands (equal to the GPU's, as just checked).  The decode GEMVs and the W6A6
GEMM are checked on every output.  The two large GEMMs are checked on every
output of every row and every column that sits on either side of a 128-row or
128-column tile boundary (0, 127, 128, 255, 256, ...), plus a seeded sample of
4096 outputs computed one by one by the oracle's plain product.  Row and column
blocks are the oracle's exact decode of each operand (in double) multiplied by a
float64 library matmul.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import boundary_index, check_products, dev_tensor, host_bytes, products_by_blocks, sample_pairs

pytestmark = pytest.mark.gpu

W = S.WORKLOADS
CHUNK_ROWS = 2048          # rows decoded at a time (a multiple of the 128-row scale tile)


def check_quantized_mx(x, fmt, codes_d, scales_d, g_d):
    oc, os_, og = O.quantize_mx(x, fmt)
    assert np.float32(g_d.item()) == np.float32(og)
    assert np.array_equal(host_bytes(codes_d).reshape(oc.shape), oc)
    assert np.array_equal(host_bytes(scales_d), os_)
    return oc, os_, og


def check_quantized_nvfp4(x, codes_d, scales_d, g_d):
    oc, os_, og = O.quantize_nvfp4(x)
    assert np.float32(g_d.item()) == np.float32(og)
    assert np.array_equal(codes_d.cpu().numpy().view(np.uint32).reshape(oc.shape), oc)
    assert np.array_equal(host_bytes(scales_d), os_)
    return oc, os_, og


def decoded_chunks(codes, scales, K, fmt=None):
    """(r0, r1, exact decode of rows [r0, r1) without the tensor factor), whole
    128-row scale tiles at a time.  fmt None: nvfp4."""
    R = codes.shape[0]
    blk = 16 if fmt is None else 32
    tile_bytes = -(-(K // blk) // 4) * 512
    for r0 in range(0, R, CHUNK_ROWS):
        r1 = min(R, r0 + CHUNK_ROWS)
        sc = scales[(r0 // 128) * tile_bytes:(-(-r1 // 128)) * tile_bytes]
        if fmt is None:
            d = O.dequant_nvfp4(codes[r0:r1], sc, 1.0, r1 - r0, K)
        else:
            d = O.dequant_mx(codes[r0:r1], fmt, sc, 1.0, r1 - r0, K)
        yield r0, r1, d


def gather_rows(codes, scales, K, rows, fmt=None):
    out = np.empty((rows.size, K))
    for r0, r1, d in decoded_chunks(codes, scales, K, fmt):
        sel = (rows >= r0) & (rows < r1)
        out[sel] = d[rows[sel] - r0]
    return out


def check_gemm_boundaries(y, A, sA, fa, W_, sW, fw, g, M, N, K, what):
    """Every output of the tile-boundary rows and columns of Y = g * A W^T."""
    rb, cb = boundary_index(M), boundary_index(N)
    a_rows = gather_rows(A, sA, K, rb, fa)
    w_rows = gather_rows(W_, sW, K, cb, fw)
    yr = np.empty((rb.size, N)); sr = np.empty_like(yr)
    for r0, r1, dw in decoded_chunks(W_, sW, K, fw):
        yr[:, r0:r1], sr[:, r0:r1] = products_by_blocks(a_rows, dw, g)
    check_products(y[torch.from_numpy(rb)], yr, sr, f"{what}: boundary rows")
    yc = np.empty((M, cb.size)); sc = np.empty_like(yc)
    for r0, r1, da in decoded_chunks(A, sA, K, fa):
        yc[r0:r1], sc[r0:r1] = products_by_blocks(da, w_rows, g)
    check_products(y[:, torch.from_numpy(cb)], yc, sc, f"{what}: boundary columns")


def test_nvfp4_one_row_gemv_256(bsq):
    c = W["nvfp4_gemv_1x256x256"]
    M, N, K = c["M"], c["N"], c["K"]
    x = S.normal_bf16((M, K), c["x_std"], c["seed"])
    Wc = S.random_words((N, K // 8), c["seed"] + 1)
    sc = S.choice_bytes(O.scale_bytes(N, K // 16), c["seed"] + 2, S.UE4M3_POW2_M4_TO_P4)
    g = torch.tensor([c["g_w"]], device="cuda")
    y = bsq.gemv_nvfp4(dev_tensor(x), dev_tensor(Wc), dev_tensor(sc), g, K, out_dtype=torch.float32)
    want, s = O.gemv_nvfp4(x, Wc, sc, c["g_w"], M, N, K)
    check_products(y, want, s, "config 1")


def test_mxfp6_w6a6_e3m2_128x4096x4096(bsq):
    c = W["mxfp6_e3m2_w6a6_128x4096x4096"]
    M, N, K = c["M"], c["N"], c["K"]
    a = S.normal_bf16((M, K), c["a_std"], c["seed"] + 1, outlier_frac=c["outlier_frac"], outlier_mult=c["outlier_mult"])
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 2, outlier_frac=c["outlier_frac"], outlier_mult=c["outlier_mult"])
    ca, sa, ga = bsq.quantize_mxfp6(dev_tensor(a), "e3m2")
    cw, sw, gw = bsq.quantize_mxfp6(dev_tensor(w), "e3m2")
    y = bsq.gemm_mxfp6(ca, "e3m2", sa, ga, cw, "e3m2", sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    oca, osa, oga = check_quantized_mx(a, O.E3M2, ca, sa, ga)
    ocw, osw, ogw = check_quantized_mx(w, O.E3M2, cw, sw, gw)
    g = float(np.float32(oga)) * float(np.float32(ogw))
    da = gather_rows(oca, osa, K, np.arange(M), O.E3M2)
    yw = np.empty((M, N)); sw_ = np.empty_like(yw)
    for r0, r1, dw in decoded_chunks(ocw, osw, K, O.E3M2):
        yw[:, r0:r1], sw_[:, r0:r1] = products_by_blocks(da, dw, g)
    check_products(y, yw, sw_, "config 2: every output")


@pytest.mark.parametrize("M", [1, 8, 32])
def test_nvfp4_decode_gemv_28672x8192(bsq, M):
    c = W["nvfp4_decode_gemv_Mx28672x8192"]
    N, K = c["N"], c["K"]
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 1)
    cw, sw, gw = bsq.quantize_nvfp4(dev_tensor(w))
    x = S.normal_bf16((M, K), c["x_std"], c["seed"] + 2 + M)
    y = bsq.gemv_nvfp4(dev_tensor(x), cw, sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ocw, osw, ogw = check_quantized_nvfp4(w, cw, sw, gw)
    xd = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = np.empty((M, N)); s = np.empty_like(want)
    for r0, r1, dw in decoded_chunks(ocw, osw, K):
        want[:, r0:r1], s[:, r0:r1] = products_by_blocks(xd, dw, float(np.float32(ogw)))
    check_products(y, want, s, f"config 3 M={M}: every output")
    # and a seeded sample through the oracle's one-by-one product
    mi, ni = sample_pairs(M, N, 4096, 7 + M)
    want1, s1 = O.gemv_nvfp4(x, ocw, osw, ogw, M, N, K, mi=mi, ni=ni)
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want1, s1, f"config 3 M={M}: sample")


def test_nvfp4_prefill_gemm_8192(bsq):
    c = W["nvfp4_prefill_gemm_8192"]
    M, N, K = c["M"], c["N"], c["K"]
    a = S.normal_bf16((M, K), c["a_std"], c["seed"] + 1)
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 2)
    ca, sa, ga = bsq.quantize_nvfp4(dev_tensor(a))
    cw, sw, gw = bsq.quantize_nvfp4(dev_tensor(w))
    y = bsq.gemm_nvfp4(ca, sa, ga, cw, sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    oca, osa, oga = check_quantized_nvfp4(a, ca, sa, ga)
    ocw, osw, ogw = check_quantized_nvfp4(w, cw, sw, gw)
    mi, ni = sample_pairs(M, N, 4096, 11)
    want, s = O.gemm_nvfp4(oca, osa, oga, ocw, osw, ogw, M, N, K, mi=mi, ni=ni)
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, "config 4: sample")
    g = float(np.float32(oga)) * float(np.float32(ogw))
    check_gemm_boundaries(y, oca, osa, None, ocw, osw, None, g, M, N, K, "config 4")


def test_w6a8_e4m3xe2m3_4096x14336x4096(bsq):
    c = W["w6a8_e4m3xe2m3_4096x14336x4096"]
    M, N, K = c["M"], c["N"], c["K"]
    a = S.normal_bf16((M, K), c["a_std"], c["seed"] + 1)
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 2)
    ca, sa, ga = bsq.quantize_mxfp6(dev_tensor(a), "e4m3")
    cw, sw, gw = bsq.quantize_mxfp6(dev_tensor(w), "e2m3")
    y = bsq.gemm_mxfp6(ca, "e4m3", sa, ga, cw, "e2m3", sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    oca, osa, oga = check_quantized_mx(a, O.E4M3, ca, sa, ga)
    ocw, osw, ogw = check_quantized_mx(w, O.E2M3, cw, sw, gw)
    mi, ni = sample_pairs(M, N, 4096, 13)
    want, s = O.gemm_mx(oca, O.E4M3, osa, oga, ocw, O.E2M3, osw, ogw, M, N, K, mi=mi, ni=ni)
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, "config 5 GEMM: sample")
    g = float(np.float32(oga)) * float(np.float32(ogw))
    check_gemm_boundaries(y, oca, osa, O.E4M3, ocw, osw, O.E2M3, g, M, N, K, "config 5 GEMM")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w6a8_small_m_quantizer(bsq, M):
    c = W["w6a8_e4m3xe2m3_4096x14336x4096"]
    K = c["K"]
    x = S.normal_bf16((M, K), 1.0, c["seed"] + 10 + M)
    bsq.reset_launch_counts()
    codes, scales, g = bsq.quantize_mxfp6(dev_tensor(x), "e2m3")
    torch.cuda.synchronize()
    assert bsq.launch_count("quant_small") == 1 and bsq.launch_count("amax") == 0
    oc, os_, og = O.quantize_mx(x, O.E2M3)
    assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
    assert np.array_equal(host_bytes(scales), os_)
    assert np.float32(g.item()) == np.float32(og)
