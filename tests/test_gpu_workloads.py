"""The five workloads at full size, in the launch configuration the benchmark
times.  Quantizer outputs are compared bit for bit on a seeded sample of rows
(plus the first and last rows); products on a seeded sample of outputs plus all
tile-edge rows and columns.  For every sampled output the oracle quantizes the
rows it needs itself, from the same bf16 inputs (the tensor amax spans the whole
tensor), and sums the product in double -- it never reads a GPU result."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import check_products, dev_tensor, host_bytes, sample_pairs

pytestmark = pytest.mark.gpu

W = S.WORKLOADS


def swizzled(plain, rows, blocks):
    """Row-major [rows, blocks] scale bytes -> the swizzled buffer (oracle layout rule)."""
    buf = np.zeros(O.scale_bytes(rows, blocks), dtype=np.uint8)
    for r in range(rows):
        for b in range(blocks):
            buf[O.swz_offset(r, b, blocks)] = plain[r, b]
    return buf


def check_rows_mx(x, fmt, codes_d, scales_d, g_d, rows):
    K = x.shape[1]
    oc, oue, og = O.quantize_mx_rows(x, fmt, rows)
    row_bytes = oc.shape[1]
    gc = host_bytes(codes_d).reshape(-1, row_bytes)
    gs = host_bytes(scales_d)
    assert np.float32(g_d.item()) == np.float32(og)
    assert np.array_equal(gc[rows], oc)
    nb = K // 32
    for i, r in enumerate(rows):
        offs = [O.swz_offset(int(r), b, nb) for b in range(nb)]
        assert np.array_equal(gs[offs], oue[i]), int(r)
    return oc, oue, og


def check_rows_nvfp4(x, codes_d, scales_d, g_d, rows):
    K = x.shape[1]
    oc, osb, og = O.quantize_nvfp4_rows(x, rows)
    gc = codes_d.cpu().numpy().view(np.uint32)
    gs = host_bytes(scales_d)
    assert np.float32(g_d.item()) == np.float32(og)
    assert np.array_equal(gc[rows], oc)
    nb = K // 16
    for i, r in enumerate(rows):
        offs = [O.swz_offset(int(r), b, nb) for b in range(nb)]
        assert np.array_equal(gs[offs], osb[i]), int(r)
    return oc, osb, og


def row_sample(R, n, seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, R - 1, min(127, R - 1), min(128, R - 1)], g.integers(0, R, n)])).astype(np.int64)


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
    arows = np.arange(M, dtype=np.int64)
    oca, oua, oga = check_rows_mx(a, O.E3M2, ca, sa, ga, arows)
    mi, ni = sample_pairs(M, N, 2048, 5)
    wrows = np.unique(ni)
    ocw, ouw, ogw = check_rows_mx(w, O.E3M2, cw, sw, gw, wrows)
    pos = {int(r): i for i, r in enumerate(wrows)}
    want, s = O.gemm_mx(oca, O.E3M2, swizzled(oua, M, K // 32), oga, ocw, O.E3M2,
                        swizzled(ouw, wrows.size, K // 32), ogw, M, wrows.size, K,
                        mi=mi, ni=np.array([pos[int(n)] for n in ni]))
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, "config 2")


@pytest.mark.parametrize("M", [1, 8, 32])
def test_nvfp4_decode_gemv_28672x8192(bsq, M):
    c = W["nvfp4_decode_gemv_Mx28672x8192"]
    N, K = c["N"], c["K"]
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 1)
    cw, sw, gw = bsq.quantize_nvfp4(dev_tensor(w))
    x = S.normal_bf16((M, K), c["x_std"], c["seed"] + 2 + M)
    y = bsq.gemv_nvfp4(dev_tensor(x), cw, sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    mi, ni = sample_pairs(M, N, 1024, 7 + M)
    rows = np.unique(ni)
    ocw, osb, ogw = check_rows_nvfp4(w, cw, sw, gw, rows)
    pos = {int(r): i for i, r in enumerate(rows)}
    want, s = O.gemv_nvfp4(x, ocw, swizzled(osb, rows.size, K // 16), ogw, M, rows.size, K,
                           mi=mi, ni=np.array([pos[int(n)] for n in ni]))
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, f"config 3 M={M}")


def test_nvfp4_prefill_gemm_8192(bsq):
    c = W["nvfp4_prefill_gemm_8192"]
    M, N, K = c["M"], c["N"], c["K"]
    a = S.normal_bf16((M, K), c["a_std"], c["seed"] + 1)
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 2)
    ca, sa, ga = bsq.quantize_nvfp4(dev_tensor(a))
    cw, sw, gw = bsq.quantize_nvfp4(dev_tensor(w))
    y = bsq.gemm_nvfp4(ca, sa, ga, cw, sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    mi, ni = sample_pairs(M, N, 1024, 11)
    ar, wr = np.unique(mi), np.unique(ni)
    oca, osa, oga = check_rows_nvfp4(a, ca, sa, ga, ar)
    ocw, osw, ogw = check_rows_nvfp4(w, cw, sw, gw, wr)
    pa = {int(r): i for i, r in enumerate(ar)}
    pw = {int(r): i for i, r in enumerate(wr)}
    want, s = O.gemm_nvfp4(oca, swizzled(osa, ar.size, K // 16), oga, ocw, swizzled(osw, wr.size, K // 16), ogw,
                           ar.size, wr.size, K, mi=np.array([pa[int(m)] for m in mi]),
                           ni=np.array([pw[int(n)] for n in ni]))
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, "config 4")


def test_w6a8_e4m3xe2m3_4096x14336x4096(bsq):
    c = W["w6a8_e4m3xe2m3_4096x14336x4096"]
    M, N, K = c["M"], c["N"], c["K"]
    a = S.normal_bf16((M, K), c["a_std"], c["seed"] + 1)
    w = S.normal_bf16((N, K), c["w_std"], c["seed"] + 2)
    ca, sa, ga = bsq.quantize_mxfp6(dev_tensor(a), "e4m3")
    cw, sw, gw = bsq.quantize_mxfp6(dev_tensor(w), "e2m3")
    y = bsq.gemm_mxfp6(ca, "e4m3", sa, ga, cw, "e2m3", sw, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    mi, ni = sample_pairs(M, N, 1024, 13)
    ar, wr = np.unique(mi), np.unique(ni)
    oca, oua, oga = check_rows_mx(a, O.E4M3, ca, sa, ga, ar)
    ocw, ouw, ogw = check_rows_mx(w, O.E2M3, cw, sw, gw, wr)
    pa = {int(r): i for i, r in enumerate(ar)}
    pw = {int(r): i for i, r in enumerate(wr)}
    want, s = O.gemm_mx(oca, O.E4M3, swizzled(oua, ar.size, K // 32), oga, ocw, O.E2M3,
                        swizzled(ouw, wr.size, K // 32), ogw, ar.size, wr.size, K,
                        mi=np.array([pa[int(m)] for m in mi]), ni=np.array([pw[int(n)] for n in ni]))
    check_products(y[torch.from_numpy(mi), torch.from_numpy(ni)], want, s, "config 5 GEMM")


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
