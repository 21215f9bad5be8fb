"""GPU parity of the grouped (MoE) path against the oracle (b12x _lib/fp6.py
quantize_grouped_mxfp6_torch and its grouped layouts): the grouped MX quantizer
(per-group global scales and row counts; bit-exact codes, scales, s_global) and
the grouped tcgen05 GEMM over experts (fp32 outputs within 1e-5 * sum|a*w|;
rows past a group's count untouched)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import check_products, dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

FMTS = {"e3m2": O.E3M2, "e2m3": O.E2M3, "e4m3": O.E4M3}
FMAX = {"e3m2": 28.0, "e2m3": 7.5, "e4m3": 448.0}


def groups(G, R, C, seed, std=0.5):
    return S.normal_bf16((G * R, C), std, seed, outlier_frac=0.01).reshape(G, R, C)


def group_gs(x, rc, fmt):
    out = []
    for g, n in enumerate(rc):
        v = np.abs((x[g, :max(n, 1)].astype(np.uint32) << 16).view(np.float32)).max()
        out.append(np.float32(448.0 * FMAX[fmt]) / np.float32(v) if v > 0 else np.float32(1.0))
    return np.array(out, dtype=np.float32)


def gpu_quantize(bsq, x, rc, gs, fmt):
    G, R, C = x.shape
    rb = C if fmt == "e4m3" else 3 * C // 4
    codes = torch.empty((G, R, rb), dtype=torch.uint8, device="cuda")
    scales = torch.empty((G, bsq.scale_bytes(R, C // 32)), dtype=torch.uint8, device="cuda")
    sg = torch.empty(G, dtype=torch.float32, device="cuda")
    bsq.quantize_grouped_mxfp6_(dev_tensor(x).view(torch.bfloat16), torch.tensor(rc, dtype=torch.int32, device="cuda"),
                                torch.from_numpy(gs).cuda(), {"e3m2": 0, "e2m3": 1, "e4m3": 2}[fmt], codes, scales, sg)
    return codes, scales, sg


@pytest.mark.parametrize("fmt", list(FMTS))
def test_grouped_quantize_bit_exact(bsq, fmt):
    G, R, C = 4, 200, 256
    x = groups(G, R, C, 601)
    rc = [200, 0, 37, 129]
    gs = group_gs(x, rc, fmt) * np.float32(0.75)            # not a power of two away from the amax recipe
    codes, scales, sg = gpu_quantize(bsq, x, rc, gs, fmt)
    torch.cuda.synchronize()
    oc, osc, og = O.quantize_grouped_mx(x, rc, gs, FMTS[fmt])
    assert np.array_equal(host_bytes(codes), oc)
    assert np.array_equal(host_bytes(scales), osc)
    assert np.array_equal(sg.cpu().numpy(), og)


def run_grouped_gemm(bsq, G, R, N, K, rc, fa, fw, out, seed):
    x = groups(G, R, K, seed)
    w = groups(G, N, K, seed + 1, std=0.02)
    gsa, gsw = group_gs(x, rc, fa), group_gs(w, [N] * G, fw)
    A, sA, gA = gpu_quantize(bsq, x, rc, gsa, fa)
    W, sW, gW = gpu_quantize(bsq, w, [N] * G, gsw, fw)
    Y = torch.full((G, R, N), float("nan"), dtype=out, device="cuda")
    bsq.gemm_grouped_mxfp6_(A, {"e3m2": 0, "e2m3": 1, "e4m3": 2}[fa], sA, gA, W, {"e3m2": 0, "e2m3": 1, "e4m3": 2}[fw],
                            sW, gW, torch.tensor(rc, dtype=torch.int32, device="cuda"), Y, G, R, N, K)
    torch.cuda.synchronize()
    oA, osA, ogA = O.quantize_grouped_mx(x, rc, gsa, FMTS[fa])
    oW, osW, ogW = O.quantize_grouped_mx(w, [N] * G, gsw, FMTS[fw])
    assert np.array_equal(host_bytes(A), oA) and np.array_equal(host_bytes(W), oW)
    return Y, (oA, osA, ogA, oW, osW, ogW)


@pytest.mark.parametrize("fa,fw", [("e3m2", "e2m3"), ("e4m3", "e3m2"), ("e2m3", "e2m3")])
def test_grouped_gemm_matches_oracle(bsq, fa, fw):
    G, R, N, K = 3, 200, 320, 256
    rc = [200, 1, 131]
    Y, (oA, osA, ogA, oW, osW, ogW) = run_grouped_gemm(bsq, G, R, N, K, rc, fa, fw, torch.float32, 611)
    want, s = O.gemm_grouped_mx(oA, FMTS[fa], osA, ogA, oW, FMTS[fw], osW, ogW, rc, K)
    for g in range(G):
        check_products(Y[g, :rc[g]], want[g, :rc[g]], s[g, :rc[g]], f"grouped gemm group {g}")
        assert torch.isnan(Y[g, rc[g]:]).all(), f"group {g}: rows past the count were written"


def test_grouped_gemm_256_wide_tiles_sampled(bsq):
    """More 256-wide tiles than SMs, random row counts (some zero), bf16 out,
    checked on a seeded sample of each group's valid outputs."""
    G, R, N, K = 8, 512, 2048, 512
    rc = [512, 0, 77, 300, 129, 1, 511, 256]
    Y, (oA, osA, ogA, oW, osW, ogW) = run_grouped_gemm(bsq, G, R, N, K, rc, "e3m2", "e3m2", torch.bfloat16, 621)
    rng = np.random.default_rng(5)
    for g in range(G):
        if rc[g] == 0:
            assert torch.isnan(Y[g].float()).all()
            continue
        mi = rng.integers(0, rc[g], 256)
        ni = rng.integers(0, N, 256)
        want, s = O.gemm_mx(np.ascontiguousarray(oA[g, :rc[g]]), O.E3M2, np.ascontiguousarray(osA[g]), float(ogA[g]),
                            np.ascontiguousarray(oW[g]), O.E3M2, np.ascontiguousarray(osW[g]), float(ogW[g]),
                            rc[g], N, K, mi=mi, ni=ni)
        check_products(Y[g][torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()], want, s, f"group {g}")
        assert torch.isnan(Y[g, rc[g]:].float()).all()


def test_grouped_gemm_with_no_rows_writes_nothing(bsq):
    G, R, N, K = 2, 64, 128, 128
    Y, _ = run_grouped_gemm(bsq, G, R, N, K, [0, 0], "e2m3", "e2m3", torch.float32, 631)
    assert torch.isnan(Y).all()
