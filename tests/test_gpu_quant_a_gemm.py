"""GPU parity of the GEMM with the activation quantizer fused into it
(b12x fp6.py, the _containers quantize-then-MMA variants): bf16 activations are
MX-quantized inside the GEMM, straight into the tensor cores' shared-memory
operand layout.

Pinned two ways: bit for bit against bsq_quantize_mxfp6 followed by
bsq_gemm_mxfp6 (same codes, scales, global factor and MMA order, so the same
Y and the same s_global), and against the oracle's quantizer and product
(fp32 outputs within 1e-5 * sum|a*w|, bf16 within one ulp)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import check_products, dev_tensor

pytestmark = pytest.mark.gpu

FMT = {"e3m2": O.E3M2, "e2m3": O.E2M3, "e4m3": O.E4M3}


def weight(N, K, fw, seed):
    w = S.normal_bf16((N, K), 0.02, seed, outlier_frac=0.01)
    return O.quantize_mx(w, FMT[fw])


def two_step(bsq, x, fa, W, fw, sW, gW, K, out):
    codes, scales, g = bsq.quantize_mxfp6(dev_tensor(x), fa)
    y = bsq.gemm_mxfp6(codes, fa, scales, g, W, fw, sW, gW, K, out_dtype=out)
    return y, g


# (M, N, K): split-K 4 (the W6A6 shape), split-K 8 with a ragged row block,
# one activation row, and a persistent-size grid (one tile per CTA here)
SHAPES = [(128, 4096, 4096), (200, 1000, 1024), (1, 300, 256), (1100, 2048, 256)]


@pytest.mark.parametrize("fa,fw", [("e3m2", "e3m2"), ("e4m3", "e2m3"), ("e2m3", "e4m3"), ("e2m3", "e2m3")])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_equals_quantize_then_gemm(bsq, fa, fw, M, N, K):
    x = S.normal_bf16((M, K), 0.5, 901 + M, outlier_frac=0.01, outlier_mult=20.0)
    Wc, sWc, gWc = weight(N, K, fw, 903 + N)
    W, sW = dev_tensor(Wc), dev_tensor(sWc)
    gW = torch.tensor([gWc], device="cuda")
    for out in (torch.bfloat16, torch.float32):
        y2, g2 = two_step(bsq, x, fa, W, fw, sW, gW, K, out)
        y1, g1 = bsq.gemm_mxfp6_quant_a(dev_tensor(x), fa, W, fw, sW, gW, K, out_dtype=out)
        torch.cuda.synchronize()
        assert torch.equal(g1, g2), (g1.item(), g2.item())
        assert torch.equal(y1.view(torch.int16) if out == torch.bfloat16 else y1.view(torch.int32),
                           y2.view(torch.int16) if out == torch.bfloat16 else y2.view(torch.int32)), \
            f"{fa}x{fw} {M}x{N}x{K} {out}: fused and two-step products differ"


@pytest.mark.parametrize("fa,fw", [("e3m2", "e2m3"), ("e4m3", "e3m2"), ("e2m3", "e2m3")])
def test_fused_matches_oracle(bsq, fa, fw):
    M, N, K = 77, 384, 640
    x = S.normal_bf16((M, K), 1.0, 911, outlier_frac=0.01, outlier_mult=20.0)
    Wc, sWc, gWc = weight(N, K, fw, 913)
    y, g = bsq.gemm_mxfp6_quant_a(dev_tensor(x), fa, dev_tensor(Wc), fw, dev_tensor(sWc),
                                  torch.tensor([gWc], device="cuda"), K, out_dtype=torch.float32)
    torch.cuda.synchronize()
    Ac, sAc, gAc = O.quantize_mx(x, FMT[fa])
    assert np.float32(g.item()) == np.float32(gAc)
    want, s = O.gemm_mx(Ac, FMT[fa], sAc, gAc, Wc, FMT[fw], sWc, gWc, M, N, K)
    check_products(y, want, s, f"fused {fa}x{fw}")


def test_fused_all_zero_activations(bsq):
    """amax = 0: gs = 0, every code and scale 0, s_global 0, Y exactly 0."""
    M, N, K = 64, 256, 512
    x = np.zeros((M, K), dtype=np.uint16)
    Wc, sWc, gWc = weight(N, K, "e3m2", 921)
    y, g = bsq.gemm_mxfp6_quant_a(dev_tensor(x), "e3m2", dev_tensor(Wc), "e3m2", dev_tensor(sWc),
                                  torch.tensor([gWc], device="cuda"), K, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert g.item() == 0.0
    assert torch.count_nonzero(y).item() == 0
