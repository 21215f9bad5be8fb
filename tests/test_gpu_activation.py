"""GPU parity of the fused activation + MX quantizer (bsq_quantize_mxfp6_act)
against the oracle (b12x _lib/fp6.py relu2_quantize_grouped_mxfp6_torch,
silu_mul_quantize_grouped_mxfp6_torch): both launch shapes (one cluster for
small tensors, amax pass + encode pass for large ones), every MX format.

ReLU^2: activated values, codes, scales and s_global bit-exact.
SiLU * up: CUDA's expf and the C library's may round differently in the last
place, so activated values are compared within one bf16 ulp; the codes,
scales and s_global must then be bit-exact against the oracle's quantizer run
on the GPU's own activated tensor."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

FMTS = {"e3m2": O.E3M2, "e2m3": O.E2M3, "e4m3": O.E4M3}
SHAPES = [(16, 4096), (3, 96), (300, 1024), (128, 4096)]      # the first two fit one cluster


def run(bsq, x, act, fmt):
    xd = dev_tensor(x).view(torch.bfloat16)
    codes, scales, sg, a = bsq.quantize_mxfp6_act(xd, act, fmt, want_act=True)
    torch.cuda.synchronize()
    return (host_bytes(codes), host_bytes(scales), float(sg.item()),
            a.view(torch.int16).cpu().numpy().view(np.uint16))


def ordinal(bits):
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("fmt", list(FMTS))
def test_relu2_quantize_bit_exact(bsq, M, K, fmt):
    x = S.normal_bf16((M, K), 2.0, 211 + M + K, outlier_frac=0.01)
    codes, scales, sg, a = run(bsq, x, bsq.ACT_RELU2, fmt)
    oc, osc, og, oa = O.quantize_mx_act(x, O.ACT_RELU2, FMTS[fmt])
    assert np.array_equal(a, oa), "activated values"
    assert np.array_equal(codes, oc.view(np.uint8).reshape(codes.shape)), "codes"
    assert np.array_equal(scales, osc), "scales"
    assert sg == og, "s_global"


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("fmt", list(FMTS))
def test_silu_mul_quantize(bsq, M, K, fmt):
    x = S.normal_bf16((M, 2 * K), 2.0, 311 + M + K, outlier_frac=0.01)
    codes, scales, sg, a = run(bsq, x, bsq.ACT_SILU_MUL, fmt)
    oa = O.activate(x, O.ACT_SILU_MUL)
    d = np.abs(ordinal(a) - ordinal(oa))
    assert d.max() <= 1, "activated values beyond one bf16 ulp"
    assert (d == 0).mean() > 0.99
    oc, osc, og = O.quantize_mx(a, FMTS[fmt])                     # the oracle on the GPU's activation
    assert np.array_equal(codes, oc.reshape(codes.shape)), "codes"
    assert np.array_equal(scales, osc), "scales"
    assert sg == og, "s_global"


def test_relu2_of_all_negative_input_is_all_zero(bsq):
    M, K = 200, 512
    x = S.normal_bf16((M, K), 1.0, 5) | np.uint16(0x8000)          # every value <= -0
    codes, scales, sg, a = run(bsq, x, bsq.ACT_RELU2, "e3m2")
    assert not a.any() and not codes.any() and not scales.any() and sg == 0.0


def test_activated_output_is_optional(bsq):
    M, K = 130, 1024
    x = S.normal_bf16((M, 2 * K), 1.0, 7)
    xd = dev_tensor(x).view(torch.bfloat16)
    c1, s1, g1, _ = bsq.quantize_mxfp6_act(xd, bsq.ACT_SILU_MUL, "e2m3", want_act=True)
    c2, s2, g2 = bsq.quantize_mxfp6_act(xd, bsq.ACT_SILU_MUL, "e2m3")
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(s1, s2) and torch.equal(g1, g2)
