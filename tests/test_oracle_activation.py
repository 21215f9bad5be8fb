"""CPU pins for the oracle's fused activation + MX quantizer (b12x _lib/fp6.py,
relu2_quantize_grouped_mxfp6_torch and silu_mul_quantize_grouped_mxfp6_torch):
the activation in f32 rounded to bf16, then the MX quantizer.

Independent references: float64 math for the activations and torch's own
f32 -> bf16 cast for the rounding; the SiLU minimum from its closed form."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S


def torch_bf16_bits(v64: np.ndarray) -> np.ndarray:
    """float64 -> f32 (numpy) -> bf16 by torch's round-to-nearest-even cast."""
    t = torch.from_numpy(np.asarray(v64, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def test_relu2_is_the_exact_square_rounded_to_bf16():
    x = S.normal_bf16((64, 256), 3.0, 101)
    x[0, :4] = [0x8000, 0x0000, 0xFF80 & 0xC000, 0x0001]       # -0, +0, -2, a subnormal
    got = O.activate(x, O.ACT_RELU2)
    v = bf16_values(x)
    want = torch_bf16_bits(np.maximum(v, 0.0) ** 2)               # the square is exact in f32
    assert np.array_equal(got, want)
    assert not (got & 0x8000).any(), "ReLU^2 is never negative"


def test_silu_mul_matches_float64_within_one_bf16_ulp():
    M, K = 32, 512
    g = S.normal_bf16((M, K), 2.0, 102)
    u = S.normal_bf16((M, K), 1.0, 103)
    got = O.activate(np.concatenate([g, u], axis=1), O.ACT_SILU_MUL)
    gv, uv = bf16_values(g), bf16_values(u)
    ref = gv / (1.0 + np.exp(-gv)) * uv
    want = torch_bf16_bits(ref)
    d = np.abs(ordinal(got) - ordinal(want))
    assert d.max() <= 1
    assert (d == 0).mean() > 0.99                                  # differs only next to a rounding tie


def test_silu_special_values_and_its_minimum():
    # up = 1 isolates SiLU: silu(0) = 0, silu(g) -> g for large g, -> -0 for very negative g, and its
    # global minimum is -0.27846454276107... at g = -1.27846454276107... (x = -1 - W(1/e))
    gs = np.linspace(-1.6, -1.0, 1024)
    g = torch_bf16_bits(np.concatenate([[0.0, 60.0, -200.0], gs]))[None, :]
    g = np.ascontiguousarray(np.pad(g, ((0, 0), (0, (-g.shape[1]) % 32))))
    u = np.full_like(g, 0x3F80)                                     # 1.0
    a = bf16_values(O.activate(np.concatenate([g, u], axis=1), O.ACT_SILU_MUL))[0]
    assert a[0] == 0.0 and a[1] == 60.0 and a[2] == 0.0
    assert abs(a[3:].min() - (-0.27846454276107)) <= 2.0 ** -9    # one bf16 ulp at 0.28


@pytest.mark.parametrize("act", [O.ACT_RELU2, O.ACT_SILU_MUL])
@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3])
def test_fused_quantizer_is_quantize_of_the_activation(act, fmt):
    M, K = 40, 192
    x = S.normal_bf16((M, K * (2 if act == O.ACT_SILU_MUL else 1)), 1.5, 104 + act, outlier_frac=0.01)
    codes, scales, g, a = O.quantize_mx_act(x, act, fmt)
    assert np.array_equal(a, O.activate(x, act))
    c2, s2, g2 = O.quantize_mx(a, fmt)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2) and g == g2
    if act == O.ACT_RELU2:                                          # non-negative input: no sign bits
        sign = 0x80 if fmt == O.E4M3 else None
        if sign is not None:
            assert not (codes & sign).any()
        else:
            assert not (O.unpack_fp6(codes, M * K) & 0x20).any()
