"""Pins for the oracle's products: the worked nvfp4 example of the cubecl-tile
page, exact rational brute force on tiny matrices (the test unpacks the codes
itself and sums in Fractions), dequantization, and the tolerance scale S."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.test_oracle_quantize import swizzle_by_permute, pack6, f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_nvfp4_shaped_decode_worked_example():
    """cubecl-tile tests/tile/packed.rs, nvfp4_shaped_decode: every e2m1 code
    cycled, 16-blocks on 8-value words, halves as block scales, g = 1/4; the
    page's reference is exact.  Page orientation c[m,n] = sum_k w[m,k] s g x[k,n];
    here Y[n', m'] with the weight as W (N = rows) and x^T as the activations."""
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_shaped_decode.json")))
    rows, cols, block, blocks, gg = g["rows"], g["cols"], g["block"], g["blocks"], g["g"]
    ladder = [Fraction(v) for v in g["e2m1_magnitudes"]]
    depth = block * blocks
    codes = np.arange(rows * depth) % 16
    words = np.zeros(rows * depth // 8, dtype=np.uint32)
    for i, c in enumerate(codes):
        words[i // 8] |= np.uint32(c) << np.uint32(4 * (i % 8))
    x = np.array([(i % 7) - 3 for i in range(depth * cols)], dtype=np.float32).reshape(depth, cols)
    s = [(i + 1) / 2 for i in range(rows * blocks)]
    s_codes = np.array([O.encode(O.E4M3, v) for v in s], dtype=np.uint8).reshape(rows, blocks)
    scales = swizzle_by_permute(s_codes, rows, blocks)
    xT = S.f32_to_bf16_bits(np.ascontiguousarray(x.T))           # [cols, depth]
    y, _ = O.gemv_nvfp4(xT, words.reshape(rows, depth // 8), scales, gg, cols, rows, depth)
    y = y.reshape(cols, rows)

    def e2m1(c):
        v = ladder[c & 7]
        return -v if c & 8 else v
    for m in range(rows):
        for n in range(cols):
            want = sum(e2m1(int(codes[m * depth + k])) * Fraction(s[m * blocks + k // block])
                       * Fraction(gg) * Fraction(int(x[k, n])) for k in range(depth))
            assert Fraction(y[n, m]) == want, (m, n)


def exact_nvfp4_value(words, sc_plain, r, k):
    c = int((words[r, k // 8] >> np.uint32(4 * (k % 8))) & np.uint32(0xF))
    return Fraction(O.decode(O.E2M1, c)) * Fraction(O.decode(O.E4M3, int(sc_plain[r, k // 16])))


def exact_mx_value(codes, fmt, ue_plain, r, k):
    return Fraction(O.decode(fmt, int(codes[r, k]))) * Fraction(2) ** (int(ue_plain[r, k // 32]) - 127)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_nvfp4_gemm_brute_force(seed):
    M, N, K = 3, 4, 64
    A = S.random_words((M, K // 8), seed)
    W = S.random_words((N, K // 8), seed + 100)
    sa = S.choice_bytes(M * K // 16, seed + 1, range(1, 0x7F)).reshape(M, K // 16)
    sw = S.choice_bytes(N * K // 16, seed + 2, range(1, 0x7F)).reshape(N, K // 16)
    gA, gW = 0.375, 1.5
    y, s = O.gemm_nvfp4(A, swizzle_by_permute(sa, M, K // 16), gA, W, swizzle_by_permute(sw, N, K // 16),
                        gW, M, N, K)
    y, s = y.reshape(M, N), s.reshape(M, N)
    for m in range(M):
        for n in range(N):
            terms = [exact_nvfp4_value(A, sa, m, k) * exact_nvfp4_value(W, sw, n, k) for k in range(K)]
            exact = sum(terms) * Fraction(gA) * Fraction(gW)
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -50 * s[m, n] + Fraction(0)
            assert abs(Fraction(s[m, n]) - sum(abs(t) for t in terms) * Fraction(gA * gW)) \
                <= Fraction(2) ** -50 * s[m, n]


@pytest.mark.parametrize("fa,fw", [(O.E3M2, O.E3M2), (O.E4M3, O.E2M3), (O.E2M3, O.E3M2)])
def test_mx_gemm_brute_force(fa, fw):
    M, N, K = 2, 3, 64
    rng = np.random.default_rng(fa * 10 + fw)

    def operand(R, fmt):
        codes = rng.integers(0, 256 if fmt == O.E4M3 else 64, size=(R, K)).astype(np.uint8)
        if fmt == O.E4M3:
            codes[(codes & 0x7F) == 0x7F] = 0            # no NaN codes
            packed = codes
        else:
            packed = pack6(codes).reshape(R, 3 * K // 4)
        ue = rng.integers(110, 140, size=(R, K // 32)).astype(np.uint8)
        return codes, packed, ue, swizzle_by_permute(ue, R, K // 32)
    ca, pa, ua, sa = operand(M, fa)
    cw, pw, uw, sw = operand(N, fw)
    y, s = O.gemm_mx(pa, fa, sa, 0.5, pw, fw, sw, 2.0, M, N, K)
    y = y.reshape(M, N)
    for m in range(M):
        for n in range(N):
            exact = sum(exact_mx_value(ca, fa, ua, m, k) * exact_mx_value(cw, fw, uw, n, k) for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -50 * Fraction(s[m * N + n])


@pytest.mark.parametrize("fw", [O.E3M2, O.E2M3, "nvfp4"])
def test_gemv_brute_force_bf16_activations(fw):
    M, N, K = 2, 3, 64
    x = S.normal_bf16((M, K), 1.0, 77)
    xf = f32(x)
    rng = np.random.default_rng(5)
    if fw == "nvfp4":
        W = S.random_words((N, K // 8), 6)
        sc = S.choice_bytes(N * K // 16, 7, range(1, 0x7F)).reshape(N, K // 16)
        y, _ = O.gemv_nvfp4(x, W, swizzle_by_permute(sc, N, K // 16), 0.25, M, N, K)
        val = lambda n, k: exact_nvfp4_value(W, sc, n, k) * Fraction(0.25)
    else:
        codes = rng.integers(0, 64, size=(N, K)).astype(np.uint8)
        ue = rng.integers(115, 135, size=(N, K // 32)).astype(np.uint8)
        y, _ = O.gemv_mx(x, pack6(codes).reshape(N, 3 * K // 4), fw, swizzle_by_permute(ue, N, K // 32),
                         0.25, M, N, K)
        val = lambda n, k: exact_mx_value(codes, fw, ue, n, k) * Fraction(0.25)
    y = y.reshape(M, N)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(xf[m, k])) * val(n, k) for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(2) ** -45 * (abs(exact) + 1)


def test_dequant_is_code_times_scale_times_g():
    R, K = 3, 64
    W = S.random_words((R, K // 8), 9)
    sc = S.choice_bytes(R * K // 16, 10, range(1, 0x7F)).reshape(R, K // 16)
    d = O.dequant_nvfp4(W, swizzle_by_permute(sc, R, K // 16), 0.5, R, K)
    for r in range(R):
        for k in range(K):
            assert Fraction(d[r, k]) == exact_nvfp4_value(W, sc, r, k) * Fraction(0.5)


def test_quantize_then_dequantize_round_trip_error():
    """The dequant of a quantized tensor stays within half a code step of x
    (relative to each block's scale): the two halves agree on the factor."""
    xb = S.normal_bf16((8, 128), 0.02, 3)
    x = f32(xb).astype(np.float64)
    for fmt, step in ((O.E3M2, 2.0 ** -2), (O.E2M3, 2.0 ** -3), (O.E4M3, 2.0 ** -3)):
        codes, scales, g = O.quantize_mx(xb, fmt)
        d = O.dequant_mx(codes, fmt, scales, g, 8, 128)
        for r in range(8):
            for b in range(4):
                blk = slice(b * 32, b * 32 + 32)
                amax_b = np.abs(x[r, blk]).max()
                # half a relative step of the block max bounds every element's error
                assert np.abs(d[r, blk] - x[r, blk]).max() <= amax_b * step * 1.01 + 1e-30
    w, sc, g = O.quantize_nvfp4(xb)
    d = O.dequant_nvfp4(w, sc, g, 8, 128)
    assert np.abs(d - x).max() <= np.abs(x).max() * 0.26
