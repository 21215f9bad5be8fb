"""Pins for the oracle's quantizers (MX per 32 with UE8M0, nvfp4 per 16 with ue4m3).

The MX quantizer is checked against an independent numpy restatement of the
b12x _lib/fp6.py recipe (quantize_grouped_mxfp6_torch with the exact ceil of
fp6_block_ue8m0_exact computed in rational arithmetic, the test's own
bit-level encoder and packer, and the page's permute form of the scale
layout), and against invariants that hold for any correct quantizer:
containment under the ceil rule, the per-element error bound, power-of-two
equivariance and zero blocks.  The rival readings the pages leave open are
shown to be observable on the fixtures (each gives different bytes).

The nvfp4 recipe is a reading (the pages give none); it is pinned by the
same independent restatement of that reading and by invariants only.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.test_oracle_formats import LAYOUT, BITS, magnitudes, rne_encode

FMAX = {O.E3M2: 28.0, O.E2M3: 7.5, O.E4M3: 448.0, O.E2M1: 6.0}


def f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def exact_ceil_log2(r):
    """Smallest e with 2^e >= r, in exact rationals (r > 0 finite)."""
    fr = Fraction(float(r))
    e = math.frexp(float(r))[1] - 1
    while Fraction(2) ** e < fr:
        e += 1
    while Fraction(2) ** (e - 1) >= fr:
        e -= 1
    return e


def swizzle_by_permute(plain, rows, blocks):
    """Place row-major [rows, blocks] scale bytes into the swizzled buffer using the
    forward permute that unswizzle_mxfp6_scales (b12x _lib/fp6.py) inverts."""
    rp, cp = -(-rows // 128) * 128, -(-blocks // 4) * 4
    full = np.zeros((rp, cp), dtype=np.uint8)
    full[:rows, :blocks] = plain
    # orig = sw.reshape(rp/128, cp/4, 32, 4, 4).permute(0, 3, 2, 1, 4) => sw = orig viewed
    # as (rp/128, 4, 32, cp/4, 4) permuted by the same (0, 3, 2, 1, 4).
    return full.reshape(rp // 128, 4, 32, cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1).copy()


def pack6(codes):
    c = np.asarray(codes, dtype=np.uint32).reshape(-1, 4)
    bits = c[:, 0] | (c[:, 1] << 6) | (c[:, 2] << 12) | (c[:, 3] << 18)
    return np.stack([bits & 0xFF, (bits >> 8) & 0xFF, (bits >> 16) & 0xFF], 1).astype(np.uint8).reshape(-1)


def ref_quantize_mx(xb, fmt):
    x = f32(xb)
    M, K = x.shape
    fmax = np.float32(FMAX[fmt])
    amax = np.max(np.abs(x)) if x.size else np.float32(0)
    gs = np.float32(np.float32(448.0) * fmax) / amax if amax > 0 else np.float32(0)
    codes = np.zeros((M, K), dtype=np.uint8)
    ue = np.zeros((M, K // 32), dtype=np.uint8)
    for r in range(M):
        for b in range(K // 32):
            blk = x[r, b * 32:(b + 1) * 32]
            if gs == 0:
                continue
            amax_b = np.max(np.abs(blk))
            t = np.float32(amax_b * gs)
            ratio = np.float32(t / fmax)
            u = 0 if ratio <= 0 else min(max(exact_ceil_log2(ratio) + 127, 0), 255)
            ue[r, b] = u
            if u == 0:
                continue
            inv = np.float32(gs * np.float32(2.0 ** (127 - u)))
            if inv == 0:
                continue
            q = (blk * inv).astype(np.float32)
            codes[r, b * 32:(b + 1) * 32] = [rne_encode(fmt, v) for v in q]
    packed = codes if fmt == O.E4M3 else pack6(codes).reshape(M, 3 * K // 4)
    sg = np.float32(np.float32(1.0) / gs) if gs != 0 else np.float32(0)
    return packed, swizzle_by_permute(ue, M, K // 32), float(sg), ue, codes


def ref_quantize_nvfp4(xb):
    x = f32(xb)
    M, K = x.shape
    amax = np.max(np.abs(x)) if x.size else np.float32(0)
    gs = np.float32(2688.0) / amax if amax > 0 else np.float32(0)
    codes = np.zeros((M, K), dtype=np.uint8)
    sb = np.zeros((M, K // 16), dtype=np.uint8)
    for r in range(M):
        for b in range(K // 16):
            blk = x[r, b * 16:(b + 1) * 16]
            if gs == 0:
                continue
            t = np.float32(np.max(np.abs(blk)) * gs)
            ratio = np.float32(t / np.float32(6.0))
            s = rne_encode(O.E4M3, ratio)
            sb[r, b] = s
            if s == 0:
                continue
            inv = np.float32(gs / np.float32(O.decode(O.E4M3, s)))
            q = (blk * inv).astype(np.float32)
            codes[r, b * 16:(b + 1) * 16] = [rne_encode(O.E2M1, v) for v in q]
    c = codes.astype(np.uint32).reshape(M, K // 8, 8)
    words = np.zeros((M, K // 8), dtype=np.uint32)
    for j in range(8):
        words |= c[:, :, j] << (4 * j)
    sg = np.float32(np.float32(1.0) / gs) if gs != 0 else np.float32(0)
    return words, swizzle_by_permute(sb, M, K // 16), float(sg), sb, codes


def fixture(M, K, seed, std=1.0, outliers=0.01):
    xb = S.normal_bf16((M, K), std, seed, outlier_frac=outliers)
    if M * K >= 64:
        xb[0, :32] = 0                      # an all-zero block
        xb.ravel()[40] = 0x8000             # a negative zero
        xb.ravel()[41] = 0x8001             # a tiny negative (bf16 subnormal)
    return xb


CASES = [(1, 32, 1), (3, 64, 2), (5, 96, 3), (130, 64, 4), (7, 256, 5)]


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3])
@pytest.mark.parametrize("M,K,seed", CASES)
def test_mx_quantizer_matches_independent_restatement(fmt, M, K, seed):
    xb = fixture(M, K, seed)
    codes, scales, sg = O.quantize_mx(xb, fmt)
    rc, rs, rsg, _, _ = ref_quantize_mx(xb, fmt)
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales, rs)
    assert np.float32(sg) == np.float32(rsg)


@pytest.mark.parametrize("M,K,seed", CASES)
def test_nvfp4_quantizer_matches_restated_reading(M, K, seed):
    xb = fixture(M, K, seed)
    codes, scales, sg = O.quantize_nvfp4(xb)
    rc, rs, rsg, _, _ = ref_quantize_nvfp4(xb)
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales, rs)
    assert np.float32(sg) == np.float32(rsg)


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3])
def test_mx_row_subset_equals_full(fmt):
    xb = fixture(131, 128, 21)
    codes, scales, sg = O.quantize_mx(xb, fmt)
    rows = np.array([0, 5, 127, 128, 130])
    c2, ue2, sg2 = O.quantize_mx_rows(xb, fmt, rows)
    assert sg2 == sg and np.array_equal(c2, codes[rows])
    for i, r in enumerate(rows):
        for b in range(4):
            assert ue2[i, b] == scales[O.swz_offset(int(r), b, 4)]
    w, sw, g = O.quantize_nvfp4(xb)
    w2, sb2, g2 = O.quantize_nvfp4_rows(xb, rows)
    assert g2 == g and np.array_equal(w2, w[rows])
    for i, r in enumerate(rows):
        for b in range(8):
            assert sb2[i, b] == sw[O.swz_offset(int(r), b, 8)]


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3])
def test_mx_containment_and_error_bound(fmt):
    """Under the ceil rule no element needs more than the format's maximum (up to
    the two f32 roundings of the ratio), and every code is the nearest value."""
    xb = fixture(64, 256, 31)
    codes, scales, sg = O.quantize_mx(xb, fmt)
    _, _, _, ue, plain = ref_quantize_mx(xb, fmt)
    x = f32(xb).astype(np.float64)
    gs = 1.0 / sg
    mags = magnitudes(fmt)
    for r in range(64):
        for b in range(8):
            u = int(ue[r, b])
            if u == 0:
                continue
            inv = np.float32(np.float32(gs) * np.float32(2.0 ** (127 - u)))
            for i in range(32):
                v = float(np.float32(np.float32(x[r, b * 32 + i]) * inv))
                assert abs(v) <= FMAX[fmt] * (1 + 2 ** -21)
                got = O.decode(fmt, int(plain[r, b * 32 + i]))
                # nearest: no representable magnitude is strictly closer
                assert min(abs(abs(v) - m) for m in mags) == abs(abs(v) - abs(got))


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3, "nvfp4"])
def test_power_of_two_equivariance(fmt):
    xb = S.normal_bf16((16, 128), 1.0, 41)
    x = f32(xb)
    for j in (-3, 5):
        y = S.f32_to_bf16_bits(x * np.float32(2.0 ** j))
        if fmt == "nvfp4":
            a, b = O.quantize_nvfp4(xb), O.quantize_nvfp4(y)
        else:
            a, b = O.quantize_mx(xb, fmt), O.quantize_mx(y, fmt)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        assert b[2] == a[2] * 2.0 ** j


def test_zero_tensor_and_zero_blocks():
    z = np.zeros((3, 64), dtype=np.uint16)
    for fmt in (O.E3M2, O.E2M3, O.E4M3):
        c, s, g = O.quantize_mx(z, fmt)
        assert not c.any() and not s.any() and g == 0.0
    c, s, g = O.quantize_nvfp4(z)
    assert not c.any() and not s.any() and g == 0.0


# ------------------------------------------------------------- rival readings --
def test_rival_readings_are_observable():
    """Each reading the pages leave open, replaced by its rival, changes the
    fixture's output (so the tests above can tell them apart)."""
    xb = fixture(32, 256, 51)
    fmt = O.E3M2
    codes, scales, sg = O.quantize_mx(xb, fmt)
    _, _, _, ue, plain = ref_quantize_mx(xb, fmt)
    x = f32(xb)
    gs = np.float32(1.0) / np.float32(sg)
    # floor instead of ceil for the UE8M0 exponent
    floor_ue = np.zeros_like(ue)
    for r in range(32):
        for b in range(8):
            amax_b = np.max(np.abs(x[r, b * 32:(b + 1) * 32]))
            ratio = np.float32(np.float32(amax_b * gs) / np.float32(28.0))
            floor_ue[r, b] = 0 if ratio <= 0 else math.floor(math.log2(float(ratio))) + 127
    assert not np.array_equal(floor_ue, ue)
    # dequant multiplying by gs instead of dividing
    d_right = O.dequant_mx(codes, fmt, scales, sg, 32, 256)
    d_rival = O.dequant_mx(codes, fmt, scales, float(gs), 32, 256)
    assert np.abs(d_right - f32(xb)).max() < np.abs(d_rival - f32(xb)).max()
    # double rounding (f32 -> bf16 -> fp6) instead of a single rounding
    diffs = 0
    for r in range(32):
        for b in range(8):
            u = int(ue[r, b])
            if u == 0:
                continue
            inv = np.float32(gs * np.float32(2.0 ** (127 - u)))
            q = (x[r, b * 32:(b + 1) * 32] * inv).astype(np.float32)
            qb = f32(S.f32_to_bf16_bits(q))
            diffs += sum(rne_encode(fmt, a) != rne_encode(fmt, c) for a, c in zip(q, qb))
    assert diffs > 0
    # row-major scales instead of swizzled
    assert not np.array_equal(scales[:ue.size], ue.reshape(-1))
    # nvfp4 nibbles high field first instead of low field first
    w, _, _ = O.quantize_nvfp4(xb)
    w_hi = np.zeros_like(w)
    for j in range(8):
        w_hi |= ((w >> (4 * j)) & 0xF) << (4 * (7 - j))
    assert not np.array_equal(w, w_hi)


def test_ties_to_lower_rival_is_observable():
    """A value exactly between two codes whose lower neighbour is odd."""
    mags = magnitudes(O.E3M2)
    a, b = mags[1], mags[2]                     # codes 1 (odd) and 2 (even)
    assert O.encode(O.E3M2, (a + b) / 2) == 2   # ties to even, not to the lower code


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3])
def test_byte_container_output_is_the_unpacked_codes(fmt):
    """b12x fp6.py quantize_block_fp6_*_bytes: identical quantization, one code
    per byte (bits [5:0]) in K order instead of the 4-in-3 packing."""
    x = S.normal_bf16((48, 320), 0.02, 77, outlier_frac=0.01)
    c, s, g = O.quantize_mx_containers(x, fmt)
    p, s2, g2 = O.quantize_mx(x, fmt)
    assert c.shape == (48, 320)
    assert not (c & 0xC0).any()
    assert np.array_equal(c.ravel(), O.unpack_fp6(p, 48 * 320))
    assert np.array_equal(s, s2) and g == g2
