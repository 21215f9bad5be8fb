"""Step-by-step pins of the oracle's nvfp4 quantizer.

The pages give no nvfp4 quantization recipe (cubecl-tile tests/tile/packed.rs,
nvfp4_shaped_decode, only decodes), so the recipe itself is a reading: the MX
recipe of b12x _lib/fp6.py (quantize_grouped_mxfp6_torch) carried over with
e2m1's maximum 6 and a round-to-nearest ue4m3 block scale:

    gs   = fl(2688 / amax)                     (2688 = 448 * 6)
    s_b  = e4m3_rn(fl(fl(amax_b * gs) / 6))
    inv  = fl(gs / s_b)                        (0 when s_b == 0)
    code = e2m1 nearest to fl(x * inv), ties to even, saturating at 6.

The choice of recipe stays "parity unpinned" by the pages.  What these tests
pin is that the oracle carries out each step of that reading correctly, every
step against something that is not the oracle's own code:

  * the global factor against IEEE f32 division done by numpy;
  * every stored ue4m3 byte against torch's float8_e4m3fn cast (a separate
    library's round-to-nearest-even of the same f32 ratio);
  * every e2m1 code against the nearest grid value to fl(x * inv), decided in
    exact rational arithmetic, with ties to the even code and saturation;
  * every dequantized element against a per-element bound of half an e2m1 step
    times s_b / gs (plus the f32 roundings of inv and x * inv).

The fixtures hold exact ties (blocks whose scale makes inv a power of two),
saturating blocks (s_b rounded down, so the block maximum lands above 6),
e4m3-subnormal block scales, block scales that round to zero, all-zero blocks,
negative zeros, and seeded normal data with outliers.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S

E2M1_GRID = [Fraction(v) for v in ("0", "1/2", "1", "3/2", "2", "3", "4", "6")]


def f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def bf16(vals):
    return S.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def scale_index(rows, blocks):
    """pos[r, b] = offset of (r, b) in the swizzled buffer, built from the page's
    permute (b12x _lib/fp6.py, unswizzle_mxfp6_scales inverts
    reshape(rp/128, cp/4, 32, 4, 4).permute(0, 3, 2, 1, 4))."""
    rp, cp = -(-rows // 128) * 128, -(-blocks // 4) * 4
    order = np.arange(rp * cp).reshape(rp // 128, 4, 32, cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    pos = np.empty(rp * cp, dtype=np.int64)
    pos[order] = np.arange(rp * cp)
    return pos.reshape(rp, cp)[:rows, :blocks]


def unpack_words(words):
    """[M, K/8] u32 -> [M, K] e2m1 codes, element k in bits 4(k%8) of word k/8."""
    w = np.asarray(words, dtype=np.uint32)
    return np.stack([(w >> (4 * j)) & 0xF for j in range(8)], axis=-1).reshape(w.shape[0], -1).astype(np.uint8)


def e2m1_value(code):
    mag = E2M1_GRID[code & 7]
    return -mag if code & 8 else mag


def torch_e4m3(ratio: np.float32) -> int:
    """torch's own f32 -> float8_e4m3fn cast (round to nearest even), as a byte."""
    assert ratio < 464.0        # below torch's NaN threshold; the recipe's ratio is <= 448 (1 + 2^-22)
    return int(torch.tensor([float(ratio)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def nearest_e2m1_code(v: np.float32) -> int:
    """The e2m1 code nearest to v in exact rationals: ties to the even code
    (mantissa bit 0), magnitudes above 6 saturate to 6, the sign kept (a negative
    value, -0 included, takes the sign bit)."""
    a = abs(Fraction(float(v)))
    if a >= 6:
        mag_code = 7
    else:
        best = None
        for c, g in enumerate(E2M1_GRID):
            d = abs(a - g)
            if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
                best = (d, c)
        mag_code = best[1]
    neg = np.signbit(v)
    return mag_code | (8 if neg else 0)


def half_step(v_abs: float) -> Fraction:
    """Half the e2m1 grid step of the binade holding |v| (saturated values use the top one)."""
    if v_abs < 2:
        return Fraction(1, 4)
    if v_abs < 4:
        return Fraction(1, 2)
    return Fraction(1)


# ------------------------------------------------------------------ fixtures --
def fixture_structured():
    """Row 0 carries hand-placed blocks; rows 1..7 seeded normals of several
    magnitudes.  amax = 2688 exactly, so gs = 1 and a block's inv is 1 / s_b."""
    K = 16 * 11
    rows = [np.zeros(K, dtype=np.float32) for _ in range(8)]
    r0 = rows[0]
    r0[0:16] = [2688.0] + [0.0] * 15                                   # the tensor maximum: s_b = 448
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    r0[16:32] = [6.0] + mids + [-m for m in mids] + [-6.0]             # s_b = 1, inv = 1: exact ties
    r0[32:48] = [12.0] + [2 * m for m in mids] + [-2 * m for m in mids] + [-0.0]   # s_b = 2, inv = 1/2
    r0[48:64] = [6.3125, 6.0, 5.5, -6.25] + [0.3 * i for i in range(12)]   # ratio 1.052 -> s_b = 1: saturates
    r0[64:80] = np.linspace(-0.01, 0.01, 16)                           # ratio 1/600: e4m3 subnormal scale
    r0[80:96] = np.linspace(-0.05, 0.05, 16)                           # subnormal scale, saturating maximum
    r0[96:112] = np.linspace(-0.005, 0.005, 16)                        # ratio below 2^-10: s_b = 0
    r0[112:128] = 0.0                                                  # all-zero block
    r0[128:144] = [-0.0] * 8 + [1e-30] * 4 + [-1e-30] * 4              # negative zeros and bf16-tiny values
    r0[144:160] = np.linspace(-3.0, 3.0, 16)
    # ratio 6.375 / 6 = 1.0625 exactly, the midpoint of e4m3's 1 and 1.125: ties
    # to the even 1.  Scaling in the other order, 6.375 * fl(1/6), lands just
    # above the midpoint and would store 1.125.
    r0[160:176] = [6.375, -6.375, 3.0, -0.5] + [0.25 * i for i in range(12)]
    g = np.random.default_rng(0xB5F4)
    for i, std in enumerate([1.0, 0.02, 1e-3, 30.0, 300.0, 2e-4, 5.0], start=1):
        rows[i] = (g.standard_normal(K) * std).astype(np.float32)
    return bf16(np.stack(rows))


def fixture_scale_order():
    """Block maxima for which fl(fl(amax_b * gs) / 6) and fl(amax_b * fl(gs / 6))
    round to different e4m3 scales (found by exhaustive search over bf16 maxima
    for this tensor amax): the order of the two scale steps is observable."""
    row = np.zeros(48, dtype=np.float32)
    row[0] = 0.001190185546875                                        # the tensor maximum
    row[16:32] = [5.448237061500549e-08, -2.0e-08] + [1.0e-09 * i for i in range(14)]
    row[32:48] = [1.0896474123001099e-07, 3.0e-08] + [-2.0e-09 * i for i in range(14)]
    return bf16(row[None, :])


FIXTURES = {
    "structured": fixture_structured,
    "scale_order": fixture_scale_order,
    "normal_outliers": lambda: S.normal_bf16((64, 256), 1.0, 0xB5F5, outlier_frac=0.01),
    "small_weights": lambda: S.normal_bf16((32, 512), 0.02, 0xB5F6, outlier_frac=0.01),
}


@pytest.fixture(params=sorted(FIXTURES), scope="module")
def quantized(request):
    xb = FIXTURES[request.param]()
    words, scales, sg = O.quantize_nvfp4(xb)
    M, K = xb.shape
    sb = np.asarray(scales)[scale_index(M, K // 16)]
    return request.param, xb, unpack_words(words), sb, np.float32(sg)


# --------------------------------------------------------------------- pins --
def test_global_factor_is_the_f32_quotient(quantized):
    _, xb, _, _, sg = quantized
    amax = np.max(np.abs(f32(xb)))
    gs = np.float32(2688.0) / np.float32(amax)            # IEEE f32 division
    assert sg == np.float32(1.0) / gs


def test_block_scale_bytes_are_torch_e4m3_casts(quantized):
    _, xb, _, sb, _ = quantized
    x = f32(xb)
    gs = np.float32(2688.0) / np.max(np.abs(x))
    M, K = x.shape
    for r in range(M):
        for b in range(K // 16):
            amax_b = np.max(np.abs(x[r, 16 * b:16 * b + 16]))
            ratio = np.float32(np.float32(amax_b * gs) / np.float32(6.0))
            assert int(sb[r, b]) == torch_e4m3(ratio), (r, b, float(ratio))


def test_every_code_is_the_nearest_e2m1_value(quantized):
    name, xb, codes, sb, _ = quantized
    x = f32(xb)
    gs = np.float32(2688.0) / np.max(np.abs(x))
    M, K = x.shape
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    counts = {"tie": 0, "saturated": 0, "zero_scale": 0, "subnormal_scale": 0}
    for r in range(M):
        for b in range(K // 16):
            s = int(sb[r, b])
            blk = slice(16 * b, 16 * b + 16)
            if s == 0:
                counts["zero_scale"] += 1
                assert not codes[r, blk].any(), "a zero block scale leaves every code 0"
                continue
            if s < 0x08:
                counts["subnormal_scale"] += 1
            inv = np.float32(gs / np.float32(e4m3[s]))
            for k in range(16 * b, 16 * b + 16):
                v = np.float32(x[r, k] * inv)
                want = nearest_e2m1_code(v)
                assert int(codes[r, k]) == want, (name, r, k, float(v))
                a = abs(Fraction(float(v)))
                counts["saturated"] += a > 6
                counts["tie"] += a < 6 and any(abs(a - g) == abs(a - h) and g != h
                                               for g, h in zip(E2M1_GRID, E2M1_GRID[1:]) if g <= a <= h)
    if name == "structured":
        # the fixture reaches every case it was built for
        assert counts["tie"] >= 28 and counts["saturated"] >= 2
        assert counts["zero_scale"] >= 2 and counts["subnormal_scale"] >= 2


def test_structured_ties_round_to_even():
    """inv = 1 on the tie block: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2,
    2.5 -> 2, 3.5 -> 4, 5 -> 4 (the even neighbour of each midpoint)."""
    xb = fixture_structured()
    words, _, _ = O.quantize_nvfp4(xb)
    codes = unpack_words(words)[0]
    vals = [float(e2m1_value(int(c))) for c in codes[17:24]]
    assert vals == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert [float(e2m1_value(int(c))) for c in codes[24:31]] == [-0.0, -1.0, -1.0, -2.0, -2.0, -4.0, -4.0]
    assert all(int(c) & 8 for c in codes[24:31])          # the sign is kept, -0 included
    # inv = 1/2 on the next block: the same ties one binade up
    assert [float(e2m1_value(int(c))) for c in codes[33:40]] == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert int(codes[47]) == 0x8                            # -0.0 -> the negative zero code
    # saturation: 6.3125 and -6.25 at inv = 1 store +-6
    assert float(e2m1_value(int(codes[48]))) == 6.0 and float(e2m1_value(int(codes[51]))) == -6.0


def test_block_scale_tie_rounds_to_even():
    """amax_b * gs / 6 = 1.0625, halfway between the e4m3 values 1 and 1.125:
    the stored scale is 1 (byte 0x38, even mantissa), not 1.125 (0x39)."""
    xb = fixture_structured()
    _, scales, _ = O.quantize_nvfp4(xb)
    sb = np.asarray(scales)[scale_index(*xb.shape[:1], xb.shape[1] // 16)]
    assert int(sb[0, 10]) == 0x38


def test_per_element_error_bound(quantized):
    """|dequant - x| <= (half an e2m1 step at |x * inv|) * s_b / gs, plus the f32
    roundings of inv, x * inv and s_global; with a normal ue4m3 scale (relative
    rounding <= 2^-4) a saturated element stays within the top step's half too.
    The dequantization is the oracle's own (decode * scale * s_global)."""
    _, xb, codes, sb, sg = quantized
    x = f32(xb).astype(np.float64)
    M, K = x.shape
    gs = np.float32(2688.0) / np.float32(np.max(np.abs(x)))
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    words, scales, _ = O.quantize_nvfp4(xb)
    d = O.dequant_nvfp4(words, scales, float(sg), M, K)
    for r in range(M):
        for b in range(K // 16):
            s = int(sb[r, b])
            if s == 0:
                continue
            sv = e4m3[s]
            inv = np.float32(gs / np.float32(sv))
            for k in range(16 * b, 16 * b + 16):
                v = abs(float(np.float32(np.float32(x[r, k]) * inv)))
                if s < 0x08 and v > 6:
                    continue                                  # subnormal scale: saturation is checked above
                bound = float(half_step(v)) * sv / float(gs)
                slack = abs(x[r, k]) * 2.0 ** -20 + sv / float(gs) * 2.0 ** -20
                assert abs(d[r, k] - x[r, k]) <= bound + slack, (r, k, d[r, k], x[r, k], bound)
