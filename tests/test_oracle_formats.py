"""Pins for the oracle's codecs, packers, block-scale layout and rounding.

Each test checks the oracle against something other than itself: values the
pages print, a library routine (torch's float8_e4m3fn, numpy's rint/ldexp),
an independent algorithm (a bit-level round-to-nearest-even encoder, exact
rational arithmetic) or an invariant chosen so that a plausible slip (wrong
bias, wrong subnormal step, wrong sign bit, transposed index) fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)

FMTS6 = [O.E3M2, O.E2M3]
BITS = {O.E3M2: 6, O.E2M3: 6, O.E4M3: 8, O.E2M1: 4}
# (exponent bits, mantissa bits, bias) of each element format, from the
# formats' definitions (b12x _lib/fp6.py _decode_fp6_*; OCP e2m1/e4m3).
LAYOUT = {O.E3M2: (3, 2, 3), O.E2M3: (2, 3, 1), O.E4M3: (4, 3, 7), O.E2M1: (2, 1, 1)}


def magnitudes(fmt):
    n = 1 << (BITS[fmt] - 1)
    vals = [O.decode(fmt, c) for c in range(n)]
    return [v for v in vals if not math.isnan(v)]


# ------------------------------------------------------------------ decoders --
def test_printed_maxima_and_numerators():
    # b12x _lib/fp6.py constants and mx_gs_numerator; cubecl-tile packed.rs
    # fp4_codes_unpack_on_read ("0b0111 is 6.0") and fp8_codes_unpack_placed
    # (e4m3's smallest step 2^-9).  Values in tests/golden/printed_constants.json.
    g = golden("printed_constants.json")
    assert max(magnitudes(O.E3M2)) == g["FLOAT6_E3M2_MAX"]
    assert max(magnitudes(O.E2M3)) == g["FLOAT6_E2M3_MAX"]
    assert max(magnitudes(O.E4M3)) == g["FLOAT8_E4M3_MAX"]
    for name, fmt in (("e3m2", O.E3M2), ("e2m3", O.E2M3), ("e4m3", O.E4M3)):
        assert O.gs_numerator(fmt) == g["gs_numerator"][name]
    assert O.decode(O.E2M1, 0b0111) == g["e2m1_code_0b0111"]
    assert max(magnitudes(O.E2M1)) == 6.0
    assert O.decode(O.E4M3, 1) == 2.0 ** g["e4m3_smallest_step_log2"]


def test_e4m3_every_code_matches_torch():
    # check_fp8_codes_unpack (cubecl-tile packed.rs): every e4m3 code, bit for bit.
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = O.decode(O.E4M3, c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E2M1, O.E4M3])
def test_minifloat_structure(fmt):
    """Magnitudes rise with the code; within a binade the step is constant; the
    subnormal step equals the first normal binade's step (gradual underflow);
    the sign bit only flips the sign."""
    E, Mb, bias = LAYOUT[fmt]
    n = 1 << (BITS[fmt] - 1)
    vals = [O.decode(fmt, c) for c in range(n)]
    finite = [v for v in vals if not math.isnan(v)]
    assert all(b > a for a, b in zip(finite, finite[1:]))
    assert vals[0] == 0.0 and math.copysign(1, vals[0]) == 1.0
    per = 1 << Mb
    sub_step = vals[1] - vals[0]
    assert sub_step == 2.0 ** (1 - bias - Mb)
    for e in range(1 << E):
        binade = [v for v in vals[e * per:(e + 1) * per] if not math.isnan(v)]
        steps = {b - a for a, b in zip(binade, binade[1:])}
        want = 2.0 ** (max(e, 1) - bias - Mb)
        assert steps <= {want}, (e, steps)
    for c in range(n):
        neg = O.decode(fmt, c | n)
        if math.isnan(vals[c]):
            continue
        assert neg == -vals[c] and math.copysign(1, neg) == -1.0


def test_ue8m0_and_ue4m3_scales():
    # check_ue8m0_scales (cubecl-tile packed.rs): exponents -2..2, "the code is
    # the exponent biased by 127", so the scales are exact powers of two.
    for e in range(-2, 3):
        assert O.decode_ue8m0(e + 127) == 2.0 ** e
    assert math.isnan(O.decode_ue8m0(255))
    for c in range(0, 255):
        assert O.decode_ue8m0(c) == math.ldexp(1.0, c - 127)
    # e4m3_scales_reach_the_promoted_block: its sixteen scales (i+1)/2, i < 4*4,
    # are halves "which e4m3 holds exactly".
    for i in range(16):
        v = (i + 1) / 2
        assert O.decode(O.E4M3, O.encode(O.E4M3, v)) == v
    assert math.isnan(O.lib().bsqo_decode_ue4m3(0x80))


# ------------------------------------------------------------------ encoders --
def rne_encode(fmt, v):
    """Independent encoder: scale |v| to the format's integer grid of its binade
    and round with numpy's rint (ties to even), saturating at the maximum."""
    E, Mb, bias = LAYOUT[fmt]
    mx = max(magnitudes(fmt))
    a = min(abs(float(v)), mx)
    e = max(math.frexp(a)[1] - 1, 1 - bias) if a > 0 else 1 - bias
    step = 2.0 ** (e - Mb)
    q = float(np.rint(a / step)) * step
    q = min(q, mx)
    mags = magnitudes(fmt)
    code = mags.index(q)
    if math.copysign(1.0, float(v)) < 0:
        code |= 1 << (BITS[fmt] - 1)
    return code


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E2M1, O.E4M3])
def test_encoder_against_bitlevel_rne(fmt):
    mags = magnitudes(fmt)
    probes = set()
    for a, b in zip(mags, mags[1:]):
        mid = (a + b) / 2
        for v in (a, b, mid, np.nextafter(np.float32(mid), np.float32(0)),
                  np.nextafter(np.float32(mid), np.float32(np.inf))):
            probes.add(float(np.float32(v)))
    probes |= {0.0, mags[-1] * 1.01, mags[-1] * 100, 1e30, 1e-30, 2.0 ** -140}
    rng = np.random.default_rng(7)
    probes |= set(float(v) for v in (rng.standard_normal(4000) * mags[-1] / 3).astype(np.float32))
    for v in sorted(probes):
        for s in (v, -v):
            assert O.encode(fmt, s) == rne_encode(fmt, s), (fmt, s)


def test_e4m3_encoder_matches_torch_in_range():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
                        np.linspace(-463.9, 463.9, 4001)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.encode(O.E4M3, float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E2M1, O.E4M3])
def test_ties_go_to_even_code_and_saturate(fmt):
    mags = magnitudes(fmt)
    for i, (a, b) in enumerate(zip(mags, mags[1:])):
        mid = (a + b) / 2
        c = O.encode(fmt, mid)
        assert c in (i, i + 1) and c % 2 == 0, (fmt, mid, c)
    top = len(mags) - 1
    assert O.encode(fmt, mags[-1] * 4) == top
    assert O.encode(fmt, float("inf")) == top
    sign = 1 << (BITS[fmt] - 1)
    # Reading: the sign is kept on a zero result (IEEE conversion with saturation).
    assert O.encode(fmt, -0.0) == sign
    assert O.encode(fmt, -mags[1] / 4) == sign
    assert O.encode(fmt, 0.0) == 0


# ------------------------------------------------------------------- packing --
def test_fp6_pack_layout_printed_rule():
    # pack_4_fp6_codes: bits = c0 | c1<<6 | c2<<12 | c3<<18, bytes low first.
    assert list(O.pack_fp6(np.array([1, 0, 0, 0]))) == [1, 0, 0]
    assert list(O.pack_fp6(np.array([0, 1, 0, 0]))) == [0x40, 0, 0]
    assert list(O.pack_fp6(np.array([0, 0, 1, 0]))) == [0, 0x10, 0]
    assert list(O.pack_fp6(np.array([0, 0, 0, 1]))) == [0, 0, 0x04]
    assert list(O.pack_fp6(np.array([0x3F, 0x3F, 0x3F, 0x3F]))) == [0xFF, 0xFF, 0xFF]


def test_fp6_pack_is_a_bijection_on_all_24bit_patterns():
    allb = np.arange(1 << 24, dtype=np.uint32)
    packed = np.stack([allb & 0xFF, (allb >> 8) & 0xFF, (allb >> 16) & 0xFF], axis=1).astype(np.uint8)
    codes = O.unpack_fp6(packed.ravel(), 4 << 24)
    assert codes.max() < 64
    back = O.pack_fp6(codes)
    assert np.array_equal(back, packed.ravel())


# ---------------------------------------------------------------- swizzle ----
@pytest.mark.parametrize("rows,blocks", [(1, 1), (128, 4), (130, 5), (300, 128), (256, 16), (77, 3)])
def test_swizzle_closed_form_matches_permute_inverse(rows, blocks):
    """mxfp6_swizzled_scale_offset (closed form) against unswizzle_mxfp6_scales'
    flat path (reshape to (rp/128, cp/4, 32, 4, 4), permute (0,3,2,1,4)); and the
    map is a bijection of the padded grid."""
    rp, cp = -(-rows // 128) * 128, -(-blocks // 4) * 4
    assert O.scale_bytes(rows, blocks) == rp * cp
    flat = np.arange(rp * cp, dtype=np.int64)
    orig = flat.reshape(rp // 128, cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(rp, cp)
    seen = set()
    for r in range(rp):
        for b in range(cp):
            off = O.swz_offset(r, b, blocks)
            assert off == orig[r, b]
            seen.add(off)
    assert len(seen) == rp * cp


# ---------------------------------------------------------- scale arithmetic --
def test_ue8m0_exact_ceil_contains_the_ratio():
    """fp6_block_ue8m0_exact: the byte is ceil(log2 r) + 127, so
    2^(ue-127) >= r > 2^(ue-128) for every positive normal ratio r."""
    rng = np.random.default_rng(3)
    ratios = np.concatenate([np.exp2(rng.uniform(-120, 120, 20000)),
                             np.exp2(np.arange(-126, 127, dtype=np.float64))]).astype(np.float32)
    for r in ratios:
        r = float(r)
        ue = O.ue8m0_from_block_max(r, 1.0, 1.0)
        assert 2.0 ** (ue - 127) >= r > 2.0 ** (ue - 128), (r, ue)
    for k in range(-100, 100):
        assert O.ue8m0_from_block_max(2.0 ** k, 1.0, 1.0) == k + 127
        just_above = float(np.nextafter(np.float32(2.0 ** k), np.float32(np.inf)))
        assert O.ue8m0_from_block_max(just_above, 1.0, 1.0) == k + 128
    assert O.ue8m0_from_block_max(0.0, 5.0, 28.0) == 0
    assert O.ue8m0_from_block_max(2.0 ** -140, 1.0, 1.0) == 1     # subnormal ratio
    # the ratio is (amax*gs)/fmt_max with two rounded f32 steps
    a, g = np.float32(0.37), np.float32(12544.0 / 5.1)
    t = np.float32(a * g)
    r = np.float32(t / np.float32(28.0))
    assert O.ue8m0_from_block_max(float(a), float(g), 28.0) == O.ue8m0_from_block_max(float(r), 1.0, 1.0)


def test_ue8m0_output_scale_is_an_exact_power_of_two_times_gs():
    rng = np.random.default_rng(5)
    for gs in rng.uniform(1e-3, 1e5, 50).astype(np.float32):
        for ue in range(1, 254):
            with np.errstate(over="ignore"):
                want = np.float32(np.ldexp(np.float32(gs), 127 - ue))
            got = O.ue8m0_output_scale(ue, float(gs))
            assert np.float32(got) == want or (not np.isfinite(want) and not np.isfinite(got))
    assert O.ue8m0_output_scale(0, 3.0) == 0.0


# ------------------------------------------------------------------ rounding --
def test_f32_to_bf16_rule_and_vectors():
    # Winery-Strata elementwise_parity.cpp: the printed test words and the rule.
    words = [int(w, 16) for w in golden("bf16_rounding_words.json")["words"]]
    for w in words:
        f = float(np.array([w], dtype=np.uint32).view(np.float32)[0])
        got = O.f32_to_bf16(f)
        if (w & 0x7FFFFFFF) > 0x7F800000:
            assert (got & 0x7FFF) > 0x7F80                  # a NaN stays a NaN
        else:
            ref = torch.tensor([f], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert got == ref, hex(w)
    assert O.f32_to_bf16(float(np.array([0x3F808000], np.uint32).view(np.float32)[0])) == 0x3F80
    assert O.f32_to_bf16(float(np.array([0x3F818000], np.uint32).view(np.float32)[0])) == 0x3F82


def test_double_to_bf16_single_rounding():
    rng = np.random.default_rng(9)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-30, 30, 3000))
    vals += [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -40, 2.0 ** -133, 2.0 ** -134,
             3 * 2.0 ** -135, 1e39, -1e39, 0.0, -0.0]
    grid = [Fraction(0)]
    for v in vals:
        got = O.double_to_bf16(v)
        f = np.array([got << 16], dtype=np.uint32).view(np.float32)[0]
        x = Fraction(v)
        if abs(v) >= 2.0 ** 128 * (1 - 2 ** -9):
            assert np.isinf(f)
            continue
        # f is a nearest bf16; on a tie its mantissa LSB is even
        e = max(math.frexp(abs(v))[1] - 8, -133) if v != 0 else -133
        step = Fraction(2) ** e
        q = x / step
        lo = math.floor(q)
        if q - lo > Fraction(1, 2) or (q - lo == Fraction(1, 2) and lo % 2 == 1):
            lo += 1
        assert Fraction(float(f)) == lo * step, v
