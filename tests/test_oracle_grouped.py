"""CPU pins for the oracle's grouped (MoE) MX quantizer and grouped product
(b12x _lib/fp6.py quantize_grouped_mxfp6_torch, pack_grouped_fp6_values,
as_grouped_mxfp6_scale_view): per-group global scales given by the caller,
row_counts valid rows per group, group-major codes, per-group swizzled scales."""
import numpy as np
import pytest

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S

FMAX = {O.E3M2: 28.0, O.E2M3: 7.5, O.E4M3: 448.0}


def groups(G, R, C, seed):
    return S.normal_bf16((G * R, C), 0.5, seed, outlier_frac=0.01).reshape(G, R, C)


def amax_gs(xg, fmt):
    a = np.abs((xg.astype(np.uint32) << 16).view(np.float32)).max()
    return np.float32(448.0 * FMAX[fmt]) / np.float32(a)


@pytest.mark.parametrize("fmt", [O.E3M2, O.E2M3, O.E4M3])
def test_group_with_amax_scale_is_the_tensor_quantizer(fmt):
    """Given gs = 448*fmt_max/amax of its rows, a group quantizes exactly like the
    per-tensor quantizer on those rows (codes, scales of valid rows, s_global)."""
    G, R, C = 3, 150, 96
    x = groups(G, R, C, 21)
    rc = [150, 61, 128]
    gs = [amax_gs(x[g, :rc[g]], fmt) for g in range(G)]
    codes, scales, sg = O.quantize_grouped_mx(x, rc, gs, fmt)
    for g in range(G):
        c, s, g1 = O.quantize_mx(np.ascontiguousarray(x[g, :rc[g]]), fmt)
        assert np.array_equal(codes[g, :rc[g]], c)
        assert sg[g] == np.float32(g1)
        ue = O.quantize_mx_rows(np.ascontiguousarray(x[g, :rc[g]]), fmt, np.arange(rc[g]))[1]
        for r in range(rc[g]):
            for b in range(C // 32):
                assert scales[g, O.swz_offset(r, b, C // 32)] == ue[r, b]


def test_rows_past_the_count_are_zero():
    G, R, C = 4, 130, 64
    x = groups(G, R, C, 22)
    rc = [0, 1, 129, 500]                                   # 500 clamps to R
    codes, scales, sg = O.quantize_grouped_mx(x, rc, [1.0, 2.0, 3.0, 4.0], O.E3M2)
    assert not codes[0].any() and not scales[0].any()
    assert not codes[1, 1:].any() and not codes[2, 129:].any()
    for g, n in ((1, 1), (2, 129), (3, 130)):
        live = {O.swz_offset(r, b, C // 32) for r in range(n) for b in range(C // 32)}
        dead = np.array(sorted(set(range(scales.shape[1])) - live), dtype=np.int64)
        assert not scales[g, dead].any()
    assert codes[3].any() and sg[1] == np.float32(0.5)


def test_doubling_the_global_scale_raises_every_scale_by_one():
    """The page's codes are x*gs/block_scale: doubling gs doubles each block ratio,
    so every nonzero UE8M0 byte grows by one and the codes do not change."""
    G, R, C = 2, 64, 128
    x = groups(G, R, C, 23)
    a = O.quantize_grouped_mx(x, [64, 40], [300.0, 77.0], O.E2M3)
    b = O.quantize_grouped_mx(x, [64, 40], [600.0, 154.0], O.E2M3)
    assert np.array_equal(a[0], b[0])
    nz = a[1] != 0
    assert np.array_equal(b[1][nz], a[1][nz] + 1) and not b[1][~nz].any()
    assert np.array_equal(b[2] * 2, a[2])


def test_page_layouts():
    """Codes in the page's [R, 3C/4, G] order are the group-major codes
    transposed; the page's 6-D scale view [32, 4, R/128, 4, C/128, G] of the
    storage addresses (row 128rb + 32i4 + i32, block 4cb + j4) of group g."""
    G, R, C = 2, 256, 256
    x = groups(G, R, C, 24)
    codes, scales, _ = O.quantize_grouped_mx(x, [256, 200], [900.0, 400.0], O.E3M2)
    page_codes = codes.transpose(1, 2, 0)
    for g in range(G):
        unpacked = np.stack([O.unpack_fp6(np.ascontiguousarray(page_codes[r, :, g]), C) for r in range(R)])
        assert np.array_equal(O.pack_fp6(unpacked).reshape(R, -1), codes[g])
    view = scales.reshape(G, R // 128, (C // 32) // 4, 32, 4, 4).transpose(3, 4, 1, 5, 2, 0)
    ue = [O.quantize_mx_rows(np.ascontiguousarray(x[g]), O.E3M2, np.arange(R))[1] for g in range(G)]
    gs = [900.0, 400.0]
    for g, n in ((0, 256), (1, 200)):
        ug = O.quantize_grouped_mx(x[g:g + 1], [n], [gs[g]], O.E3M2)[1][0]
        v = ug.reshape(R // 128, (C // 32) // 4, 32, 4, 4).transpose(2, 3, 0, 4, 1)
        assert np.array_equal(v, view[..., g])
        rb, i4, i32, cb, j4 = 1, 2, 5, 1, 3
        assert view[i32, i4, rb, j4, cb, g] == scales[g, O.swz_offset(128 * rb + 32 * i4 + i32, 4 * cb + j4, C // 32)]


def test_grouped_product_is_the_plain_product_per_group():
    G, R, N, K = 2, 130, 64, 128
    x = groups(G, R, K, 25)
    w = groups(G, N, K, 26)
    rc = [130, 33]
    A, sA, gA = O.quantize_grouped_mx(x, rc, [2000.0, 1500.0], O.E3M2)
    W, sW, gW = O.quantize_grouped_mx(w, [N, N], [2500.0, 2600.0], O.E2M3)
    y, s = O.gemm_grouped_mx(A, O.E3M2, sA, gA, W, O.E2M3, sW, gW, rc, K)
    assert not y[1, 33:].any() and not s[1, 33:].any()
    # one output by brute force from the dequantized operands
    dA = O.dequant_mx(np.ascontiguousarray(A[1, :33]), O.E3M2, np.ascontiguousarray(sA[1]), float(gA[1]), 33, K)
    dW = O.dequant_mx(np.ascontiguousarray(W[1]), O.E2M3, np.ascontiguousarray(sW[1]), float(gW[1]), N, K)
    ref = np.asarray(dA, dtype=np.float64).reshape(33, K)[7] @ np.asarray(dW, dtype=np.float64).reshape(N, K)[5]
    assert abs(y[1, 7, 5] - ref) <= 1e-12 * max(1.0, abs(ref)) + 1e-9 * s[1, 7, 5]
