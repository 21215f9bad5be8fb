"""The products partition by N with no exchange: a weight split into shards at
128-row boundaries (its scale buffer splits there into contiguous pieces: the
swizzle atoms are row-block major) gives, shard by shard, exactly the columns of
the unsharded product -- what a multi-GPU split of W would compute, run here
one shard after another on one GPU.  The shapes keep the same K split in the
sharded and unsharded GEMMs, so the summation order, and the bits, agree."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor

pytestmark = pytest.mark.gpu


def _scale_rows(sc, row0, rows, blocks):
    """The bytes of rows [row0, row0 + rows) of a swizzled scale buffer (row0, rows multiples of 128)."""
    per_rb = O.scale_bytes(128, blocks)
    return sc[row0 // 128 * per_rb:(row0 + rows) // 128 * per_rb]


@pytest.mark.parametrize("M", [1, 8, 32])
def test_gemv_nvfp4_sharded_by_n_is_bit_identical(bsq, M):
    N, K, cut = 768, 2048, 384
    x = dev_tensor(S.normal_bf16((M, K), 1.0, 60 + M))
    W = S.random_words((N, K // 8), 61)
    sc = S.choice_bytes(O.scale_bytes(N, K // 16), 62, list(range(0x08, 0x68)))
    g = torch.tensor([0.75], device="cuda")
    full = bsq.gemv_nvfp4(x, dev_tensor(W), dev_tensor(sc), g, K, out_dtype=torch.float32)
    parts = []
    for r0, r1 in ((0, cut), (cut, N)):
        parts.append(bsq.gemv_nvfp4(x, dev_tensor(W[r0:r1]), dev_tensor(_scale_rows(sc, r0, r1 - r0, K // 16)), g, K,
                                    out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), full)


def test_gemm_nvfp4_sharded_by_n_is_bit_identical(bsq):
    M, N, K, cut = 256, 512, 512, 256
    A = S.random_words((M, K // 8), 63)
    sA = S.choice_bytes(O.scale_bytes(M, K // 16), 64, list(range(0x08, 0x68)))
    W = S.random_words((N, K // 8), 65)
    sW = S.choice_bytes(O.scale_bytes(N, K // 16), 66, list(range(0x08, 0x68)))
    gA, gW = torch.tensor([0.5], device="cuda"), torch.tensor([1.25], device="cuda")
    Ad, sAd = dev_tensor(A), dev_tensor(sA)
    full = bsq.gemm_nvfp4(Ad, sAd, gA, dev_tensor(W), dev_tensor(sW), gW, K, out_dtype=torch.float32)
    parts = [bsq.gemm_nvfp4(Ad, sAd, gA, dev_tensor(W[r0:r1]), dev_tensor(_scale_rows(sW, r0, r1 - r0, K // 16)), gW,
                            K, out_dtype=torch.float32) for r0, r1 in ((0, cut), (cut, N))]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), full)


def test_gemm_mx_sharded_by_n_is_bit_identical(bsq):
    M, N, K, cut = 128, 1024, 1024, 512
    a = S.normal_bf16((M, K), 0.02, 67, outlier_frac=0.01)
    w = S.normal_bf16((N, K), 0.02, 68, outlier_frac=0.01)
    ca, sa, ga = O.quantize_mx(a, O.E3M2)
    cw, sw, gw = O.quantize_mx(w, O.E3M2)
    gA, gW = torch.tensor([ga], device="cuda"), torch.tensor([gw], device="cuda")
    cad, sad = dev_tensor(ca), dev_tensor(sa)
    full = bsq.gemm_mxfp6(cad, "e3m2", sad, gA, dev_tensor(cw), "e3m2", dev_tensor(sw), gW, K, out_dtype=torch.float32)
    parts = [bsq.gemm_mxfp6(cad, "e3m2", sad, gA, dev_tensor(np.ascontiguousarray(cw[r0:r1])), "e3m2",
                            dev_tensor(_scale_rows(sw, r0, r1 - r0, K // 32)), gW, K, out_dtype=torch.float32)
             for r0, r1 in ((0, cut), (cut, N))]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), full)
