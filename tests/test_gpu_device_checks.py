"""The device bounds-check build (-DBSQ_DEVICE_CHECKS), end to end.

In that copy of the library every global store of the kernels, and every
global load whose address a kernel computes, is checked against the extent of
its buffer as the call's sizes give it; an access that leaves its buffer is
skipped and the first one is recorded in the device error word (bit 31, the
site in bits 24..30, the low 24 bits of the access's offset).  The checks only
add guards, so on legal calls the checked build must (a) record nothing and
(b) write exactly the bytes the regular build writes -- whose outputs the
parity tests hold to the oracle.  Every entry point runs here on ragged shapes
that span several tiles and take each kernel path (cluster / one-pass /
two-pass quantizers; persistent, CTA-pair, split-K and grouped GEMMs; the
resident, staged and tensor-core nvfp4 GEMVs and the MX GEMV; dequantizers).

A second test build tightens one site's extent by one unit (the GEMV's y
store), so exactly one legal store -- the last element of y -- is recorded and
skipped: the status, the site and the offset come back through the C ABI, that
element keeps its canary, every other output matches, and the context stays
usable.  Neither build makes an out-of-bounds access."""
import contextlib
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor

pytestmark = pytest.mark.gpu

BSQ_ERR_DEVICE_CHECK = 7
CHECK_FLAG = 0x80000000
SITE_GEMV_Y = 0x24
UE4M3_CODES = list(range(0x08, 0x68))


@pytest.fixture(scope="module")
def checked_path(bsq):
    from block_scaled_precision_packed_gb300 import build as B
    return B.build_variant("devchecks", ["BSQ_DEVICE_CHECKS"], rebuilt=tuple(B.SOURCES))


@pytest.fixture(scope="module")
def tight_path(bsq):
    from block_scaled_precision_packed_gb300 import build as B
    return B.build_variant("devtight", ["BSQ_DEVICE_CHECKS", f"BSQ_TEST_CHECK_TIGHT_SITE={SITE_GEMV_Y}"],
                           rebuilt=("gemv.cu",))


@contextlib.contextmanager
def library(bsq, path):
    """Route the binding's calls to another build of the library for a while."""
    saved = bsq._lib
    bsq._lib = None
    try:
        bsq.load(path)
        yield
    finally:
        bsq._lib = saved


def nvfp4_operand(R, K, seed):
    return (dev_tensor(S.random_words((R, K // 8), seed)),
            dev_tensor(S.choice_bytes(((R + 127) // 128 * 128) * ((K // 16 + 3) // 4 * 4), seed + 1, UE4M3_CODES)))


def x_bf16(M, K, seed, std=0.5):
    return dev_tensor(S.normal_bf16((M, K), std, seed, outlier_frac=0.01)).view(torch.bfloat16)


def every_entry_point(bsq, mx_ops):
    """One call of each entry point and path; returns {name: [output tensors]}."""
    out = {}
    g = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")   # noqa: E731
    # quantizers: one cluster (<= 64 Ki values), one-pass, two-pass (amax + encode)
    for M, K in [(100, 512), (1000, 4160), (4100, 8192)]:
        x = x_bf16(M, K, M + K)
        for f in ("e3m2", "e2m3", "e4m3"):
            out[f"quant_{f}_{M}x{K}"] = list(bsq.quantize_mxfp6(x, f))
        out[f"quant_nvfp4_{M}x{K}"] = list(bsq.quantize_nvfp4(x))
        for f in ("e3m2", "e2m3"):
            M_, K_ = x.shape
            codes = torch.empty((M_, K_), dtype=torch.uint8, device="cuda")
            sc = torch.empty(bsq.scale_bytes(M_, K_ // 32), dtype=torch.uint8, device="cuda")
            sg = torch.empty(1, dtype=torch.float32, device="cuda")
            ws = torch.empty(max(16, bsq.quantize_workspace_bytes(M_, K_)), dtype=torch.uint8, device="cuda")
            bsq.quantize_mxfp6_containers_(x, bsq.FMT_IDS[f], codes, sc, sg, ws)
            out[f"containers_{f}_{M}x{K}"] = [codes, sc, sg]
    for M, K in [(100, 256), (1000, 4096)]:
        out[f"act_relu2_{M}"] = list(bsq.quantize_mxfp6_act(x_bf16(M, K, 7), bsq.ACT_RELU2, "e3m2", want_act=True))
        out[f"act_silu_{M}"] = list(bsq.quantize_mxfp6_act(x_bf16(M, 2 * K, 8), bsq.ACT_SILU_MUL, "e2m3",
                                                           want_act=True))
    xs = [x_bf16(130, 512, 9), x_bf16(64, 1024, 10)]
    batch = []
    for x in xs:
        M_, K_ = x.shape
        batch.append((x, torch.empty((M_, 3 * K_ // 4), dtype=torch.uint8, device="cuda"),
                      torch.empty(bsq.scale_bytes(M_, K_ // 32), dtype=torch.uint8, device="cuda"),
                      torch.empty(1, dtype=torch.float32, device="cuda")))
    bsq.quantize_mxfp6_batch_(batch, bsq.E3M2,
                              torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda"))
    out["quant_batch"] = [t for b in batch for t in b[1:]]
    G, R, C = 3, 200, 256
    xg = dev_tensor(S.normal_bf16((G * R, C), 0.5, 11)).view(torch.bfloat16).reshape(G, R, C)
    rc = torch.tensor([200, 0, 77], dtype=torch.int32, device="cuda")
    gq = [torch.empty((G, R, 3 * C // 4), dtype=torch.uint8, device="cuda"),
          torch.empty((G, bsq.scale_bytes(R, C // 32)), dtype=torch.uint8, device="cuda"),
          torch.empty(G, dtype=torch.float32, device="cuda")]
    bsq.quantize_grouped_mxfp6_(xg, rc, torch.full((G,), 30.0, device="cuda"), bsq.E3M2, *gq)
    out["quant_grouped"] = gq

    # GEMMs: CTA pairs (ragged rows and N), single 256-wide CTAs, split-K, MX, grouped, quantizer in the GEMM
    for M, N, K in [(300, 9800, 320), (1, 256, 64), (100, 300, 4096), (200, 333, 320)]:
        A, sA = nvfp4_operand(M, K, M)
        W, sW = nvfp4_operand(N, K, N)
        for dt in (torch.float32, torch.bfloat16):
            out[f"gemm_nvfp4_{M}x{N}x{K}_{dt}"] = [bsq.gemm_nvfp4(A, sA, g(0.5), W, sW, g(0.25), K, out_dtype=dt)]
    (A, sA, gA), (W, sW, gW) = mx_ops["e4m3", 200, 384], mx_ops["e2m3", 333, 384]
    for dt in (torch.float32, torch.bfloat16):
        out[f"gemm_mx_{dt}"] = [bsq.gemm_mxfp6(A, "e4m3", sA, gA, W, "e2m3", sW, gW, 384, out_dtype=dt)]
    (A, sA, gA), (W, sW, gW) = mx_ops["e3m2", 1100, 128], mx_ops["e3m2", 4400, 128]
    out["gemm_mx_many_tiles"] = [bsq.gemm_mxfp6(A, "e3m2", sA, gA, W, "e3m2", sW, gW, 128)]
    Wq, sWq, gWq = mx_ops["e2m3", 333, 384]
    out["gemm_quant_a"] = list(bsq.gemm_mxfp6_quant_a(x_bf16(200, 384, 12), "e3m2", Wq, "e2m3", sWq, gWq, 384))
    Yg = torch.full((G, R, 320), float("nan"), dtype=torch.float32, device="cuda")
    Wg = [torch.empty((G, 320, 3 * C // 4), dtype=torch.uint8, device="cuda"),
          torch.empty((G, bsq.scale_bytes(320, C // 32)), dtype=torch.uint8, device="cuda"),
          torch.empty(G, dtype=torch.float32, device="cuda")]
    bsq.quantize_grouped_mxfp6_(dev_tensor(S.normal_bf16((G * 320, C), 0.02, 13)).view(torch.bfloat16).reshape(G, 320, C),
                                torch.full((G,), 320, dtype=torch.int32, device="cuda"),
                                torch.full((G,), 1000.0, device="cuda"), bsq.E2M3, *Wg)
    bsq.gemm_grouped_mxfp6_(gq[0], bsq.E3M2, gq[1], gq[2], Wg[0], bsq.E2M3, Wg[1], Wg[2], rc, Yg, G, R, 320, C)
    out["gemm_grouped"] = [Yg]

    # GEMVs: resident (M = 1), staged (M = 2..16), tensor-core (M = 17..32), MX
    for M, N, K in [(1, 1000, 2048), (2, 300, 320), (8, 1000, 2048), (13, 129, 1024), (32, 2 * 152 * 128 + 100, 512)]:
        W, sW = nvfp4_operand(N, K, 3 * N)
        x = x_bf16(M, K, M, std=1.0)
        for dt in (torch.float32, torch.bfloat16):
            out[f"gemv_nvfp4_{M}x{N}x{K}_{dt}"] = [bsq.gemv_nvfp4(x, W, sW, g(0.375), K, out_dtype=dt)]
    for f in ("e3m2", "e4m3"):
        W, sW, gW = mx_ops[f, 333, 384]
        for M in (1, 8, 32):
            out[f"gemv_{f}_{M}"] = [bsq.gemv_mxfp6(x_bf16(M, 384, 20 + M, std=1.0), W, f, sW, gW, 384)]

    # dequantizers
    W, sW = nvfp4_operand(200, 320, 5)
    d = torch.empty((200, 320), dtype=torch.float32, device="cuda")
    bsq.dequant_nvfp4_(W, sW, g(0.5), d, 200, 320)
    out["dequant_nvfp4"] = [d]
    W, sW, gW = mx_ops["e3m2", 333, 384]
    d = torch.empty((333, 384), dtype=torch.float32, device="cuda")
    bsq.dequant_mxfp6_(W, bsq.E3M2, sW, gW, d, 333, 384)
    out["dequant_mx"] = [d]
    torch.cuda.synchronize()
    return out


def mx_operands(bsq):
    """MX operands made once by the regular library and shared by both builds."""
    ops = {}
    for f, R, K in [("e4m3", 200, 384), ("e2m3", 333, 384), ("e3m2", 1100, 128), ("e3m2", 4400, 128),
                    ("e3m2", 333, 384), ("e4m3", 333, 384)]:
        ops[f, R, K] = bsq.quantize_mxfp6(x_bf16(R, K, R + K, std=0.05), f)
    torch.cuda.synchronize()
    return ops


def as_bytes(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def test_checked_build_records_nothing_and_writes_the_same_bytes(bsq, checked_path):
    ops = mx_operands(bsq)
    want = every_entry_point(bsq, ops)
    with library(bsq, checked_path):
        assert bsq.device_error() == (0, 0)
        got = every_entry_point(bsq, ops)
        st, code = bsq.device_error()
    assert (st, code) == (0, 0), f"a device check fired on a legal call: status {st}, word 0x{code:08x}"
    assert got.keys() == want.keys()
    for name in want:
        for i, (a, b) in enumerate(zip(want[name], got[name])):
            assert np.array_equal(as_bytes(a), as_bytes(b)), f"{name}[{i}] differs in the checked build"


@pytest.mark.parametrize("M", [1, 3, 32])
def test_a_failed_check_is_recorded_skipped_and_reported(bsq, tight_path, M):
    N, K = 300, 512
    W, sW = nvfp4_operand(N, K, 77)
    x = x_bf16(M, K, 78, std=1.0)
    g = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    want = bsq.gemv_nvfp4(x, W, sW, g, K, out_dtype=torch.float32)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with library(bsq, tight_path):
        bsq.gemv_nvfp4_(x, W, sW, g, y, N, K)
        st, code = bsq.device_error()
        assert bsq.device_error() == (0, 0), "reading the word clears it"
    assert st == BSQ_ERR_DEVICE_CHECK
    assert code == CHECK_FLAG | SITE_GEMV_Y << 24 | (M * N - 1), f"word 0x{code:08x}"
    yf, wf = y.flatten().cpu(), want.flatten().cpu()
    assert torch.isnan(yf[-1]), "the recorded store was skipped"
    assert torch.equal(yf[:-1], wf[:-1]), "every other output is written as by the regular build"
    # the regular library in the same process: the context is usable
    again = bsq.gemv_nvfp4(x, W, sW, g, K, out_dtype=torch.float32)
    assert torch.equal(again.cpu(), want.cpu())
