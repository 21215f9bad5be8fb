"""Sanitizer-free memory and behaviour checks of the C ABI on the GPU
(techniques of the Winery-Strata elementwise_parity.cpp and vllm.cpp
test_ops_gdn.cpp pages): guard bands around every output stay untouched,
inputs are never modified, a captured CUDA graph replays to the same bits on
the caller's stream (so the calls neither synchronize nor allocate), bad
arguments return a status without launching, and the launch counters show
which kernel ran."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

GUARD = 0xA5


def guarded(nbytes, dev="cuda"):
    """A byte buffer with 256 guard bytes on each side; returns (whole, inner view)."""
    whole = torch.full((nbytes + 512,), GUARD, dtype=torch.uint8, device=dev)
    return whole, whole[256:256 + nbytes]


def guards_intact(whole, nbytes):
    h = whole.cpu().numpy()
    return (h[:256] == GUARD).all() and (h[256 + nbytes:] == GUARD).all()


def test_quantize_writes_only_its_outputs_and_keeps_inputs(bsq):
    M, K = 130, 1056
    x = S.normal_bf16((M, K), 0.02, 3, outlier_frac=0.01)
    xd = dev_tensor(x)
    x_before = xd.clone()
    for name in ("e3m2", "e2m3", "e4m3"):
        f = bsq.FMT_IDS[name]
        cb = M * (K if name == "e4m3" else 3 * K // 4)
        sb = bsq.scale_bytes(M, K // 32)
        cw, c = guarded(cb)
        sw, s = guarded(sb)
        gw, g = guarded(4)
        wsb = bsq.quantize_workspace_bytes(M, K)
        ww, ws = guarded(wsb)
        bsq.quantize_mxfp6_(xd, f, c, s, g.view(torch.float32), ws if wsb else None)
        torch.cuda.synchronize()
        assert guards_intact(cw, cb) and guards_intact(sw, sb) and guards_intact(gw, 4), name
        oc, os_, _ = O.quantize_mx(x, O.MX_FMTS[name])
        assert np.array_equal(host_bytes(c), oc.ravel()) and np.array_equal(host_bytes(s), os_)
    assert torch.equal(xd, x_before)


def test_products_write_only_their_outputs(bsq):
    M, N, K = 37, 300, 512
    x = S.normal_bf16((M, K), 1.0, 5)
    W = S.random_words((N, K // 8), 6)
    sc = S.choice_bytes(bsq.scale_bytes(N, K // 16), 7, list(range(0x10, 0x50)))
    Wd, scd, xd = dev_tensor(W), dev_tensor(sc), dev_tensor(x[:32])
    before = [t.clone() for t in (Wd, scd, xd)]
    yw, y = guarded(32 * N * 4)
    bsq.gemv_nvfp4_(xd, Wd, scd, None, y.view(torch.float32).view(32, N), N, K)
    torch.cuda.synchronize()
    assert guards_intact(yw, 32 * N * 4)
    A = S.random_words((M, K // 8), 8)
    sA = S.choice_bytes(bsq.scale_bytes(M, K // 16), 9, list(range(0x10, 0x50)))
    Ad, sAd = dev_tensor(A), dev_tensor(sA)
    gw_, Y = guarded(M * N * 2)
    bsq.gemm_nvfp4_(Ad, sAd, None, Wd, scd, None, Y.view(torch.bfloat16).view(M, N), M, N, K)
    torch.cuda.synchronize()
    assert guards_intact(gw_, M * N * 2)
    for b, t in zip(before, (Wd, scd, xd)):
        assert torch.equal(b, t)


def test_graph_capture_replays_on_the_callers_stream(bsq):
    """Capture quantize + GEMM + a following scale in a graph on a side stream and
    replay twice: identical bits both times, equal to the eager result doubled.
    The activation quantizer is the single cluster launch, the weight quantizer
    the cooperative one-pass launch (memset of its counter + the kernel)."""
    M, N, K = 128, 1024, 256
    a = dev_tensor(S.normal_bf16((M, K), 0.02, 1))
    w = dev_tensor(S.normal_bf16((N, K), 0.02, 2))
    # eager (also loads the kernels before capture)
    ca, sa, ga = bsq.quantize_mxfp6(a, "e3m2")
    cw, sw, gw = bsq.quantize_mxfp6(w, "e3m2")
    y_eager = bsq.gemm_mxfp6(ca, "e3m2", sa, ga, cw, "e3m2", sw, gw, K, out_dtype=torch.float32)
    torch.cuda.synchronize()
    y = torch.empty_like(y_eager)
    ws = torch.empty(bsq.quantize_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            bsq.quantize_mxfp6_(a, 0, ca, sa, ga, stream=s)
            bsq.quantize_mxfp6_(w, 0, cw, sw, gw, ws, stream=s)
            bsq.gemm_mxfp6_(ca, 0, sa, ga, cw, 0, sw, gw, y, M, N, K, stream=s)
            y.mul_(2.0)
    outs = []
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], y_eager * 2.0)


def test_bad_arguments_return_status_and_launch_nothing(bsq):
    L = bsq.load()
    bsq.reset_launch_counts()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4 * 48, dtype=torch.uint8, device="cuda")
    s = torch.zeros(bsq.scale_bytes(4, 2), dtype=torch.uint8, device="cuda")
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    null = ctypes.c_void_p(0)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.bsq_quantize_mxfp6(null, 4, 64, 0, p(c), p(s), p(g), null, 0, st) == 1     # null input
    assert L.bsq_quantize_mxfp6(p(x), 4, 48, 0, p(c), p(s), p(g), null, 0, st) == 1      # K % 32
    assert L.bsq_quantize_mxfp6(p(x), 4, 64, 9, p(c), p(s), p(g), null, 0, st) == 1      # bad format
    assert L.bsq_quantize_mxfp6(ctypes.c_void_p(x.data_ptr() + 2), 4, 64, 0, p(c), p(s), p(g), null, 0, st) == 3
    big = torch.zeros((4096, 4096), dtype=torch.bfloat16, device="cuda")
    cb = torch.zeros(4096 * 3072, dtype=torch.uint8, device="cuda")
    sb = torch.zeros(bsq.scale_bytes(4096, 128), dtype=torch.uint8, device="cuda")
    assert L.bsq_quantize_mxfp6(p(big), 4096, 4096, 0, p(cb), p(sb), p(g), null, 0, st) == 4   # no workspace
    assert L.bsq_gemv_nvfp4(p(x), p(c), p(s), null, p(g), 1, 33, 8, 64, st) == 1             # M > 32
    assert L.bsq_gemm_nvfp4(p(c), p(s), null, p(c), p(s), null, p(g), 1, 4, 4, 96, st) == 1  # K % 64
    assert L.bsq_gemm_mxfp6(p(c), 0, p(s), null, p(c), 0, p(s), null, p(g), 1, 4, 4, 64, st) == 1  # K % 128
    assert L.bsq_quantize_mxfp6_act(p(x), 4, 64, 3, 0, p(c), p(s), p(g), null, null, 0, st) == 1      # bad activation
    assert L.bsq_quantize_mxfp6_act(p(x), 4, 48, 1, 0, p(c), p(s), p(g), null, null, 0, st) == 1      # K % 32
    assert L.bsq_quantize_mxfp6_containers(p(x), 4, 64, 2, p(c), p(s), p(g), null, 0, st) == 1       # e4m3 has bytes
    rc = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert L.bsq_quantize_grouped_mxfp6(p(x), 0, 2, 64, p(rc), p(g), 0, p(c), p(s), p(g), st) == 1   # G < 1
    assert L.bsq_quantize_grouped_mxfp6(p(x), 2, 2, 64, null, p(g), 0, p(c), p(s), p(g), st) == 1    # no counts
    assert L.bsq_gemm_grouped_mxfp6(p(c), 0, p(s), p(g), p(c), 0, p(s), p(g), p(rc), p(g), 0,
                                    2, 2, 4, 64, st) == 1                                            # K % 128
    assert L.bsq_gemm_grouped_mxfp6(p(c), 0, p(s), p(g), p(c), 0, p(s), p(g), p(rc), p(g), 0,
                                    300, 2, 4, 128, st) == 1                                         # G > 256
    xa = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(bsq.gemm_quant_a_workspace_bytes(), dtype=torch.uint8, device="cuda")
    wsb = ws.numel()
    assert L.bsq_gemm_mxfp6_quant_a(null, 0, p(c), 0, p(s), null, p(g), 1, null, 4, 4, 128, p(ws), wsb, st) == 1  # null x
    assert L.bsq_gemm_mxfp6_quant_a(p(xa), 0, p(c), 0, p(s), null, p(g), 1, null, 4, 4, 64, p(ws), wsb, st) == 1  # K % 128
    assert L.bsq_gemm_mxfp6_quant_a(p(xa), 0, p(c), 0, p(s), null, p(g), 1, null, 4, 4, 128, p(ws), 64, st) == 4  # small ws
    assert L.bsq_gemm_mxfp6_quant_a(p(xa), 0, p(c), 0, p(s), null, p(g), 1, null, 4, 4, 128, null, wsb, st) == 4  # no ws
    assert L.bsq_gemm_mxfp6_quant_a(ctypes.c_void_p(xa.data_ptr() + 2), 0, p(c), 0, p(s), null, p(g), 1, null,
                                    4, 4, 128, p(ws), wsb, st) == 3                                               # x misaligned
    assert sum(bsq.launch_count(k) for k in bsq.KERNEL_IDS) == 0


def test_launch_counters_show_the_dispatch(bsq):
    bsq.reset_launch_counts()
    x = dev_tensor(S.normal_bf16((16, 4096), 1.0, 4))
    bsq.quantize_mxfp6(x, "e2m3")                   # small: one cluster launch
    assert bsq.launch_count("quant_small") == 1 and bsq.launch_count("amax") == 0
    xb = dev_tensor(S.normal_bf16((1024, 2048), 1.0, 5))
    bsq.quantize_nvfp4(xb)                          # fits shared memory: one cooperative launch
    assert bsq.launch_count("amax") == 0 and bsq.launch_count("quant_nvfp4") == 1
    xc = dev_tensor(S.normal_bf16((4480, 4096), 1.0, 6))
    bsq.quantize_nvfp4(xc)                          # beyond it: amax pass + encode pass
    assert bsq.launch_count("amax") == 1 and bsq.launch_count("quant_nvfp4") == 2
    torch.cuda.synchronize()
