"""The allocation-free quantizer entry point, bsq_quantize_mxfp6_noalloc.

It exists for callers that cannot allocate device memory on this path (a
plugin whose host framework owns all device memory, or a latency-critical loop
where an allocation is not acceptable): its scratch -- the amax pass's partial
maxima -- lives in a device array inside the library.  This test calls it
through the C ABI and checks its codes, scales and s_global byte for byte
against bsq_quantize_mxfp6 (with a caller workspace) on two calls in a row with
different shapes, so a stale scratch from the first call cannot go unnoticed.
It sits in its own file, collected last, and passes alone or after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor, host_bytes

pytestmark = pytest.mark.gpu


def _outputs(bsq, M, K, fmt, dev):
    row_bytes = K if fmt == bsq.E4M3 else 3 * K // 4
    return (torch.empty((M, row_bytes), dtype=torch.uint8, device=dev),
            torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev),
            torch.empty(1, dtype=torch.float32, device=dev))


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(bsq):
    L = bsq.load()
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    cases = [(1024, 1280, "e3m2", 21), (600, 2048, "e2m3", 22)]    # both above the single-launch size
    for M, K, name, seed in cases:
        fmt = bsq.FMT_IDS[name]
        x = dev_tensor(S.normal_bf16((M, K), 0.02, seed, outlier_frac=0.01))
        c0, s0, g0 = _outputs(bsq, M, K, fmt, dev)
        c1, s1, g1 = _outputs(bsq, M, K, fmt, dev)
        ws = torch.empty(bsq.quantize_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
        assert L.bsq_quantize_mxfp6(p(x), M, K, fmt, p(c0), p(s0), p(g0), p(ws), ws.numel(), stream) == 0
        assert L.bsq_quantize_mxfp6_noalloc(p(x), M, K, fmt, p(c1), p(s1), p(g1), stream) == 0
        torch.cuda.synchronize()
        assert np.array_equal(host_bytes(c1), host_bytes(c0)), (M, K, name)
        assert np.array_equal(host_bytes(s1), host_bytes(s0)), (M, K, name)
        assert np.array_equal(host_bytes(g1), host_bytes(g0)), (M, K, name)


def test_noalloc_small_and_invalid(bsq):
    L = bsq.load()
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    M, K = 16, 4096                                                  # the single cluster launch
    x = dev_tensor(S.normal_bf16((M, K), 1.0, 23))
    c0, s0, g0 = bsq.quantize_mxfp6(x, "e4m3")
    c1, s1, g1 = _outputs(bsq, M, K, bsq.E4M3, dev)
    assert L.bsq_quantize_mxfp6_noalloc(p(x), M, K, bsq.E4M3, p(c1), p(s1), p(g1), stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(g0, g1)
    assert L.bsq_quantize_mxfp6_noalloc(p(x), M, 48, bsq.E4M3, p(c1), p(s1), p(g1), stream) == 1
