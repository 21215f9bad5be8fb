"""A bounded device wait that runs out, end to end: failure detection without a
GPU fault.

A test-only copy of the library is built with two compile-time hooks: every
spin-wait gives up after 10 ms (instead of 2 s), and the one-pass quantizer's
last CTA never counts itself in at the grid-wide barrier.  The other CTAs'
bounded waits then run out with nothing in flight (the barrier comes after the
slice loads have landed, and the quantizer holds no TMEM), record the barrier's
site in the device error word and return; the skipped CTA's own wait runs out
the same way.  The test reads the status back through the C ABI, checks that
reading clears it, and then runs the regular library on the same workspace in
the same process: the aborting CTAs re-armed the workspace's control block, the
context is still usable and the result matches the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

BSQ_ERR_TIMEOUT = 6
SITE_QUANT_BARRIER = 0x302


@pytest.fixture(scope="module")
def waittest_lib(bsq):
    from block_scaled_precision_packed_gb300 import build as B
    path = B.build_variant("waittest", ["BSQ_WAIT_LIMIT_NS=10000000ull", "BSQ_TEST_BARRIER_SKIP_LAST_CTA"])
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.bsq_quantize_mxfp6.restype = i32
    lib.bsq_quantize_mxfp6.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.bsq_get_device_error.restype = i32
    lib.bsq_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    return lib


def test_grid_barrier_timeout_is_reported_and_the_context_stays_usable(bsq, waittest_lib):
    M, K = 1024, 4096                                   # the one-pass (grid barrier) path
    x = S.normal_bf16((M, K), 0.02, 0xB5A0, outlier_frac=0.01)
    xd = dev_tensor(x)
    codes = torch.empty((M, 3 * K // 4), dtype=torch.uint8, device="cuda")
    scales = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device="cuda")
    sg = torch.empty(1, dtype=torch.float32, device="cuda")
    wsb = bsq.quantize_workspace_bytes(M, K)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    st = waittest_lib.bsq_quantize_mxfp6(xd.data_ptr(), M, K, bsq.E3M2, codes.data_ptr(), scales.data_ptr(),
                                         sg.data_ptr(), ws.data_ptr(), wsb, stream)
    assert st == 0, "the launch itself succeeds"
    code = ctypes.c_uint32(0)
    st = waittest_lib.bsq_get_device_error(stream, ctypes.byref(code))
    assert (st, code.value) == (BSQ_ERR_TIMEOUT, SITE_QUANT_BARRIER)
    st = waittest_lib.bsq_get_device_error(stream, ctypes.byref(code))
    assert (st, code.value) == (0, 0), "reading the word clears it"

    # the regular library, same process, same workspace: one-pass again, exact
    bsq.reset_launch_counts()
    bsq.quantize_mxfp6_(xd, bsq.E3M2, codes, scales, sg, ws)
    torch.cuda.synchronize()
    assert bsq.launch_count("quant_mx") == 1 and bsq.launch_count("amax") == 0
    oc, os_, og = O.quantize_mx(x, O.E3M2)
    assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
    assert np.array_equal(host_bytes(scales), os_)
    assert np.float32(sg.item()) == np.float32(og)
    assert bsq.device_error() == (0, 0)
