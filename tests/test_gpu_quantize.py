"""GPU quantizers against the oracle: codes, block scales (whole swizzled
buffer, padding included) and s_global bit for bit, on all three launch
shapes -- the single cluster launch for small tensors, the one-pass
cooperative launch for tensors that fit the GPU's shared memory (including a
grid with idle CTAs, (600, 128)), and amax pass + encode pass beyond that
((4480, 4096), and nvfp4 rows that are not a whole number of 32-value slots)
-- on ragged shapes and on the degenerate inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from block_scaled_precision_packed_gb300 import synthetic as S
from tests.parity import dev_tensor, host_bytes

pytestmark = pytest.mark.gpu

MX = [("e3m2", O.E3M2), ("e2m3", O.E2M3), ("e4m3", O.E4M3)]
SHAPES = [(1, 32), (3, 96), (16, 4096), (130, 1056), (200, 2048), (257, 4128), (1100, 1024), (600, 128),
          (4480, 4096)]


def fixture(M, K, seed, std=0.02):
    x = S.normal_bf16((M, K), std, seed, outlier_frac=0.01)
    flat = x.ravel()
    if flat.size >= 64:
        x[0, :32] = 0                 # an all-zero block
        flat[40] = 0x8000             # -0
        flat[41] = 0x8001             # tiny negative (bf16 subnormal)
        flat[42] = 0x0001             # tiny positive
    return x


@pytest.mark.parametrize("name,fmt", MX)
@pytest.mark.parametrize("M,K", SHAPES)
def test_quantize_mx_bit_exact(bsq, name, fmt, M, K):
    x = fixture(M, K, 100 + M + K)
    codes, scales, g = bsq.quantize_mxfp6(dev_tensor(x), name)
    torch.cuda.synchronize()
    oc, os_, og = O.quantize_mx(x, fmt)
    assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
    assert np.array_equal(host_bytes(scales), os_)
    assert np.float32(g.item()) == np.float32(og)


@pytest.mark.parametrize("M,K", SHAPES + [(5, 16), (7, 48), (5000, 48)])
def test_quantize_nvfp4_bit_exact(bsq, M, K):
    x = fixture(M, K, 300 + M + K, std=1.0)
    codes, scales, g = bsq.quantize_nvfp4(dev_tensor(x))
    torch.cuda.synchronize()
    oc, os_, og = O.quantize_nvfp4(x)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), oc)
    assert np.array_equal(host_bytes(scales), os_)
    assert np.float32(g.item()) == np.float32(og)


@pytest.mark.parametrize("kind", ["zeros", "negzeros", "single", "tiny", "huge"])
def test_quantize_degenerate_inputs(bsq, kind):
    M, K = 4, 128
    x = np.zeros((M, K), dtype=np.uint16)
    if kind == "negzeros":
        x[:] = 0x8000
    elif kind == "single":
        x[2, 77] = 0xC2C8            # -100
    elif kind == "tiny":
        x[:] = S.normal_bf16((M, K), 1e-30, 7)
    elif kind == "huge":
        x[:] = S.normal_bf16((M, K), 1e30, 8)
    for name, fmt in MX:
        c, s, g = bsq.quantize_mxfp6(dev_tensor(x), name)
        oc, os_, og = O.quantize_mx(x, fmt)
        assert np.array_equal(host_bytes(c).reshape(oc.shape), oc), name
        assert np.array_equal(host_bytes(s), os_), name
        assert np.float32(g.item()) == np.float32(og)
    c, s, g = bsq.quantize_nvfp4(dev_tensor(x))
    oc, os_, og = O.quantize_nvfp4(x)
    assert np.array_equal(c.cpu().numpy().view(np.uint32), oc)
    assert np.array_equal(host_bytes(s), os_)
    assert np.float32(g.item()) == np.float32(og)


def test_sign_of_zero_reading(bsq):
    """Negative values that round to zero keep the sign bit (the reading for
    the sign of zero): the hardware conversion and the oracle agree."""
    M, K = 1, 32
    x = np.zeros((M, K), dtype=np.uint16)
    x[0, 0] = 0x4480                 # 1024: sets the block scale
    x[0, 1] = 0x8001                 # a negative that underflows to zero
    x[0, 2] = 0x8000                 # -0
    for name, fmt in MX:
        c, s, g = bsq.quantize_mxfp6(dev_tensor(x), name)
        oc, _, _ = O.quantize_mx(x, fmt)
        assert np.array_equal(host_bytes(c).reshape(oc.shape), oc), name
    c, s, g = bsq.quantize_nvfp4(dev_tensor(x))
    oc, _, _ = O.quantize_nvfp4(x)
    assert np.array_equal(c.cpu().numpy().view(np.uint32), oc)
    assert (oc[0, 0] >> 4) & 0xF == 0x8 and (oc[0, 0] >> 8) & 0xF == 0x8


@pytest.mark.parametrize("name,fmt", MX)
def test_dequant_matches_oracle(bsq, name, fmt):
    M, K = 130, 256
    x = fixture(M, K, 5)
    c, s, g = bsq.quantize_mxfp6(dev_tensor(x), name)
    out = torch.empty((M, K), dtype=torch.float32, device="cuda")
    bsq.dequant_mxfp6_(c, bsq.FMT_IDS[name], s, g, out, M, K)
    want = O.dequant_mx(host_bytes(c).reshape(M, -1), fmt, host_bytes(s), float(g.item()), M, K)
    assert np.array_equal(out.cpu().numpy(), want.astype(np.float32))
    w, sw, gw = bsq.quantize_nvfp4(dev_tensor(x))
    out2 = torch.empty((M, K), dtype=torch.float32, device="cuda")
    bsq.dequant_nvfp4_(w, sw, gw, out2, M, K)
    want2 = O.dequant_nvfp4(w.cpu().numpy().view(np.uint32), host_bytes(sw), float(gw.item()), M, K)
    assert np.array_equal(out2.cpu().numpy(), want2.astype(np.float32))


# ---- batched quantizers: each tensor exactly as its own call would be ----
BATCH = [(128, 4096), (3, 96), (1100, 1024), (257, 4128), (16, 64)]


def _mx_outputs(M, K, name):
    codes = torch.empty((M, K if name == "e4m3" else 3 * K // 4), dtype=torch.uint8, device="cuda")
    scales = torch.empty(O.scale_bytes(M, K // 32), dtype=torch.uint8, device="cuda")
    return codes, scales, torch.empty(1, dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("name,fmt", MX)
def test_quantize_mx_batch_bit_exact(bsq, name, fmt):
    xs = [fixture(M, K, 500 + i) for i, (M, K) in enumerate(BATCH)]
    xs[1][:] = 0                                   # an all-zero tensor in the batch: gs = 0
    outs = [_mx_outputs(M, K, name) for M, K in BATCH]
    ws = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda")
    bsq.reset_launch_counts()
    bsq.quantize_mxfp6_batch_([(dev_tensor(x),) + o for x, o in zip(xs, outs)], bsq.FMT_IDS[name], ws)
    torch.cuda.synchronize()
    assert bsq.launch_count("quant_mx") == 1 and bsq.launch_count("amax") == 0   # one launch for all
    for x, (codes, scales, g) in zip(xs, outs):
        oc, os_, og = O.quantize_mx(x, fmt)
        assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
        assert np.array_equal(host_bytes(scales), os_)
        assert np.float32(g.item()) == np.float32(og)


@pytest.mark.parametrize("name,fmt", MX)
def test_quantize_mx_batch_w6a6_size_bit_exact(bsq, name, fmt):
    """The W6A6 step's batch at full size -- A [128, 4096] and W [4096, 4096]
    (N(0, 0.02), 1% outliers x20) in one one-pass launch, rows a whole number of
    4-block groups, so whole warps store their codes through shared memory --
    every code, scale and global factor bit-exact."""
    shapes = [(128, 4096), (4096, 4096)]
    xs = [S.normal_bf16(sh, 0.02, 700 + i, outlier_frac=0.01, outlier_mult=20.0) for i, sh in enumerate(shapes)]
    outs = [_mx_outputs(M, K, name) for M, K in shapes]
    ws = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda")
    bsq.reset_launch_counts()
    bsq.quantize_mxfp6_batch_([(dev_tensor(x),) + o for x, o in zip(xs, outs)], bsq.FMT_IDS[name], ws)
    torch.cuda.synchronize()
    assert bsq.launch_count("quant_mx") == 1 and bsq.launch_count("amax") == 0
    for x, (codes, scales, g) in zip(xs, outs):
        oc, os_, og = O.quantize_mx(x, fmt)
        assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
        assert np.array_equal(host_bytes(scales), os_)
        assert np.float32(g.item()) == np.float32(og)


def test_quantize_nvfp4_batch_bit_exact(bsq):
    shapes = BATCH + [(7, 4096)]
    xs = [fixture(M, K, 600 + i, std=1.0) for i, (M, K) in enumerate(shapes)]
    outs = [(torch.empty((M, K // 8), dtype=torch.int32, device="cuda"),
             torch.empty(O.scale_bytes(M, K // 16), dtype=torch.uint8, device="cuda"),
             torch.empty(1, dtype=torch.float32, device="cuda")) for M, K in shapes]
    ws = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda")
    bsq.quantize_nvfp4_batch_([(dev_tensor(x),) + o for x, o in zip(xs, outs)], ws)
    torch.cuda.synchronize()
    for x, (codes, scales, g) in zip(xs, outs):
        oc, os_, og = O.quantize_nvfp4(x)
        assert np.array_equal(codes.cpu().numpy().view(np.uint32), oc)
        assert np.array_equal(host_bytes(scales), os_)
        assert np.float32(g.item()) == np.float32(og)


def test_quantize_batch_beyond_one_launch_runs_one_by_one(bsq):
    """Two tensors whose slices do not fit the GPU's shared memory together: the
    call falls back to one quantizer per tensor, with the same results."""
    shapes = [(4096, 4096), (1024, 4096)]
    xs = [fixture(M, K, 700 + i) for i, (M, K) in enumerate(shapes)]
    outs = [_mx_outputs(M, K, "e2m3") for M, K in shapes]
    ws = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda")
    bsq.reset_launch_counts()
    bsq.quantize_mxfp6_batch_([(dev_tensor(x),) + o for x, o in zip(xs, outs)], bsq.FMT_IDS["e2m3"], ws)
    torch.cuda.synchronize()
    assert bsq.launch_count("quant_mx") == 2
    for x, (codes, scales, g) in zip(xs, outs):
        oc, os_, og = O.quantize_mx(x, O.E2M3)
        assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
        assert np.array_equal(host_bytes(scales), os_)
        assert np.float32(g.item()) == np.float32(og)


def test_quantize_batch_bad_arguments(bsq):
    import ctypes
    L = bsq.load()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    c, s, g = _mx_outputs(4, 64, "e3m2")
    ws = torch.empty(bsq.quantize_batch_workspace_bytes(), dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    wsp, wsb = ctypes.c_void_p(ws.data_ptr()), ws.numel()
    bsq.reset_launch_counts()
    one = bsq._qtensors([(x, c, s, g)])
    assert L.bsq_quantize_mxfp6_batch(ctypes.cast(one, ctypes.c_void_p), 0, 0, wsp, wsb, st) == 1       # n = 0
    nine = bsq._qtensors([(x, c, s, g)] * 9)
    assert L.bsq_quantize_mxfp6_batch(ctypes.cast(nine, ctypes.c_void_p), 9, 0, wsp, wsb, st) == 1      # n > 8
    bad = bsq._qtensors([(x, c, s, g)])
    bad[0].K = 48
    assert L.bsq_quantize_mxfp6_batch(ctypes.cast(bad, ctypes.c_void_p), 1, 0, wsp, wsb, st) == 1       # K % 32
    assert L.bsq_quantize_mxfp6_batch(ctypes.cast(one, ctypes.c_void_p), 1, 0, wsp, 64, st) == 4        # workspace
    assert sum(bsq.launch_count(k) for k in bsq.KERNEL_IDS) == 0


@pytest.mark.parametrize("fill", ["zeros", "ones", "random"])
def test_one_pass_accepts_any_workspace_contents(bsq, fill):
    """The one-pass path keeps its grid-wait control block in the workspace with
    no memset per call: a fresh workspace of any contents is initialized by the
    first call, and the next calls on the same workspace see it ready."""
    M, K = 512, 2048
    wsb = bsq.quantize_workspace_bytes(M, K)
    if fill == "zeros":
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    elif fill == "ones":
        ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device="cuda")
    else:
        ws = torch.from_numpy(np.random.default_rng(5).integers(0, 256, wsb, dtype=np.uint8)).cuda()
    for call in range(3):
        x = fixture(M, K, 800 + call)
        codes, scales, g = _mx_outputs(M, K, "e3m2")
        bsq.reset_launch_counts()
        bsq.quantize_mxfp6_(dev_tensor(x), O.E3M2, codes, scales, g, ws)
        torch.cuda.synchronize()
        assert bsq.launch_count("quant_mx") == 1 and bsq.launch_count("amax") == 0   # the one-pass path
        oc, os_, og = O.quantize_mx(x, O.E3M2)
        assert np.array_equal(host_bytes(codes).reshape(oc.shape), oc)
        assert np.array_equal(host_bytes(scales), os_)
        assert np.float32(g.item()) == np.float32(og)


@pytest.mark.parametrize("fmt", [0, 1])                       # e3m2, e2m3
@pytest.mark.parametrize("M,K", [(16, 4096), (3, 96), (1000, 2048), (129, 4160)])
def test_quantize_byte_containers_bit_exact(bsq, fmt, M, K):
    """bsq_quantize_mxfp6_containers: one fp6 code per byte, bit-identical to the
    oracle and to the unpacked codes of the packed quantizer."""
    x = S.normal_bf16((M, K), 0.02, 501 + M + K, outlier_frac=0.01)
    xd = dev_tensor(x)
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty(bsq.scale_bytes(M, K // 32), dtype=torch.uint8, device="cuda")
    sg = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(16, bsq.quantize_workspace_bytes(M, K)), dtype=torch.uint8, device="cuda")
    bsq.quantize_mxfp6_containers_(xd, fmt, codes, scales, sg, ws)
    torch.cuda.synchronize()
    oc, osc, og = O.quantize_mx_containers(x, (O.E3M2, O.E2M3)[fmt])
    assert np.array_equal(host_bytes(codes), oc)
    assert np.array_equal(host_bytes(scales), osc)
    assert float(sg.item()) == og
    pc, _, _ = bsq.quantize_mxfp6(xd.view(torch.bfloat16), ("e3m2", "e2m3")[fmt])
    torch.cuda.synchronize()
    assert np.array_equal(O.unpack_fp6(host_bytes(pc), M * K), host_bytes(codes).ravel())
