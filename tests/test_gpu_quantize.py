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
