"""Seeded synthetic inputs, shared by the tests and the benchmark.

This module draws the workloads' raw inputs and nothing else: bf16 tensors
from a normal distribution (with an optional outlier mix), uniformly random
packed e2m1 words, and block-scale bytes drawn from a stated set.  It holds
none of the method's arithmetic (no quantizer, no decoder, no product); the
GPU library and the CPU oracle both consume exactly the bytes it returns.

Recipes (each workload's seed is fixed below; sub-tensors use seed+1, +2, ...):
  * ``normal_bf16``: numpy PCG64 standard normals * std, in f32, rounded to
    bf16 by torch's round-to-nearest-even cast.  "1% outliers x20" multiplies
    each sample independently, with probability 0.01, by 20.
  * ``random_words``: uniformly random u32 words, i.e. eight independent
    uniform e2m1 codes per word (all 16 codes, both zeros included).
  * ``choice_bytes``: bytes drawn uniformly from a given list of codes.
"""
from __future__ import annotations

import numpy as np
import torch

# The ue4m3 codes of the powers of two 2^-4 .. 2^4 (sign 0, exponent field
# e + 7, mantissa 0): the block scales of the one-row nvfp4 workload.
UE4M3_POW2_M4_TO_P4 = [0x18, 0x20, 0x28, 0x30, 0x38, 0x40, 0x48, 0x50, 0x58]

SEED_BASE = 0xB500


def generator(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round an f32 array to bf16 (torch's RNE cast) and return the raw bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(shape, std: float, seed: int, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    g = generator(seed)
    v = g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    if outlier_frac > 0.0:
        hit = g.random(size=shape) < outlier_frac
        v = np.where(hit, v * np.float32(outlier_mult), v).astype(np.float32)
    return f32_to_bf16_bits(v)


def random_words(shape, seed: int) -> np.ndarray:
    g = generator(seed)
    return g.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)


def random_bytes(n: int, seed: int, lo: int = 0, hi: int = 256) -> np.ndarray:
    g = generator(seed)
    return g.integers(lo, hi, size=n, dtype=np.int64).astype(np.uint8)


def choice_bytes(n: int, seed: int, codes) -> np.ndarray:
    g = generator(seed)
    codes = np.asarray(codes, dtype=np.uint8)
    return codes[g.integers(0, codes.size, size=n)]


# The five workloads, by what they are.  Shapes follow Y[M,N] = X[M,K] W[N,K]^T.
WORKLOADS = {
    "nvfp4_gemv_1x256x256": dict(seed=SEED_BASE + 1, M=1, N=256, K=256, x_std=1.0, g_w=0.5),
    "mxfp6_e3m2_w6a6_128x4096x4096": dict(seed=SEED_BASE + 2, M=128, N=4096, K=4096,
                                          a_std=0.02, w_std=0.02, outlier_frac=0.01,
                                          outlier_mult=20.0),
    "nvfp4_decode_gemv_Mx28672x8192": dict(seed=SEED_BASE + 3, Ms=(1, 8, 32), N=28672, K=8192,
                                           x_std=1.0, w_std=0.02),
    "nvfp4_prefill_gemm_8192": dict(seed=SEED_BASE + 4, M=8192, N=8192, K=8192,
                                    a_std=1.0, w_std=0.02),
    "w6a8_e4m3xe2m3_4096x14336x4096": dict(seed=SEED_BASE + 5, M=4096, N=14336, K=4096,
                                           a_std=1.0, w_std=0.02, small_Ms=(1, 4, 16)),
}
