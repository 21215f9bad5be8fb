"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (the acceptance bar of the path):
  * quantizer codes, scales, packed bytes and s_global: bit-exact;
  * fp32 products: |got - y| <= 1e-5 * S with S = |gA gW| sum_k |a_k w_k|;
  * bf16 products: within 1 bf16 ulp of round_bf16(y).  Only an output whose
    exact value is so small that the fp32 accumulation bound alone exceeds half
    a bf16 ulp of it -- |y| < 2^8 * 1e-5 * S, heavy cancellation -- may instead
    pass with |got - y| <= 1e-5 * S + ulp(got)/2 (the fp32 bound plus the final
    rounding); every other output is held to the 1-ulp rule.
"""
import numpy as np
import torch

import oracle as O

REL = 1e-5


def dev_tensor(a: np.ndarray, device="cuda"):
    """numpy -> torch CUDA tensor with the same bytes (uint16 -> int16, uint32 -> int32)."""
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}.get(a.dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a).to(device)


def host_bytes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_products(got: torch.Tensor, want: np.ndarray, S: np.ndarray, what: str = ""):
    """got: device/host tensor of fp32 or bf16 outputs (flattened order of want)."""
    want = np.asarray(want, dtype=np.float64).ravel()
    S = np.asarray(S, dtype=np.float64).ravel()
    if got.dtype == torch.bfloat16:
        bits = got.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).ravel()
        rb = O.double_to_bf16_array(want)
        ok = np.abs(bf16_ordinal(bits) - bf16_ordinal(rb)) <= 1
        val = bf16_value(bits)
        ulp = np.abs(bf16_value((bits & 0x7FFF) | 1) - bf16_value(bits & 0x7FFF)) + 2.0 ** -133
        cancelled = np.abs(want) < 256.0 * REL * S
        ok |= cancelled & (np.abs(val - want) <= REL * S + ulp / 2)
    else:
        val = got.detach().cpu().contiguous().numpy().astype(np.float64).ravel()
        ok = np.abs(val - want) <= REL * S + 1e-300
    ok &= np.isfinite(val)
    if not ok.all():
        i = np.flatnonzero(~ok)[:8]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outputs out of tolerance; "
                             f"first idx {i.tolist()} got {val[i].tolist()} want {want[i].tolist()} S {S[i].tolist()}")


def boundary_index(R, tile=128):
    """Every index on either side of a tile boundary: 0, 127, 128, 255, 256, ...
    up to R - 1."""
    b = {0, R - 1}
    for t in range(tile, R, tile):
        b.update((t - 1, t))
    return np.array(sorted(b), dtype=np.int64)


def products_by_blocks(dec_a, dec_w, g):
    """y = g * dec_a @ dec_w^T and S = |g| * |dec_a| @ |dec_w|^T in float64 (a
    library matmul over operands the oracle decoded exactly)."""
    return g * (dec_a @ dec_w.T), abs(g) * (np.abs(dec_a) @ np.abs(dec_w).T)


def sample_pairs(M, N, n, seed, edges=True):
    """A fixed seeded sample of (m, n) output positions plus the tile-edge rows/cols."""
    g = np.random.default_rng(seed)
    mi = g.integers(0, M, n)
    ni = g.integers(0, N, n)
    if edges:
        em = sorted({0, M - 1, min(127, M - 1), min(128, M - 1), M // 2})
        en = sorted({0, N - 1, min(127, N - 1), min(128, N - 1), min(255, N - 1), min(256, N - 1), N // 2})
        mm, nn = np.meshgrid(em, en, indexing="ij")
        mi = np.concatenate([mi, mm.ravel()])
        ni = np.concatenate([ni, nn.ravel()])
    return mi.astype(np.int64), ni.astype(np.int64)
