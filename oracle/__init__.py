"""CPU oracle for the block-scaled packed-precision path -- TEST INFRASTRUCTURE.

A thin ctypes/numpy wrapper around ``bsq_oracle.c``: the slow, plain
restatement of what the GPU library computes (decoders from the formats'
closed forms, the nearest-code encoder, the MX and nvfp4 quantizers step by
step in f32, and the products summed in double).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs import this package.  The CUDA
library never imports, links or calls it, and it shares no code with it.

Parity status: everything here is pinned by ``tests/test_oracle_*.py`` except
the nvfp4 quantizer's recipe, which the pages do not give (pinned by
invariants only; "parity unpinned" as to the recipe itself).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# format ids shared by the oracle's C entry points
E3M2, E2M3, E4M3, E2M1, UE4M3 = 0, 1, 2, 3, 4
MX_FMTS = {"e3m2": E3M2, "e2m3": E2M3, "e4m3": E4M3}

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, plain C, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L):
    d, u, i, i64, f = ctypes.c_double, ctypes.c_uint, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    p = ctypes.c_void_p
    sig = {
        "bsqo_decode_e3m2": (d, [u]), "bsqo_decode_e2m3": (d, [u]), "bsqo_decode_e2m1": (d, [u]),
        "bsqo_decode_e4m3": (d, [u]), "bsqo_decode_ue4m3": (d, [u]), "bsqo_decode_ue8m0": (d, [u]),
        "bsqo_decode": (d, [i, u]), "bsqo_encode": (u, [i, f]),
        "bsqo_pack_fp6": (None, [p, i64, p]), "bsqo_unpack_fp6": (None, [p, i64, p]),
        "bsqo_swz_offset": (i64, [i64, i64, i64]), "bsqo_scale_bytes": (i64, [i64, i64]),
        "bsqo_gs_numerator": (f, [i]),
        "bsqo_ue8m0_from_block_max": (u, [f, f, f]), "bsqo_ue8m0_output_scale": (f, [u, f]),
        "bsqo_quantize_mx": (i, [p, i64, i64, i, p, p, p]),
        "bsqo_quantize_mx_rows": (i, [p, i64, i64, i, p, i64, p, p, p]),
        "bsqo_quantize_nvfp4": (i, [p, i64, i64, p, p, p]),
        "bsqo_quantize_nvfp4_rows": (i, [p, i64, i64, p, i64, p, p, p]),
        "bsqo_dequant_mx": (i, [p, i, p, d, i64, i64, p]),
        "bsqo_dequant_nvfp4": (i, [p, p, d, i64, i64, p]),
        "bsqo_gemm_nvfp4_at": (i, [p, p, d, p, p, d, i64, p, p, i64, p, p, i]),
        "bsqo_gemm_mx_at": (i, [p, i, p, d, p, i, p, d, i64, p, p, i64, p, p, i]),
        "bsqo_gemv_nvfp4_at": (i, [p, p, p, d, i64, p, p, i64, p, p, i]),
        "bsqo_gemv_mx_at": (i, [p, p, i, p, d, i64, p, p, i64, p, p, i]),
        "bsqo_activate": (i, [p, i64, i64, i, p]),
        "bsqo_quantize_mx_containers": (i, [p, i64, i64, i, p, p, p]),
        "bsqo_quantize_grouped_mx": (i, [p, i64, i64, i64, p, p, i, p, p, p]),
        "bsqo_quantize_mx_act": (i, [p, i64, i64, i, i, p, p, p, p]),
        "bsqo_f32_to_bf16": (ctypes.c_uint16, [f]),
        "bsqo_double_to_bf16": (ctypes.c_uint16, [d]),
        "bsqo_double_to_bf16_n": (None, [p, i64, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


# ---------------------------------------------------------------- scalars ----
def decode(fmt: int, code: int) -> float:
    return lib().bsqo_decode(fmt, code)


def decode_ue8m0(code: int) -> float:
    return lib().bsqo_decode_ue8m0(code)


def encode(fmt: int, v: float) -> int:
    return lib().bsqo_encode(fmt, float(v))


def swz_offset(row: int, block: int, n_blocks: int) -> int:
    return lib().bsqo_swz_offset(row, block, n_blocks)


def scale_bytes(rows: int, n_blocks: int) -> int:
    return lib().bsqo_scale_bytes(rows, n_blocks)


def gs_numerator(fmt: int) -> float:
    return lib().bsqo_gs_numerator(fmt)


def ue8m0_from_block_max(amax_b: float, gs: float, fmax: float) -> int:
    return lib().bsqo_ue8m0_from_block_max(amax_b, gs, fmax)


def ue8m0_output_scale(ue: int, gs: float) -> float:
    return lib().bsqo_ue8m0_output_scale(ue, gs)


def f32_to_bf16(v: float) -> int:
    return lib().bsqo_f32_to_bf16(v)


def double_to_bf16(v: float) -> int:
    return lib().bsqo_double_to_bf16(v)


def double_to_bf16_array(y: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(y, dtype=np.float64).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    lib().bsqo_double_to_bf16_n(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(y))


# ---------------------------------------------------------------- packing ----
def pack_fp6(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    n = codes.size
    if n % 4:
        raise ValueError("fp6 packing needs a multiple of 4 codes")
    out = np.empty(3 * n // 4, dtype=np.uint8)
    lib().bsqo_pack_fp6(_ptr(codes), n, _ptr(out))
    return out


def unpack_fp6(packed: np.ndarray, n: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(n, dtype=np.uint8)
    lib().bsqo_unpack_fp6(_ptr(packed), n, _ptr(out))
    return out


# ------------------------------------------------------------- quantizers ----
def quantize_mx(x_bf16: np.ndarray, fmt: int):
    """bf16 bits [M, K] -> (codes, swizzled UE8M0 scales, s_global)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    row_bytes = K if fmt == E4M3 else 3 * K // 4
    codes = np.empty((M, row_bytes), dtype=np.uint8)
    scales = np.empty(scale_bytes(M, K // 32), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().bsqo_quantize_mx(_ptr(x), M, K, fmt, _ptr(codes), _ptr(scales), _ptr(g)), "quantize_mx")
    return codes, scales, float(g[0])


def quantize_grouped_mx(x_bf16: np.ndarray, row_counts, gs, fmt: int):
    """Grouped MX quantizer (b12x fp6.py quantize_grouped_mxfp6_torch): x [G, R, C]
    bf16, per-group row counts and global scales -> (codes [G, R, row_bytes]
    group-major, scales [G, pad128(R)*pad4(C/32)], s_global [G] = 1/gs)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    G, R, C = x.shape
    rc = np.ascontiguousarray(row_counts, dtype=np.int64)
    g32 = np.ascontiguousarray(gs, dtype=np.float32)
    row_bytes = C if fmt == E4M3 else 3 * C // 4
    codes = np.empty((G, R, row_bytes), dtype=np.uint8)
    scales = np.empty((G, scale_bytes(R, C // 32)), dtype=np.uint8)
    sg = np.empty(G, dtype=np.float32)
    _check(lib().bsqo_quantize_grouped_mx(_ptr(x), G, R, C, _ptr(rc), _ptr(g32), fmt, _ptr(codes), _ptr(scales),
                                          _ptr(sg)), "quantize_grouped_mx")
    return codes, scales, sg


def gemm_grouped_mx(A, fa, sA, gA, W, fw, sW, gW, row_counts, K):
    """Grouped product: for each group g, the plain product of its first
    row_counts[g] A rows with its W: Y [G, R, N] and S (rows past the count 0)."""
    G, R = A.shape[0], A.shape[1]
    N = W.shape[1]
    y = np.zeros((G, R, N))
    S = np.zeros((G, R, N))
    for g in range(G):
        rc = int(row_counts[g])
        if rc == 0:
            continue
        want, s = gemm_mx(np.ascontiguousarray(A[g, :rc]), fa, np.ascontiguousarray(sA[g]), float(gA[g]),
                          np.ascontiguousarray(W[g]), fw, np.ascontiguousarray(sW[g]), float(gW[g]), rc, N, K)
        y[g, :rc] = np.asarray(want).reshape(rc, N)
        S[g, :rc] = np.asarray(s).reshape(rc, N)
    return y, S


def quantize_mx_containers(x_bf16: np.ndarray, fmt: int):
    """The MX quantizer with fp6 codes one per byte: (codes [M, K], scales, s_global)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    codes = np.empty((M, K), dtype=np.uint8)
    scales = np.empty(scale_bytes(M, K // 32), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().bsqo_quantize_mx_containers(_ptr(x), M, K, fmt, _ptr(codes), _ptr(scales), _ptr(g)),
           "quantize_mx_containers")
    return codes, scales, float(g[0])


ACT_RELU2, ACT_SILU_MUL = 1, 2


def activate(x_bf16: np.ndarray, act: int) -> np.ndarray:
    """The activation of the fused quantizers, rounded to bf16: ReLU^2 of x [M, K],
    or SiLU(gate) * up of x [M, 2K] (gate = columns [0, K), up = [K, 2K))."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, Kin = x.shape
    K = Kin if act == ACT_RELU2 else Kin // 2
    out = np.empty((M, K), dtype=np.uint16)
    _check(lib().bsqo_activate(_ptr(x), M, K, act, _ptr(out)), "activate")
    return out


def quantize_mx_act(x_bf16: np.ndarray, act: int, fmt: int):
    """Fused activation + MX quantizer: (codes, swizzled scales, s_global, activated bf16)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, Kin = x.shape
    K = Kin if act == ACT_RELU2 else Kin // 2
    row_bytes = K if fmt == E4M3 else 3 * K // 4
    codes = np.empty((M, row_bytes), dtype=np.uint8)
    scales = np.empty(scale_bytes(M, K // 32), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    a = np.empty((M, K), dtype=np.uint16)
    _check(lib().bsqo_quantize_mx_act(_ptr(x), M, K, act, fmt, _ptr(codes), _ptr(scales), _ptr(g), _ptr(a)),
           "quantize_mx_act")
    return codes, scales, float(g[0]), a


def quantize_mx_rows(x_bf16: np.ndarray, fmt: int, rows):
    """The MX quantizer on a row subset: (codes [n, row_bytes], ue [n, K/32], s_global)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    row_bytes = K if fmt == E4M3 else 3 * K // 4
    codes = np.empty((rows.size, row_bytes), dtype=np.uint8)
    ue = np.empty((rows.size, K // 32), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().bsqo_quantize_mx_rows(_ptr(x), M, K, fmt, _ptr(rows), rows.size,
                                       _ptr(codes), _ptr(ue), _ptr(g)), "quantize_mx_rows")
    return codes, ue, float(g[0])


def quantize_nvfp4(x_bf16: np.ndarray):
    """bf16 bits [M, K] -> (u32 words [M, K/8], swizzled ue4m3 scales, s_global)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    codes = np.empty((M, K // 8), dtype=np.uint32)
    scales = np.empty(scale_bytes(M, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().bsqo_quantize_nvfp4(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(g)), "quantize_nvfp4")
    return codes, scales, float(g[0])


def quantize_nvfp4_rows(x_bf16: np.ndarray, rows):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    codes = np.empty((rows.size, K // 8), dtype=np.uint32)
    sb = np.empty((rows.size, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _check(lib().bsqo_quantize_nvfp4_rows(_ptr(x), M, K, _ptr(rows), rows.size,
                                          _ptr(codes), _ptr(sb), _ptr(g)), "quantize_nvfp4_rows")
    return codes, sb, float(g[0])


# ---------------------------------------------------------------- dequant ----
def dequant_mx(codes: np.ndarray, fmt: int, scales: np.ndarray, g: float, R: int, K: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((R, K), dtype=np.float64)
    _check(lib().bsqo_dequant_mx(_ptr(codes), fmt, _ptr(scales), float(g), R, K, _ptr(out)), "dequant_mx")
    return out


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, g: float, R: int, K: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((R, K), dtype=np.float64)
    _check(lib().bsqo_dequant_nvfp4(_ptr(codes), _ptr(scales), float(g), R, K, _ptr(out)), "dequant_nvfp4")
    return out


# --------------------------------------------------------------- products ----
def _pairs(M, N, mi, ni):
    if mi is None:
        mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    mi = np.ascontiguousarray(np.ravel(mi), dtype=np.int64)
    ni = np.ascontiguousarray(np.ravel(ni), dtype=np.int64)
    return mi, ni


def gemm_nvfp4(A, sA, gA, W, sW, gW, M, N, K, mi=None, ni=None, threads=0):
    """Y[m,n] = gA*gW*sum_k decA*decW at the (mi, ni) pairs (all pairs if None).
    Returns (y, S) with S = |gA*gW|*sum_k |decA*decW|."""
    mi, ni = _pairs(M, N, mi, ni)
    A = np.ascontiguousarray(A, dtype=np.uint32); W = np.ascontiguousarray(W, dtype=np.uint32)
    sA = np.ascontiguousarray(sA, dtype=np.uint8); sW = np.ascontiguousarray(sW, dtype=np.uint8)
    y = np.empty(mi.size); s = np.empty(mi.size)
    _check(lib().bsqo_gemm_nvfp4_at(_ptr(A), _ptr(sA), float(gA), _ptr(W), _ptr(sW), float(gW), K,
                                    _ptr(mi), _ptr(ni), mi.size, _ptr(y), _ptr(s), threads), "gemm_nvfp4")
    return y, s


def gemm_mx(A, fa, sA, gA, W, fw, sW, gW, M, N, K, mi=None, ni=None, threads=0):
    mi, ni = _pairs(M, N, mi, ni)
    A = np.ascontiguousarray(A, dtype=np.uint8); W = np.ascontiguousarray(W, dtype=np.uint8)
    sA = np.ascontiguousarray(sA, dtype=np.uint8); sW = np.ascontiguousarray(sW, dtype=np.uint8)
    y = np.empty(mi.size); s = np.empty(mi.size)
    _check(lib().bsqo_gemm_mx_at(_ptr(A), fa, _ptr(sA), float(gA), _ptr(W), fw, _ptr(sW), float(gW), K,
                                 _ptr(mi), _ptr(ni), mi.size, _ptr(y), _ptr(s), threads), "gemm_mx")
    return y, s


def gemv_nvfp4(x, W, sW, gW, M, N, K, mi=None, ni=None, threads=0):
    mi, ni = _pairs(M, N, mi, ni)
    x = np.ascontiguousarray(x, dtype=np.uint16); W = np.ascontiguousarray(W, dtype=np.uint32)
    sW = np.ascontiguousarray(sW, dtype=np.uint8)
    y = np.empty(mi.size); s = np.empty(mi.size)
    _check(lib().bsqo_gemv_nvfp4_at(_ptr(x), _ptr(W), _ptr(sW), float(gW), K,
                                    _ptr(mi), _ptr(ni), mi.size, _ptr(y), _ptr(s), threads), "gemv_nvfp4")
    return y, s


def gemv_mx(x, W, fw, sW, gW, M, N, K, mi=None, ni=None, threads=0):
    mi, ni = _pairs(M, N, mi, ni)
    x = np.ascontiguousarray(x, dtype=np.uint16); W = np.ascontiguousarray(W, dtype=np.uint8)
    sW = np.ascontiguousarray(sW, dtype=np.uint8)
    y = np.empty(mi.size); s = np.empty(mi.size)
    _check(lib().bsqo_gemv_mx_at(_ptr(x), _ptr(W), fw, _ptr(sW), float(gW), K,
                                 _ptr(mi), _ptr(ni), mi.size, _ptr(y), _ptr(s), threads), "gemv_mx")
    return y, s
