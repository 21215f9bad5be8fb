"""Thin ctypes binding of libbsq (include/bsq.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); each call passes their data pointers and the current stream.  A
missing or unloadable library raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbsq.so")

E3M2, E2M3, E4M3 = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1
FMT_IDS = {"e3m2": E3M2, "e2m3": E2M3, "e4m3": E4M3}

KERNEL_IDS = {"amax": 0, "quant_mx": 1, "quant_nvfp4": 2, "quant_small": 3, "gemm_nvfp4": 4,
              "gemm_mx": 5, "gemv_nvfp4": 6, "gemv_mx": 7, "dequant": 8}

MAX_BATCH = 8

_lib = None
_lock = threading.Lock()


class QTensor(ctypes.Structure):
    """bsq_qtensor: one tensor of a batched quantizer call."""
    _fields_ = [("x", ctypes.c_void_p), ("M", ctypes.c_int64), ("K", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("s_global", ctypes.c_void_p)]


class BsqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load(path: str | None = None):
    """Load libbsq.so (built by __graft_entry__.build / block_scaled_precision_packed_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libbsq.so not found at {p}; build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(p)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sigs = {
            "bsq_status_string": (ctypes.c_char_p, [i32]),
            "bsq_abi_version": (i32, []),
            "bsq_scale_bytes": (sz, [i64, i64]),
            "bsq_quantize_workspace_bytes": (sz, [i64, i64]),
            "bsq_quantize_mxfp6": (i32, [vp, i64, i64, i32, vp, vp, vp, vp, sz, vp]),
            "bsq_quantize_nvfp4": (i32, [vp, i64, i64, vp, vp, vp, vp, sz, vp]),
            "bsq_quantize_mxfp6_noalloc": (i32, [vp, i64, i64, i32, vp, vp, vp, vp]),
            "bsq_quantize_mxfp6_act": (i32, [vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
            "bsq_quantize_mxfp6_containers": (i32, [vp, i64, i64, i32, vp, vp, vp, vp, sz, vp]),
            "bsq_quantize_grouped_mxfp6": (i32, [vp, i64, i64, i64, vp, vp, i32, vp, vp, vp, vp]),
            "bsq_gemm_grouped_mxfp6": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, i32, i64, i64, i64, i64,
                                             vp]),
            "bsq_quantize_batch_workspace_bytes": (sz, []),
            "bsq_quantize_mxfp6_batch": (i32, [vp, i32, i32, vp, sz, vp]),
            "bsq_quantize_nvfp4_batch": (i32, [vp, i32, vp, sz, vp]),
            "bsq_gemm_nvfp4": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, vp]),
            "bsq_gemm_mxfp6": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, vp, i32, i64, i64, i64, vp]),
            "bsq_gemm_quant_a_workspace_bytes": (sz, []),
            "bsq_gemm_mxfp6_quant_a": (i32, [vp, i32, vp, i32, vp, vp, vp, i32, vp, i64, i64, i64, vp, sz, vp]),
            "bsq_gemv_nvfp4": (i32, [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp]),
            "bsq_gemv_mxfp6": (i32, [vp, vp, i32, vp, vp, vp, i32, i64, i64, i64, vp]),
            "bsq_dequant_nvfp4": (i32, [vp, vp, vp, vp, i64, i64, vp]),
            "bsq_dequant_mxfp6": (i32, [vp, i32, vp, vp, vp, i64, i64, vp]),
            "bsq_get_device_error": (i32, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
            "bsq_launch_count": (ctypes.c_uint64, [i32]),
            "bsq_reset_launch_counts": (None, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().bsq_status_string(status).decode()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise BsqError(fn, status)


def scale_bytes(rows: int, n_blocks: int) -> int:
    return load().bsq_scale_bytes(rows, n_blocks)


def quantize_workspace_bytes(M: int, K: int) -> int:
    return load().bsq_quantize_workspace_bytes(M, K)


# ------------------------------------------------------------- raw entry points
def quantize_mxfp6_(x, fmt, codes, scales, s_global, workspace=None, stream=None):
    M, K = x.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("bsq_quantize_mxfp6", load().bsq_quantize_mxfp6(
        _p(x), M, K, fmt, _p(codes), _p(scales), _p(s_global), _p(workspace), ws_bytes, _stream(stream)))


def quantize_mxfp6_noalloc_(x, fmt, codes, scales, s_global, stream=None):
    """The allocation-free quantizer entry point (no workspace argument)."""
    M, K = x.shape
    _check("bsq_quantize_mxfp6_noalloc", load().bsq_quantize_mxfp6_noalloc(
        _p(x), M, K, fmt, _p(codes), _p(scales), _p(s_global), _stream(stream)))


def quantize_grouped_mxfp6_(x, row_counts, gs, fmt, codes, scales, s_global, stream=None):
    """Grouped MX quantize: x [G, R, C] bf16, row_counts [G] int32, gs [G] float."""
    G, R, C = x.shape
    _check("bsq_quantize_grouped_mxfp6", load().bsq_quantize_grouped_mxfp6(
        _p(x), G, R, C, _p(row_counts), _p(gs), fmt, _p(codes), _p(scales), _p(s_global), _stream(stream)))


def gemm_grouped_mxfp6_(A, fa, sA, gA, W, fw, sW, gW, row_counts, Y, G, R, N, K, stream=None):
    """Grouped GEMM: Y [G, R, N] (fp32 or bf16) from grouped MX operands."""
    out = 1 if Y.dtype == torch.bfloat16 else 0
    _check("bsq_gemm_grouped_mxfp6", load().bsq_gemm_grouped_mxfp6(
        _p(A), fa, _p(sA), _p(gA), _p(W), fw, _p(sW), _p(gW), _p(row_counts), _p(Y), out, G, R, N, K,
        _stream(stream)))


def quantize_mxfp6_containers_(x, fmt, codes, scales, s_global, workspace=None, stream=None):
    """The MX quantizer with fp6 codes one per byte: codes [M, K]."""
    M, K = x.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("bsq_quantize_mxfp6_containers", load().bsq_quantize_mxfp6_containers(
        _p(x), M, K, fmt, _p(codes), _p(scales), _p(s_global), _p(workspace), ws_bytes, _stream(stream)))


ACT_RELU2, ACT_SILU_MUL = 1, 2


def quantize_mxfp6_act_(x, K, act, fmt, codes, scales, s_global, act_out=None, workspace=None, stream=None):
    """Fused activation + MX quantize: x [M, K] (ReLU^2) or [M, 2K] (SiLU(gate) * up)."""
    M = x.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("bsq_quantize_mxfp6_act", load().bsq_quantize_mxfp6_act(
        _p(x), M, K, act, fmt, _p(codes), _p(scales), _p(s_global), _p(act_out), _p(workspace), ws_bytes,
        _stream(stream)))


def quantize_nvfp4_(x, codes, scales, s_global, workspace=None, stream=None):
    M, K = x.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("bsq_quantize_nvfp4", load().bsq_quantize_nvfp4(
        _p(x), M, K, _p(codes), _p(scales), _p(s_global), _p(workspace), ws_bytes, _stream(stream)))


def quantize_batch_workspace_bytes() -> int:
    return load().bsq_quantize_batch_workspace_bytes()


def _qtensors(items):
    arr = (QTensor * len(items))()
    for i, (x, codes, scales, g) in enumerate(items):
        M, K = x.shape
        arr[i] = QTensor(x.data_ptr(), M, K, codes.data_ptr(), scales.data_ptr(), g.data_ptr())
    return arr


def quantize_mxfp6_batch_(items, fmt, workspace, stream=None):
    """items: [(x, codes, scales, s_global), ...] -- one launch for the batch."""
    arr = _qtensors(items)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("bsq_quantize_mxfp6_batch", load().bsq_quantize_mxfp6_batch(
        ctypes.cast(arr, ctypes.c_void_p), len(items), fmt, _p(workspace), ws_bytes, _stream(stream)))


def quantize_nvfp4_batch_(items, workspace, stream=None):
    arr = _qtensors(items)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("bsq_quantize_nvfp4_batch", load().bsq_quantize_nvfp4_batch(
        ctypes.cast(arr, ctypes.c_void_p), len(items), _p(workspace), ws_bytes, _stream(stream)))


def gemm_nvfp4_(A, sA, gA, W, sW, gW, Y, M, N, K, stream=None):
    out = OUT_BF16 if Y.dtype == torch.bfloat16 else OUT_F32
    _check("bsq_gemm_nvfp4", load().bsq_gemm_nvfp4(
        _p(A), _p(sA), _p(gA), _p(W), _p(sW), _p(gW), _p(Y), out, M, N, K, _stream(stream)))


def gemm_mxfp6_(A, fa, sA, gA, W, fw, sW, gW, Y, M, N, K, stream=None):
    out = OUT_BF16 if Y.dtype == torch.bfloat16 else OUT_F32
    _check("bsq_gemm_mxfp6", load().bsq_gemm_mxfp6(
        _p(A), fa, _p(sA), _p(gA), _p(W), fw, _p(sW), _p(gW), _p(Y), out, M, N, K, _stream(stream)))


def gemm_quant_a_workspace_bytes() -> int:
    return load().bsq_gemm_quant_a_workspace_bytes()


def gemm_mxfp6_quant_a_(x, fa, W, fw, sW, gW, Y, s_global_a, workspace, M, N, K, stream=None):
    """Y = gA*gW * quantize(x) W^T with x bf16 [M, K] quantized to fa inside the
    GEMM; s_global_a (device float, or None) receives A's global factor."""
    out = OUT_BF16 if Y.dtype == torch.bfloat16 else OUT_F32
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("bsq_gemm_mxfp6_quant_a", load().bsq_gemm_mxfp6_quant_a(
        _p(x), fa, _p(W), fw, _p(sW), _p(gW), _p(Y), out, _p(s_global_a), M, N, K, _p(workspace), ws_bytes,
        _stream(stream)))


def gemv_nvfp4_(x, W, sW, gW, y, N, K, stream=None):
    M = x.shape[0]
    out = OUT_BF16 if y.dtype == torch.bfloat16 else OUT_F32
    _check("bsq_gemv_nvfp4", load().bsq_gemv_nvfp4(
        _p(x), _p(W), _p(sW), _p(gW), _p(y), out, M, N, K, _stream(stream)))


def gemv_mxfp6_(x, W, fw, sW, gW, y, N, K, stream=None):
    M = x.shape[0]
    out = OUT_BF16 if y.dtype == torch.bfloat16 else OUT_F32
    _check("bsq_gemv_mxfp6", load().bsq_gemv_mxfp6(
        _p(x), _p(W), fw, _p(sW), _p(gW), _p(y), out, M, N, K, _stream(stream)))


def dequant_nvfp4_(codes, scales, g, out, R, K, stream=None):
    _check("bsq_dequant_nvfp4", load().bsq_dequant_nvfp4(
        _p(codes), _p(scales), _p(g), _p(out), R, K, _stream(stream)))


def dequant_mxfp6_(codes, fmt, scales, g, out, R, K, stream=None):
    _check("bsq_dequant_mxfp6", load().bsq_dequant_mxfp6(
        _p(codes), fmt, _p(scales), _p(g), _p(out), R, K, _stream(stream)))


def device_error(stream=None) -> tuple[int, int]:
    """(status, site) of the device error word after the work on `stream` (torch's
    current stream by default) has finished; the word is cleared when set."""
    code = ctypes.c_uint32(0)
    st = load().bsq_get_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value


def launch_count(name: str) -> int:
    return load().bsq_launch_count(KERNEL_IDS[name])


def reset_launch_counts():
    load().bsq_reset_launch_counts()


# --------------------------------------------------------- allocating helpers
def _bf16_bits(x):
    if x.dtype == torch.bfloat16:
        return x.contiguous()
    if x.dtype in (torch.int16, torch.uint16):
        return x.contiguous().view(torch.bfloat16)
    raise TypeError("activations must be bf16 (or their raw 16-bit patterns)")


def quantize_mxfp6(x, fmt="e3m2"):
    """bf16 [M, K] -> (codes uint8, swizzled UE8M0 scales uint8, s_global float32[1])."""
    f = FMT_IDS[fmt] if isinstance(fmt, str) else fmt
    x = _bf16_bits(x)
    M, K = x.shape
    dev = x.device
    codes = torch.empty((M, K if f == E4M3 else 3 * K // 4), dtype=torch.uint8, device=dev)
    scales = torch.empty(scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    wsb = quantize_workspace_bytes(M, K)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
    quantize_mxfp6_(x, f, codes, scales, g, ws)
    return codes, scales, g


def quantize_mxfp6_act(x, act, fmt="e3m2", want_act=False):
    """Fused activation + MX quantize of a bf16 CUDA tensor: (codes, scales,
    s_global[, activated bf16])."""
    fmt_id = {"e3m2": 0, "e2m3": 1, "e4m3": 2}[fmt]
    M, Kin = x.shape
    K = Kin if act == ACT_RELU2 else Kin // 2
    dev = x.device
    codes = torch.empty((M, K if fmt_id == 2 else 3 * K // 4), dtype=torch.uint8, device=dev)
    scales = torch.empty(scale_bytes(M, K // 32), dtype=torch.uint8, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    a = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if want_act else None
    ws = torch.empty(max(16, quantize_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
    quantize_mxfp6_act_(_bf16_bits(x), K, act, fmt_id, codes, scales, sg, a, ws)
    return (codes, scales, sg, a) if want_act else (codes, scales, sg)


def quantize_nvfp4(x):
    """bf16 [M, K] -> (codes int32 [M, K/8] words, swizzled ue4m3 scales, s_global)."""
    x = _bf16_bits(x)
    M, K = x.shape
    dev = x.device
    codes = torch.empty((M, K // 8), dtype=torch.int32, device=dev)
    scales = torch.empty(scale_bytes(M, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    wsb = quantize_workspace_bytes(M, K)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
    quantize_nvfp4_(x, codes, scales, g, ws)
    return codes, scales, g


def gemm_nvfp4(A, sA, gA, W, sW, gW, K, out_dtype=torch.bfloat16):
    M, N = A.shape[0], W.shape[0]
    Y = torch.empty((M, N), dtype=out_dtype, device=A.device)
    gemm_nvfp4_(A, sA, gA, W, sW, gW, Y, M, N, K)
    return Y


def gemm_mxfp6(A, fa, sA, gA, W, fw, sW, gW, K, out_dtype=torch.bfloat16):
    fa = FMT_IDS[fa] if isinstance(fa, str) else fa
    fw = FMT_IDS[fw] if isinstance(fw, str) else fw
    M, N = A.shape[0], W.shape[0]
    Y = torch.empty((M, N), dtype=out_dtype, device=A.device)
    gemm_mxfp6_(A, fa, sA, gA, W, fw, sW, gW, Y, M, N, K)
    return Y


def gemm_mxfp6_quant_a(x, fa, W, fw, sW, gW, K, out_dtype=torch.bfloat16):
    """(Y, s_global_a): the MX product with the activation quantizer in the GEMM."""
    fa = FMT_IDS[fa] if isinstance(fa, str) else fa
    fw = FMT_IDS[fw] if isinstance(fw, str) else fw
    x = _bf16_bits(x)
    M, N = x.shape[0], W.shape[0]
    Y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    sg = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(gemm_quant_a_workspace_bytes(), dtype=torch.uint8, device=x.device)
    gemm_mxfp6_quant_a_(x, fa, W, fw, sW, gW, Y, sg, ws, M, N, K)
    return Y, sg


def gemv_nvfp4(x, W, sW, gW, K, out_dtype=torch.bfloat16):
    x = _bf16_bits(x)
    y = torch.empty((x.shape[0], W.shape[0]), dtype=out_dtype, device=x.device)
    gemv_nvfp4_(x, W, sW, gW, y, W.shape[0], K)
    return y


def gemv_mxfp6(x, W, fw, sW, gW, K, out_dtype=torch.bfloat16):
    fw = FMT_IDS[fw] if isinstance(fw, str) else fw
    x = _bf16_bits(x)
    y = torch.empty((x.shape[0], W.shape[0]), dtype=out_dtype, device=x.device)
    gemv_mxfp6_(x, W, fw, sW, gW, y, W.shape[0], K)
    return y
