"""CPU checks of the C ABI: the library builds and loads without a GPU, exports
every entry point include/bsq.h declares, and its host-only helpers agree with
the layout rules.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_scaled_precision_packed_gb300 import build, bsq
    build.build()
    return bsq.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "bsq.h")).read()
    return sorted(set(re.findall(r"^BSQ_API[^(]*?\b(bsq_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for want in ("bsq_quantize_mxfp6", "bsq_quantize_nvfp4", "bsq_gemm_nvfp4", "bsq_gemm_mxfp6",
                 "bsq_gemv_nvfp4", "bsq_gemv_mxfp6", "bsq_get_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_device_check_build_compiles_and_exports_every_declared_symbol(lib):
    """The bounds-check build (-DBSQ_DEVICE_CHECKS in every kernel file) compiles
    for sm_103a and exports the same entry points; its GPU behaviour is tested
    under -m gpu."""
    from block_scaled_precision_packed_gb300 import build
    path = build.build_variant("devchecks", ["BSQ_DEVICE_CHECKS"], rebuilt=tuple(build.SOURCES))
    checked = ctypes.CDLL(path)
    for name in declared_symbols():
        assert hasattr(checked, name), name


def test_host_helpers(lib):
    from block_scaled_precision_packed_gb300 import bsq
    import oracle as O
    assert lib.bsq_abi_version() == 2
    assert bsq.status_string(0) == "BSQ_OK"
    assert bsq.status_string(3) == "BSQ_ERR_MISALIGNED"
    for rows, blocks in ((1, 1), (128, 4), (300, 257), (28672, 512)):
        assert bsq.scale_bytes(rows, blocks) == O.scale_bytes(rows, blocks)
    assert bsq.quantize_workspace_bytes(16, 4096) == 0
    assert bsq.quantize_workspace_bytes(4096, 4096) >= 1024
    assert bsq.quantize_batch_workspace_bytes() >= 4 * (1 + 1024)   # counter + a partial per CTA
    assert bsq.gemm_quant_a_workspace_bytes() >= 4 * 2048          # the amax pass's partial maxima


def test_oracle_and_library_share_nothing():
    """The oracle is a separate C file with its own header-free build; the CUDA
    sources never include it and it never includes them."""
    csrc = os.path.join(ROOT, "block_scaled_precision_packed_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "bsq_oracle" not in text and "bsqo_" not in text and "oracle/" not in text, f
    otext = open(os.path.join(ROOT, "oracle", "bsq_oracle.c")).read()
    assert "bsq.h" not in otext and "csrc" not in otext
