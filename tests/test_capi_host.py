"""Host-side checks of the C ABI that need no GPU.

The library loads without a device, exports every function the header
declares, answers its size queries, and rejects bad arguments with the
documented status before touching CUDA.
"""
import ctypes
import os
import re

import pytest

import nvfp4_moe_grouped_gb300 as moe
from nvfp4_moe_grouped_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4_moe.h")

OK, INVALID, MISALIGNED, UNSUPPORTED, RESOURCE, CUDA, TIMEOUT, WORKSPACE = range(8)


@pytest.fixture(scope="module")
def L():
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^MOE_API [^(]*?\b([a-z0-9_]+)\(", text, re.M)


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding signatures and header disagree"


def test_status_strings_and_version(L):
    assert L.moe_abi_version() == 6
    for s in range(8):
        assert L.moe_status_string(s)
    assert L.moe_status_string(99) == b"unknown status"


def test_padded_rows_bound(L):
    assert L.moe_padded_rows_max(8192, 256) == 8192 + 127 * 256
    assert L.moe_padded_rows_max(32, 8) % 128 == 0
    assert L.moe_padded_rows_max(32, 8) >= 32 + 127 * 8
    assert L.moe_padded_rows_max(3, 256) == 384  # 3 + 127*3 = 384
    assert L.moe_padded_rows_max(0, 4) == 128


def test_forward_layout_is_consistent(L):
    lay = _lib.ForwardLayout()
    assert L.moe_forward_workspace_layout(1024, 256, 8, 6144, 2048, ctypes.byref(lay)) == OK
    assert lay.padded_rows == L.moe_padded_rows_max(8192, 256)
    offs = [getattr(lay, f) for f, _ in _lib.ForwardLayout._fields_[:15]]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    assert lay.x_sf - lay.x_codes >= lay.padded_rows * 6144 // 2
    assert lay.total == L.moe_forward_workspace_size(1024, 256, 8, 6144, 2048)
    assert L.moe_forward_workspace_layout(4, 8, 9, 256, 128, ctypes.byref(lay)) == INVALID  # k > E
    # the single-launch path's scratch exists only for the small layers it takes
    SIZE_MAX = 2 ** 64 - 1
    assert L.moe_forward_workspace_layout(1024, 256, 8, 6144, 2048, ctypes.byref(lay)) == OK
    assert lay.small_scratch == SIZE_MAX
    assert L.moe_forward_workspace_layout(16, 8, 2, 256, 128, ctypes.byref(lay)) == OK
    assert lay.small_scratch != SIZE_MAX and lay.small_scratch % 256 == 0
    # 256 reserved bytes inside the workspace
    assert lay.small_scratch + 256 <= lay.total == L.moe_forward_workspace_size(16, 8, 2, 256, 128)


def test_forward_kernel_count(L):
    """One launch for the small layers the single-kernel path takes; the staged count otherwise: routing
    (1 kernel when every item fits one chunk, else 3), amax + quantiser, two GEMMs, the FINALIZE closing
    pass.  Debug flag bit 2 keeps the staged kernels."""
    assert L.moe_forward_kernel_count(16, 8, 2, 256, 128) == 1
    assert L.moe_forward_kernel_count(64, 8, 1, 1024, 512) == 1      # T * k, H, I and E * I at their limits
    assert L.moe_forward_kernel_count(64, 64, 1, 256, 64) == 1       # E at its limit
    assert L.moe_forward_kernel_count(64, 64, 1, 1024, 512) == 6     # E * I > 4096: staged
    assert L.moe_forward_kernel_count(33, 8, 2, 256, 128) == 6      # 66 items: staged, one routing chunk
    assert L.moe_forward_kernel_count(16, 65, 2, 256, 128) == 6     # E > 64
    assert L.moe_forward_kernel_count(16, 8, 2, 1152, 128) == 6     # H > 1024
    assert L.moe_forward_kernel_count(1024, 256, 8, 6144, 2048) == 8
    assert L.moe_forward_kernel_count(16, 8, 9, 256, 128) == 0      # k > E
    L.moe_debug_set_flags(4)
    try:
        assert L.moe_forward_kernel_count(16, 8, 2, 256, 128) == 6
    finally:
        L.moe_debug_set_flags(0)


def test_blocked_weight_bytes(L):
    assert L.moe_blocked_weight_bytes(256 * 4096, 6144) == 256 * 32 * 24 * 18432
    assert L.moe_blocked_weight_bytes(128, 320) == 2 * 18432      # partial last K tile takes a whole block
    assert L.moe_blocked_weight_bytes(100, 256) == 0
    assert L.moe_blocked_weight_bytes(128, 96) == 0


def test_workspace_queries(L):
    assert L.moe_grouped_gemm_workspace_size(moe.EPI_NONE, 1024, 8, 6144) == 0
    assert L.moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, 1024, 8, 6144) == 1024 * 6144 * 4      # atomics
    # past 64 MiB the atomics take column chunks; per-item rows only when one 128-column chunk is too large
    assert L.moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, 16384, 8, 6144) == 16384 * 6144 * 4
    assert L.moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, 131072, 8, 6144) == 131072 * 6144 * 4
    assert L.moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, 131073, 2, 256) == 131073 * 2 * 256 * 4
    assert L.nvfp4_quantize_workspace_size(1) == 256
    assert L.moe_route_permute_workspace_size(1024, 256, 8) >= (1024 // 32) * 256 * 4


P = ctypes.c_void_p(0x1000)       # aligned fake pointer: never dereferenced (rejected before launch)
Q = ctypes.c_void_p(0x1008)       # misaligned fake pointer


def test_route_permute_rejects_before_launch(L):
    args = [P] * 6
    assert L.moe_route_permute(None, 4, 8, 2, *args, P, 1 << 20, None) == INVALID
    assert L.moe_route_permute(P, 4, 8, 9, *args, P, 1 << 20, None) == INVALID       # k > E
    assert L.moe_route_permute(P, 0, 8, 2, *args, P, 1 << 20, None) == INVALID       # T = 0
    assert L.moe_route_permute(P, 4, 2048, 2, *args, P, 1 << 20, None) == UNSUPPORTED
    assert L.moe_route_permute(P, 4, 64, 33, *args, P, 1 << 20, None) == UNSUPPORTED  # k > 32
    assert L.moe_route_permute(P, 4, 8, 2, *args, P, 0, None) == WORKSPACE


def test_quantize_rejects_before_launch(L):
    q = L.nvfp4_quantize
    assert q(P, 0, 16, 40, 1, P, 0, 16, 1, None, P, P, 0, 16, P, 256, None) == UNSUPPORTED     # K % 16
    assert q(P, 0, 16, 96, 1, P, 0, 16, 1, None, P, P, 1, 128, P, 256, None) == UNSUPPORTED    # tiled K % 64
    assert q(P, 0, 16, 64, 1, P, 0, 16, 1, None, P, P, 1, 100, P, 256, None) == UNSUPPORTED    # tiled rows % 128
    assert q(P, 0, 16, 64, 3, P, 0, 15, 1, None, P, P, 0, 16, P, 256, None) == INVALID         # rows % groups
    assert q(P, 0, 16, 64, 1, P, 0, 17, 1, None, P, P, 0, 16, P, 256, None) == INVALID         # items > rows
    assert q(Q, 0, 16, 64, 1, P, 0, 16, 1, None, P, P, 0, 16, P, 256, None) == MISALIGNED
    assert q(P, 0, 16, 64, 1, P, 1, 16, 1, None, P, P, 0, 16, None, 0, None) == WORKSPACE
    assert q(P, 7, 16, 64, 1, P, 0, 16, 1, None, P, P, 0, 16, P, 256, None) == INVALID         # dtype
    assert q(P, 0, 16, 64, 1, P, 0, 30, 2, P, P, P, 0, 32, P, 256, None) == UNSUPPORTED       # partial fan-out
    assert q(P, 0, 2, 64, 1, P, 0, 66, 33, P, P, P, 0, 66, P, 256, None) == UNSUPPORTED       # fan-out > 32


def test_grouped_gemm_rejects_before_launch(L):
    g = L.moe_grouped_gemm_nvfp4
    base = [P] * 6
    assert g(*base, 8, 128, 256, 288, moe.EPI_NONE, None, P, None, 0, None) == UNSUPPORTED      # K % 64
    assert g(*base, 8, 128, 200, 256, moe.EPI_NONE, None, P, None, 0, None) == UNSUPPORTED      # N % 128
    assert g(*base, 8, 100, 256, 256, moe.EPI_NONE, None, P, None, 0, None) == UNSUPPORTED      # rows % 128
    assert g(*base, 2048, 128, 256, 256, moe.EPI_NONE, None, P, None, 0, None) == UNSUPPORTED   # E
    assert g(*base, 8, 128, 256, 256, 9, None, P, None, 0, None) == INVALID                     # epilogue
    assert g(Q, *[P] * 5, 8, 128, 256, 256, moe.EPI_NONE, None, P, None, 0, None) == MISALIGNED
    assert g(*base, 8, 128, 256, 256, moe.EPI_SILU_MUL_QUANT, None, None, None, 0, None) == INVALID
    ep = _lib.EpilogueArgs()
    ep.h_scale = 1.0
    ep.h_codes = P
    ep.h_sf = P
    ep.h_scale = 0.0
    assert g(*base, 8, 128, 256, 256, moe.EPI_SILU_MUL_QUANT, ctypes.byref(ep), None, None, 0, None) == INVALID
    fin = _lib.EpilogueArgs()
    fin.perm_to_expanded = P
    fin.topk_w = P
    fin.T = 4
    fin.k = 2
    assert g(*base, 8, 128, 256, 256, moe.EPI_FINALIZE, ctypes.byref(fin), P, P, 16, None) == WORKSPACE


def test_finalize_and_forward_reject_before_launch(L):
    assert L.moe_finalize(P, 8, P, P, 4, 2, 12, P, None) == UNSUPPORTED   # N % 8
    assert L.moe_finalize(Q, 8, P, P, 4, 2, 16, P, None) == MISALIGNED
    assert L.moe_finalize(P, 0, P, P, 4, 2, 16, P, None) == INVALID       # no rows of y
    w = _lib.Weights(P, P, P, P)
    assert L.moe_forward(P, P, ctypes.byref(w), 4, 8, 2, 200, 128, 1.0, P, P, 1 << 30, None) == UNSUPPORTED
    assert L.moe_forward(P, P, ctypes.byref(w), 4, 8, 2, 256, 128, 0.0, P, P, 1 << 30, None) == INVALID
    assert L.moe_forward(P, P, ctypes.byref(w), 4, 8, 2, 256, 128, 1.0, P, P, 16, None) == WORKSPACE


def test_cublaslt_reference_library_builds_and_exports():
    """The dense-GEMM timing reference (cuBLASLt, benchmark only) is a separate library beside the layer's; it
    builds with the package and exports its one entry point.  No GPU call is made."""
    import ctypes
    import os

    from nvfp4_moe_grouped_gb300 import build as nb
    path = nb.build_reference()
    if path is None:
        pytest.skip("cuBLASLt is not available to link against here")
    assert os.path.exists(path) and path != nb.LIB
    assert hasattr(ctypes.CDLL(path), "nvfp4_cublaslt_gemm_time")
