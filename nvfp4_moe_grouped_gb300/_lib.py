"""ctypes loader of libnvfp4_moe.so: argument and return types of every entry point.

There is no fallback: if the library cannot be loaded the import of the
binding raises, and every call checks its status and raises on error.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_int, c_int64, c_size_t, c_float, c_void_p, c_uint64 = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                                         ctypes.c_float, ctypes.c_void_p, ctypes.c_uint64)


class EpilogueArgs(ctypes.Structure):
    """Mirror of moe_epilogue_args."""
    _fields_ = [
        ("h_scale", c_float),
        ("h_scale_out", c_void_p),
        ("h_codes", c_void_p),
        ("h_sf", c_void_p),
        ("h_f32", c_void_p),
        ("perm_to_expanded", c_void_p),
        ("topk_w", c_void_p),
        ("T", ctypes.c_int32),
        ("k", ctypes.c_int32),
    ]


class Weights(ctypes.Structure):
    """Mirror of moe_weights."""
    _fields_ = [
        ("w13", c_void_p),
        ("w13_scale", c_void_p),
        ("w2", c_void_p),
        ("w2_scale", c_void_p),
    ]


class ForwardLayout(ctypes.Structure):
    """Mirror of moe_forward_layout."""
    _fields_ = [(n, c_size_t) for n in (
        "topk_id", "topk_w", "expert_offsets", "perm_to_expanded", "expanded_to_perm", "expanded_to_row",
        "x_scale", "x_codes", "x_sf", "h_scale", "h_codes", "h_sf", "route_ws", "quant_ws", "gemm_ws",
        "small_scratch")] + [
        ("padded_rows", c_int64), ("total", c_size_t)]


# name -> (restype, argtypes); every symbol declared in include/nvfp4_moe.h
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_abi_version": (c_int, []),
    "moe_device_error": (c_int, [c_void_p, c_void_p]),
    "moe_set_wait_timeout_ns": (None, [c_uint64]),
    "moe_debug_set_flags": (None, [c_int]),
    "moe_padded_rows_max": (c_int64, [c_int64, c_int]),
    "moe_blocked_weight_bytes": (c_size_t, [c_int64, c_int]),
    "moe_route_permute_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_route_permute": (c_int, [c_void_p, c_int, c_int, c_int] + [c_void_p] * 7 + [c_size_t, c_void_p]),
    "moe_router_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "moe_router": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int] + [c_void_p] * 9 + [c_size_t, c_void_p]),
    "moe_route_permute_static_scratch_bytes": (c_size_t, []),
    "moe_route_permute_static": (c_int, [c_void_p, c_int, c_int, c_int] + [c_void_p] * 7),
    "nvfp4_quantize_workspace_size": (c_size_t, [c_int]),
    "nvfp4_quantize": (c_int, [c_void_p, c_int, c_int64, c_int, c_int, c_void_p, c_int, c_int64, c_int, c_void_p,
                               c_void_p, c_void_p, c_int, c_int64, c_void_p, c_size_t, c_void_p]),
    "moe_grouped_gemm_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "moe_grouped_gemm_nvfp4": (c_int, [c_void_p] * 6 + [c_int, c_int64, c_int, c_int, c_int, c_void_p, c_void_p,
                                                        c_void_p, c_size_t, c_void_p]),
    "moe_finalize": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "moe_fp4_mma_probe": (c_int, [c_int, c_int, c_void_p, c_void_p]),
    "moe_fp4_mma_probe_pair": (c_int, [c_int, c_int, c_void_p, c_void_p]),
    "moe_forward_workspace_size": (c_size_t, [c_int] * 5),
    "moe_forward_gated_workspace_size": (c_size_t, [c_int] * 5),
    "moe_forward_gated": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float, c_void_p,
                                  c_void_p, c_size_t, c_void_p]),
    "moe_forward_workspace_layout": (c_int, [c_int] * 5 + [c_void_p]),
    "moe_forward_kernel_count": (c_int, [c_int] * 5),
    "moe_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float, c_void_p,
                            c_void_p, c_size_t, c_void_p]),
    "moe_forward_graph_create": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                                         c_void_p, c_void_p, c_size_t, c_int, c_void_p]),
    "moe_forward_graph_launch": (c_int, [c_void_p, c_void_p]),
    "moe_forward_graph_stage_ms": (c_int, [c_void_p, c_void_p]),
    "moe_forward_graph_run_host": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_forward_graph_destroy": (None, [c_void_p]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) the CUDA library; raises if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and _build.is_stale():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"CUDA library {path} is missing; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, call: str, status: int):
        lib = load(False)
        super().__init__(f"{call} failed: {lib.moe_status_string(status).decode()} (status {status})")
        self.status = status
