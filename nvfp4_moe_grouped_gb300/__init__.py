"""GB300-native NVFP4 Mixture-of-Experts layer.

Thin Python binding over the C ABI of ``include/nvfp4_moe.h``: every function
here allocates its outputs with PyTorch (device memory, the current stream),
marshals pointers and sizes, calls the CUDA library and raises on a non-OK
status.  All computation happens in the library's sm_103a kernels; there is no
fallback path.

Calls (same names as the C ABI): ``moe_route_permute``, ``nvfp4_quantize``,
``moe_grouped_gemm_nvfp4``, ``moe_finalize``, ``moe_forward``; plus
``prepare_expert_weights`` (quantise fp32 expert weights into the prepared
layout through ``nvfp4_quantize``) and ``MoeForward`` (a reusable workspace).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import EpilogueArgs, ForwardLayout, MoeError, Weights

EPI_NONE, EPI_SILU_MUL_QUANT, EPI_FINALIZE = 0, 1, 2
SF_LINEAR, SF_TILED, SF_BLOCKED = 0, 1, 2

__all__ = ["moe_route_permute", "nvfp4_quantize", "moe_grouped_gemm_nvfp4", "moe_finalize", "moe_forward",
           "prepare_expert_weights", "MoeForward", "padded_rows_max", "forward_kernel_count", "device_error", "EPI_NONE",
           "EPI_SILU_MUL_QUANT", "EPI_FINALIZE", "SF_LINEAR", "SF_TILED", "SF_BLOCKED", "MoeError",
           "EpilogueArgs", "ForwardGraph"]


def _L():
    return _lib.load()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors are required")
    if not t.is_contiguous():
        raise ValueError("contiguous tensors are required")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(name, status):
    if status != 0:
        raise MoeError(name, status)


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def padded_rows_max(routed_rows: int, E: int) -> int:
    return int(_L().moe_padded_rows_max(routed_rows, E))


def forward_kernel_count(T: int, E: int, k: int, H: int, I: int) -> int:
    """Kernels one moe_forward call (or graph replay) launches for this layer shape."""
    return int(_L().moe_forward_kernel_count(T, E, k, H, I))


def device_error():
    """(code, where) of the last device-side wait that gave up; clears it."""
    code, where = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("moe_device_error", _L().moe_device_error(ctypes.byref(code), ctypes.byref(where)))
    return code.value, where.value


def set_wait_timeout_ns(ns: int) -> None:
    _L().moe_set_wait_timeout_ns(int(ns))


def debug_set_flags(flags: int) -> None:
    _L().moe_debug_set_flags(int(flags))


def fp4_mma_peak_tflops(iters: int = 20000, reps: int = 5, pair: bool = False) -> float:
    """Dense NVFP4 MMA rate of this GPU (TFLOP/s), timed with CUDA events over `reps` probe launches:
    M = 128 MMAs on every SM (pair=False) or the CTA-pair form, M = 256 over two SMs (pair=True)."""
    L = _L()
    probe = L.moe_fp4_mma_probe_pair if pair else L.moe_fp4_mma_probe
    name = "moe_fp4_mma_probe_pair" if pair else "moe_fp4_mma_probe"
    flops = ctypes.c_double(0.0)
    s = torch.cuda.current_stream()
    _check(name, probe(1000, 0, ctypes.byref(flops), _stream(s)))  # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(reps):
        _check(name, probe(iters, 0, ctypes.byref(flops), _stream(s)))
    b.record(s)
    b.synchronize()
    return flops.value * reps / (a.elapsed_time(b) / 1e3) / 1e12


# ---------------------------------------------------------------- routing

@dataclass
class Routing:
    topk_id: torch.Tensor          # int32 [T, k]
    topk_w: torch.Tensor           # float32 [T, k]
    expert_offsets: torch.Tensor   # int32 [E+1]
    perm_to_expanded: torch.Tensor  # int32 [R]
    expanded_to_perm: torch.Tensor  # int32 [R]
    expanded_to_row: torch.Tensor   # int32 [R]


def moe_route_permute(logits: torch.Tensor, k: int, stream=None) -> Routing:
    T, E = logits.shape
    dev = logits.device
    R = T * k
    r = Routing(_empty((T, k), torch.int32, dev), _empty((T, k), torch.float32, dev), _empty(E + 1, torch.int32, dev),
                _empty(R, torch.int32, dev), _empty(R, torch.int32, dev), _empty(R, torch.int32, dev))
    L = _L()
    wsb = L.moe_route_permute_workspace_size(T, E, k)
    ws = _empty(max(wsb, 256), torch.uint8, dev)
    _check("moe_route_permute", L.moe_route_permute(
        _ptr(logits.float().contiguous()), T, E, k, _ptr(r.topk_id), _ptr(r.topk_w), _ptr(r.expert_offsets),
        _ptr(r.perm_to_expanded), _ptr(r.expanded_to_perm), _ptr(r.expanded_to_row), _ptr(ws), wsb, _stream(stream)))
    return r


def moe_router(x: torch.Tensor, w_gate: torch.Tensor, k: int, want_logits: bool = True, stream=None,
               out: Routing | None = None, logits: torch.Tensor | None = None, ws: torch.Tensor | None = None,
               x_scale: torch.Tensor | None = None):
    """Router logits x . w_gate^T on the tensor cores (bf16 in, FP32 sums), then moe_route_permute.

    `out`, `logits` and `ws` may be given preallocated (e.g. for graph capture); `x_scale` (f32 [1]),
    when given, receives x's NVFP4 decode multiplier.  Returns (Routing, logits f32 [T][E] or None)."""
    if x.dtype != torch.bfloat16 or w_gate.dtype != torch.bfloat16:
        raise TypeError("x and w_gate must be bf16")
    x = x.contiguous()
    w_gate = w_gate.contiguous()
    T, H = x.shape
    E = w_gate.shape[0]
    dev = x.device
    R = T * k
    r = out if out is not None else Routing(
        _empty((T, k), torch.int32, dev), _empty((T, k), torch.float32, dev), _empty(E + 1, torch.int32, dev),
        _empty(R, torch.int32, dev), _empty(R, torch.int32, dev), _empty(R, torch.int32, dev))
    if logits is None and want_logits:
        logits = _empty((T, E), torch.float32, dev)
    L = _L()
    wsb = L.moe_router_workspace_size(T, E, H, k)
    if ws is None:
        ws = _empty(max(wsb, 256), torch.uint8, dev)
    elif ws.numel() < wsb:
        raise ValueError("router workspace too small")
    _check("moe_router", L.moe_router(
        _ptr(x), _ptr(w_gate), T, E, H, k, _ptr(logits), _ptr(x_scale), _ptr(r.topk_id), _ptr(r.topk_w),
        _ptr(r.expert_offsets),
        _ptr(r.perm_to_expanded), _ptr(r.expanded_to_perm), _ptr(r.expanded_to_row), _ptr(ws), wsb,
        _stream(stream)))
    return r, logits


# ---------------------------------------------------------------- quantisation

def nvfp4_quantize(x: torch.Tensor, tensor_scale: torch.Tensor | None = None, groups: int = 1,
                   n_items: int | None = None, src_div: int = 1, dst_row: torch.Tensor | None = None,
                   sf_layout: int = SF_LINEAR, dst_rows_alloc: int | None = None, codes=None, sf=None, stream=None):
    """Quantise rows of x (bf16 or float32, [rows, K]) to NVFP4.

    tensor_scale None: dynamic per-group scale (computed and returned); else a
    float32 device tensor [groups] read as the decode multipliers.
    Returns (codes, sf, tensor_scale).
    """
    if x.dtype == torch.bfloat16:
        in_dtype = 0
    elif x.dtype == torch.float32:
        in_dtype = 1
    else:
        raise TypeError("x must be bf16 or float32")
    rows, K = x.shape
    dev = x.device
    n_items = rows * src_div if n_items is None else n_items
    if dst_rows_alloc is None:
        dst_rows_alloc = n_items if dst_row is None else int(dst_row.max().item()) + 1
        if sf_layout == SF_TILED:
            dst_rows_alloc = ((dst_rows_alloc + 127) // 128) * 128
    dynamic = tensor_scale is None
    if dynamic:
        tensor_scale = _empty(groups, torch.float32, dev)
    if sf_layout == SF_BLOCKED:
        if codes is None:
            codes = torch.zeros(int(_L().moe_blocked_weight_bytes(dst_rows_alloc, K)), dtype=torch.uint8, device=dev)
    else:
        if codes is None:
            codes = torch.zeros((dst_rows_alloc, K // 2), dtype=torch.uint8, device=dev)
        if sf is None:
            sf = torch.zeros((dst_rows_alloc * (K // 16),), dtype=torch.uint8, device=dev)
            if sf_layout == SF_LINEAR:
                sf = sf.view(dst_rows_alloc, K // 16)
    L = _L()
    wsb = L.nvfp4_quantize_workspace_size(groups)
    ws = _empty(max(wsb, 256), torch.uint8, dev)
    _check("nvfp4_quantize", L.nvfp4_quantize(
        _ptr(x.contiguous()), in_dtype, rows, K, groups, _ptr(tensor_scale), int(dynamic), n_items, src_div,
        _ptr(dst_row), _ptr(codes), _ptr(sf), sf_layout, dst_rows_alloc, _ptr(ws), wsb, _stream(stream)))
    return codes, sf, tensor_scale


@dataclass
class PreparedWeights:
    blocked: torch.Tensor  # uint8, blocked layout over E*N rows (gate/up interleaved for gate_up)
    scale: torch.Tensor    # float32 [E]
    E: int
    N: int
    K: int


def gate_up_row_map(N: int, device) -> torch.Tensor:
    """Prepared row of each gate_up row (gate rows [0, I), up rows [I, 2I)) inside one expert."""
    I = N // 2
    r = torch.arange(N, device=device, dtype=torch.int64)
    gate = r < I
    i = torch.where(gate, r, r - I)
    return (128 * (i // 64) + torch.where(gate, 0, 64) + i % 64).to(torch.int32)


def prepare_expert_weights(w: torch.Tensor, gate_up: bool, stream=None) -> PreparedWeights:
    """Quantise fp32 expert weights [E, N, K] (one dynamic scale per expert) into the prepared layout."""
    E, N, K = w.shape
    dev = w.device
    dst = None
    if gate_up:
        local = gate_up_row_map(N, dev).to(torch.int64)
        dst = (torch.arange(E, device=dev, dtype=torch.int64)[:, None] * N + local[None, :]).reshape(-1).to(torch.int32)
    blocked, _, scale = nvfp4_quantize(w.reshape(E * N, K), None, groups=E, dst_row=dst, sf_layout=SF_BLOCKED,
                                       dst_rows_alloc=E * N, stream=stream)
    return PreparedWeights(blocked, scale, E, N, K)


# ---------------------------------------------------------------- grouped GEMM

def moe_grouped_gemm_nvfp4(a_codes, a_sf, a_scale, w: PreparedWeights, expert_offsets, epilogue=EPI_NONE,
                           h_scale: float = 0.0, h_codes=None, h_sf=None, h_scale_out=None, h_f32=None,
                           perm_to_expanded=None, topk_w=None, T: int = 0, k: int = 0, out=None, stream=None):
    """Expert-grouped NVFP4 GEMM over routed rows (padded-row layout, tiled scales)."""
    rows_alloc = a_codes.shape[0]
    E = w.E
    dev = a_codes.device
    ep = EpilogueArgs()
    wsb = 0
    ws = None
    if epilogue == EPI_NONE:
        if out is None:
            out = torch.zeros((rows_alloc, w.N), dtype=torch.bfloat16, device=dev)
    elif epilogue == EPI_SILU_MUL_QUANT:
        I = w.N // 2
        if h_codes is None:
            h_codes = torch.zeros((rows_alloc, I // 2), dtype=torch.uint8, device=dev)
        if h_sf is None:
            h_sf = torch.zeros((rows_alloc * (I // 16),), dtype=torch.uint8, device=dev)
        ep.h_scale = float(h_scale)
        ep.h_scale_out = _ptr(h_scale_out)
        ep.h_codes = _ptr(h_codes)
        ep.h_sf = _ptr(h_sf)
        ep.h_f32 = _ptr(h_f32)
    else:
        if out is None:
            out = _empty((T, w.N), torch.bfloat16, dev)
        ep.perm_to_expanded = _ptr(perm_to_expanded)
        ep.topk_w = _ptr(topk_w)
        ep.T = T
        ep.k = k
        wsb = _L().moe_grouped_gemm_workspace_size(epilogue, T, k, w.N)
        ws = _empty(wsb, torch.uint8, dev)
    _check("moe_grouped_gemm_nvfp4", _L().moe_grouped_gemm_nvfp4(
        _ptr(a_codes), _ptr(a_sf), _ptr(a_scale), _ptr(w.blocked), _ptr(w.scale), _ptr(expert_offsets), E,
        rows_alloc, w.N, w.K, epilogue, ctypes.byref(ep), _ptr(out) if out is not None else None, _ptr(ws), wsb,
        _stream(stream)))
    if epilogue == EPI_SILU_MUL_QUANT:
        return h_codes, h_sf
    return out


def dense_gemm_nvfp4(a_codes, a_sf, a_scale, w: PreparedWeights, M: int, out=None, stream=None):
    """Dense NVFP4 GEMM C[M][N] = A[M][K] . B[N][K]^T (BF16 out): the grouped GEMM with one group.

    A is in the padded-row layout with tiled scales (rows_alloc = a_codes.shape[0] >= M, a multiple
    of 128), `w` one prepared matrix (E = 1).  Returns C over rows_alloc rows (rows >= M untouched)."""
    if w.E != 1:
        raise ValueError("dense_gemm_nvfp4 takes one prepared matrix (E = 1)")
    offs = torch.tensor([0, M], dtype=torch.int32, device=a_codes.device)
    return moe_grouped_gemm_nvfp4(a_codes, a_sf, a_scale, w, offs, EPI_NONE, out=out, stream=stream)


def moe_finalize(y: torch.Tensor, topk_w: torch.Tensor, row_of_item: torch.Tensor, out=None, stream=None):
    T, k = topk_w.shape
    N = y.shape[1]
    if out is None:
        out = _empty((T, N), torch.bfloat16, y.device)
    _check("moe_finalize", _L().moe_finalize(_ptr(y), y.shape[0], _ptr(topk_w), _ptr(row_of_item), T, k, N,
                                             _ptr(out), _stream(stream)))
    return out


# ---------------------------------------------------------------- fused layer

class MoeForward:
    """A reusable workspace for moe_forward at one (T, E, k, H, I)."""

    def __init__(self, T: int, E: int, k: int, H: int, I: int, device="cuda", gated: bool = False):
        self.T, self.E, self.k, self.H, self.I = T, E, k, H, I
        L = _L()
        self.layout = ForwardLayout()
        _check("moe_forward_workspace_layout", L.moe_forward_workspace_layout(T, E, k, H, I, ctypes.byref(self.layout)))
        # moe_forward_gated needs the router's workspace after moe_forward's (same layout up front)
        total = L.moe_forward_gated_workspace_size(T, E, k, H, I) if gated else self.layout.total
        if gated and total == 0:
            raise MoeError("moe_forward_gated_workspace_size", 1)
        self.ws = torch.zeros(total, dtype=torch.uint8, device=device)

    def gated(self, x, w_gate, w13: PreparedWeights, w2: PreparedWeights, h_scale: float, out=None, stream=None):
        """moe_forward_gated: the router (x . w_gate^T, top-k, permutation) in front of the layer."""
        if out is None:
            out = _empty((self.T, self.H), torch.bfloat16, x.device)
        wts = Weights(_ptr(w13.blocked), _ptr(w13.scale), _ptr(w2.blocked), _ptr(w2.scale))
        _check("moe_forward_gated", _L().moe_forward_gated(
            _ptr(x), _ptr(w_gate), ctypes.byref(wts), self.T, self.E, self.k, self.H, self.I, float(h_scale),
            _ptr(out), _ptr(self.ws), self.ws.numel(), _stream(stream)))
        return out

    def view(self, name: str, dtype, shape):
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(shape)

    def graph(self, x, logits, w13: PreparedWeights, w2: PreparedWeights, h_scale: float, out=None,
              stage_events: bool = True) -> "ForwardGraph":
        if out is None:
            out = _empty((self.T, self.H), torch.bfloat16, x.device)
        return ForwardGraph(self, x, logits, w13, w2, h_scale, out, stage_events)

    def __call__(self, x, logits, w13: PreparedWeights, w2: PreparedWeights, h_scale: float, out=None, stream=None):
        if out is None:
            out = _empty((self.T, self.H), torch.bfloat16, x.device)
        wts = Weights(_ptr(w13.blocked), _ptr(w13.scale), _ptr(w2.blocked), _ptr(w2.scale))
        _check("moe_forward", _L().moe_forward(
            _ptr(x), _ptr(logits), ctypes.byref(wts), self.T, self.E, self.k, self.H, self.I, float(h_scale),
            _ptr(out), _ptr(self.ws), self.layout.total, _stream(stream)))
        return out


class ForwardGraph:
    """The whole layer captured as one CUDA graph (see moe_forward_graph_create).

    It keeps the tensors it was created with; refill x and logits in place and call launch().
    """

    def __init__(self, fwd: "MoeForward", x, logits, w13: PreparedWeights, w2: PreparedWeights, h_scale: float, out,
                 stage_events: bool = True):
        self._keep = (fwd, x, logits, w13, w2, out)
        self.out = out
        self.handle = ctypes.c_void_p(None)
        wts = Weights(_ptr(w13.blocked), _ptr(w13.scale), _ptr(w2.blocked), _ptr(w2.scale))
        _check("moe_forward_graph_create", _L().moe_forward_graph_create(
            _ptr(x), _ptr(logits), ctypes.byref(wts), fwd.T, fwd.E, fwd.k, fwd.H, fwd.I, float(h_scale), _ptr(out),
            _ptr(fwd.ws), fwd.layout.total, int(stage_events), ctypes.byref(self.handle)))

    def launch(self, stream=None):
        _check("moe_forward_graph_launch", _L().moe_forward_graph_launch(self.handle, _stream(stream)))
        return self.out

    def run_host(self, x_host, logits_host, out_host, stream=None):
        """One step from and to host tensors (page-locked for overlap): copy in, replay, copy out, all on
        `stream`; returns out_host (valid once the stream gets there)."""
        for t in (x_host, logits_host, out_host):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("contiguous host tensors are required")
        _check("moe_forward_graph_run_host", _L().moe_forward_graph_run_host(
            self.handle, ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(logits_host.data_ptr()),
            ctypes.c_void_p(out_host.data_ptr()), _stream(stream)))
        return out_host

    def stage_ms(self):
        """(route, quantise, gate_up, down+finalize, total) of the last launch, in ms."""
        ms = (ctypes.c_float * 5)()
        _check("moe_forward_graph_stage_ms", _L().moe_forward_graph_stage_ms(self.handle, ms))
        return list(ms)

    def close(self):
        if self.handle:
            _L().moe_forward_graph_destroy(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_forward(x, logits, w13: PreparedWeights, w2: PreparedWeights, k: int, h_scale: float, out=None, stream=None):
    T, H = x.shape
    E = logits.shape[1]
    I = w2.K
    return MoeForward(T, E, k, H, I, x.device)(x, logits, w13, w2, h_scale, out, stream)
