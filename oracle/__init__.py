"""CPU oracle for the NVFP4 Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package; the product library never
does, and the oracle shares no code with the CUDA path.  The arithmetic lives
in ``moe_oracle.c`` (plain C, FP64 sums, FP32 only where a floating-point value
decides an integer); this module only marshals numpy arrays into it and
composes its steps in the order the method states them:

  route -> permute -> quantise x -> gate_up GEMM -> SiLU-mul -> requantise h
        -> down GEMM -> FINALIZE (router-weighted sum back into token rows).

The tiled scale-factor layout the GEMM kernels consume is re-derived here from
its written definition (``tiled_sf_offset``) so tests can compare the GPU's
bytes against the oracle's linear-layout bytes without touching product code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        u8p = ctypes.POINTER(ctypes.c_uint8)
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_tensor_scale_from_amax.restype = ctypes.c_float
        L.orc_tensor_scale_from_amax.argtypes = [ctypes.c_float]
        L.orc_amax.restype = ctypes.c_float
        L.orc_amax.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_void_p, ctypes.c_void_p]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_void_p]
        L.orc_exp.restype = ctypes.c_float
        L.orc_exp.argtypes = [ctypes.c_float]
        L.orc_router_logits.restype = None
        L.orc_router_logits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p]
        L.orc_route.restype = ctypes.c_int
        L.orc_route.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_void_p, ctypes.c_void_p]
        L.orc_permute.restype = ctypes.c_int
        L.orc_permute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.orc_grouped_gemm.restype = ctypes.c_int
        L.orc_grouped_gemm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p]
        L.orc_grouped_gemm_element.restype = ctypes.c_double
        L.orc_grouped_gemm_element.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
                                               ctypes.c_int]
        L.orc_silu_mul.restype = None
        L.orc_silu_mul.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
        L.orc_bf16_bits.restype = ctypes.c_uint16
        L.orc_bf16_bits.argtypes = [ctypes.c_double]
        L.orc_bf16_value.restype = ctypes.c_double
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_finalize.restype = None
        L.orc_finalize.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.orc_smem_model_bytes.restype = ctypes.c_int64
        L.orc_smem_model_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int]
        del u8p
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(code)


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(x)


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(x)


def exp32(x: float) -> float:
    return lib().orc_exp(x)


def tensor_scale_from_amax(amax: float) -> float:
    return lib().orc_tensor_scale_from_amax(amax)


def smem_model_bytes(M: int, N: int, K: int, stages: int, finalize: bool) -> int:
    return lib().orc_smem_model_bytes(M, N, K, stages, int(finalize))


# ---------------------------------------------------------------- bf16 helpers

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns (uint16) to float64."""
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    L = lib()
    flat = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, x in enumerate(flat):
        out[i] = L.orc_bf16_bits(float(x))
    return out.reshape(np.shape(v))


# ---------------------------------------------------------------- arrays

def amax(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return lib().orc_amax(_p(x), x.size)


def quantize(x: np.ndarray, scale: float):
    """NVFP4-quantise rows of x (float32 [rows, K]) with decode multiplier ``scale``.

    Returns (codes uint8 [rows, K/2], sf uint8 [rows, K/16]) in the linear layouts.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    rc = lib().orc_quantize(_p(x), rows, K, np.float32(scale), _p(codes), _p(sf))
    assert rc == 0
    return codes, sf


def quantize_dynamic(x: np.ndarray):
    """Per-tensor dynamic scale s = amax/(6*448), then ``quantize``."""
    s = tensor_scale_from_amax(amax(x))
    codes, sf = quantize(x, s)
    return codes, sf, s


def dequantize(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """FP64 values e2m1(code) * e4m3(sf), without the per-tensor multiplier."""
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    rows = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    lib().orc_dequantize(_p(codes), _p(sf), rows, K, _p(out))
    return out


def router_logits(x: np.ndarray, w_gate: np.ndarray) -> np.ndarray:
    """logits[t][e] = sum_h x[t][h] * w_gate[e][h] in FP64, rounded once to FP32 (reading R8).

    x [T][H] and w_gate [E][H] hold bf16 values (any float dtype that represents them exactly)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w_gate, dtype=np.float32)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    out = np.zeros((T, E), np.float32)
    lib().orc_router_logits(_p(x), _p(w), T, E, H, _p(out))
    return out


def route(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    assert lib().orc_route(_p(logits), T, E, k, _p(ids), _p(w)) == 0
    return ids, w


def permute(topk_id: np.ndarray, E: int):
    topk_id = np.ascontiguousarray(topk_id, np.int32)
    T, k = topk_id.shape
    R = T * k
    offs = np.zeros(E + 1, np.int32)
    p2e = np.zeros(R, np.int32)
    e2p = np.zeros(R, np.int32)
    assert lib().orc_permute(_p(topk_id), T, k, E, _p(offs), _p(p2e), _p(e2p)) == 0
    return offs, p2e, e2p


def grouped_gemm(a_codes, a_sf, a_scale, b_codes, b_sf, b_scale, expert_offsets, N, K) -> np.ndarray:
    """FP64 Y[r, n] for rows grouped by expert (linear layouts).

    b_codes: uint8 [E, N, K/2]; b_sf: uint8 [E, N, K/16]; b_scale: float32 [E].
    """
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    a_sf = np.ascontiguousarray(a_sf, np.uint8)
    b_codes = np.ascontiguousarray(b_codes, np.uint8)
    b_sf = np.ascontiguousarray(b_sf, np.uint8)
    b_scale = np.ascontiguousarray(b_scale, np.float32)
    offs = np.ascontiguousarray(expert_offsets, np.int32)
    E = offs.shape[0] - 1
    R = int(offs[-1])
    out = np.zeros((R, N), np.float64)
    assert lib().orc_grouped_gemm(_p(a_codes), _p(a_sf), float(a_scale), _p(b_codes), _p(b_sf),
                                  _p(b_scale), _p(offs), E, N, K, _p(out)) == 0
    return out


def gemm_element(a_row_codes, a_row_sf, a_scale, b_row_codes, b_row_sf, b_scale) -> float:
    a_row_codes = np.ascontiguousarray(a_row_codes, np.uint8)
    a_row_sf = np.ascontiguousarray(a_row_sf, np.uint8)
    b_row_codes = np.ascontiguousarray(b_row_codes, np.uint8)
    b_row_sf = np.ascontiguousarray(b_row_sf, np.uint8)
    K = a_row_codes.shape[0] * 2
    return lib().orc_grouped_gemm_element(_p(a_row_codes), _p(a_row_sf), float(a_scale), _p(b_row_codes),
                                          _p(b_row_sf), float(b_scale), K)


def silu_mul(y1: np.ndarray) -> np.ndarray:
    y1 = np.ascontiguousarray(y1, np.float64)
    rows, two_i = y1.shape
    h = np.empty((rows, two_i // 2), np.float64)
    lib().orc_silu_mul(_p(y1), rows, two_i // 2, _p(h))
    return h


def finalize(y: np.ndarray, topk_w: np.ndarray, row_of_expanded: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, np.float64)
    topk_w = np.ascontiguousarray(topk_w, np.float32)
    rows = np.ascontiguousarray(row_of_expanded, np.int32)
    T, k = topk_w.shape
    N = y.shape[1]
    out = np.empty((T, N), np.float64)
    lib().orc_finalize(_p(y), _p(topk_w), _p(rows), T, k, N, _p(out))
    return out


# ---------------------------------------------------------------- layouts

def tiled_sf_offset(r: np.ndarray, c: np.ndarray, K: int) -> np.ndarray:
    """Byte offset of scale (row r, column c = k/16) in the tiled layout.

    Rows come in blocks of 128 and scale columns in groups of 4 (64 elements of
    K); each (row block, column group) is one 512-byte atom, atoms ordered row
    block major.  Inside an atom the byte for row r and column c is at
    (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4.
    """
    r = np.asarray(r, np.int64)
    c = np.asarray(c, np.int64)
    atom = (r // 128) * (K // 64) + c // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def untile_sf(sf_tiled: np.ndarray, rows: np.ndarray, K: int) -> np.ndarray:
    """Gather the linear [len(rows), K/16] scales of the given rows out of a tiled buffer."""
    rows = np.asarray(rows, np.int64)
    c = np.arange(K // 16, dtype=np.int64)
    off = tiled_sf_offset(rows[:, None], c[None, :], K)
    return np.asarray(sf_tiled).reshape(-1)[off]


def padded_offsets(expert_offsets: np.ndarray, block: int = 128) -> np.ndarray:
    """Start row of each expert's segment when each segment is padded to ``block`` rows."""
    counts = np.diff(np.asarray(expert_offsets, np.int64))
    padded = ((counts + block - 1) // block) * block
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


# ---------------------------------------------------------------- full layer

@dataclass
class LayerResult:
    topk_id: np.ndarray
    topk_w: np.ndarray
    expert_offsets: np.ndarray
    perm_to_expanded: np.ndarray
    expanded_to_perm: np.ndarray
    x_codes: np.ndarray       # [R, H/2] permuted rows (linear)
    x_sf: np.ndarray          # [R, H/16]
    x_scale: float
    y1: np.ndarray            # [R, 2I] FP64 gate_up output (gate rows first)
    h: np.ndarray             # [R, I] FP64 SiLU-mul output
    h_codes: np.ndarray       # [R, I/2]
    h_sf: np.ndarray          # [R, I/16]
    y2: np.ndarray            # [R, H] FP64 down output
    out: np.ndarray           # [T, H] FP64 FINALIZE result (before the bf16 store)


def quantize_weights(w: np.ndarray):
    """Quantise expert weights float32 [E, N, K] with one dynamic scale per expert."""
    E, N, K = w.shape
    codes = np.empty((E, N, K // 2), np.uint8)
    sf = np.empty((E, N, K // 16), np.uint8)
    scales = np.empty(E, np.float32)
    for e in range(E):
        c, s, sc = quantize_dynamic(w[e])
        codes[e], sf[e], scales[e] = c, s, sc
    return codes, sf, scales


def moe_layer(x: np.ndarray, logits: np.ndarray, w13: tuple, w2: tuple, k: int, h_scale: float | None = None,
              h_override: np.ndarray | None = None) -> LayerResult:
    """The whole MoE layer in the method's order.

    x: float32 [T, H] (values of the bf16 activations); logits: float32 [T, E];
    w13 = (codes [E, 2I, H/2], sf [E, 2I, H/16], scale [E]) with gate rows first;
    w2 = (codes [E, H, I/2], sf [E, H, I/16], scale [E]).
    h_scale: static decode multiplier of the requantised intermediate; when None
    it is taken from this call's own amax(h) (the plainest reading for a test).
    h_override: FP32 h to requantise instead of the oracle's own (staged parity).
    """
    T, H = x.shape
    E = logits.shape[1]
    ids, w = route(logits, k)
    offs, p2e, e2p = permute(ids, E)
    x_codes_tok, x_sf_tok, x_scale = quantize_dynamic(x)
    tok = p2e // k
    x_codes, x_sf = x_codes_tok[tok], x_sf_tok[tok]
    c13, s13, sc13 = w13
    two_i = c13.shape[1]
    y1 = grouped_gemm(x_codes, x_sf, x_scale, c13, s13, sc13, offs, two_i, H)
    h = silu_mul(y1)
    h32 = h.astype(np.float32) if h_override is None else np.ascontiguousarray(h_override, np.float32)
    if h_scale is None:
        h_scale = tensor_scale_from_amax(amax(h32))
    h_codes, h_sf = quantize(h32, h_scale)
    c2, s2, sc2 = w2
    y2 = grouped_gemm(h_codes, h_sf, h_scale, c2, s2, sc2, offs, H, two_i // 2)
    out = finalize(y2, w, e2p)
    return LayerResult(ids, w, offs, p2e, e2p, x_codes, x_sf, x_scale, y1, h, h_codes, h_sf, y2, out)
