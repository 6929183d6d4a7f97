"""Pins of the oracle's routing, permutation, GEMM, SiLU-mul, FINALIZE and full layer.

Each check compares against something other than the oracle's own code: a
library sort, brute force over subsets, closed forms, an FP64 numpy
restatement of the layer written from the definitions, or special cases (an
identity expert, k = E, k = 1) that reduce to textbook operations.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from nvfp4_moe_grouped_gb300 import inputs


# ------------------------------------------------------------------ routing

def test_route_matches_brute_force_subsets_c1():
    T, E, k = 16, 8, 2
    logits = inputs.router_logits(T, E).numpy()
    ids, w = oracle.route(logits, k)
    for t in range(T):
        best = max(itertools.combinations(range(E), k), key=lambda s: (sum(logits[t, list(s)]), [-i for i in s]))
        assert set(ids[t]) == set(best)
        # slot order: descending logit, ties to the lower index
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert list(ids[t]) == order


def test_route_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    ids, w = oracle.route(logits, 3)
    assert list(ids[0]) == [1, 2, 4]
    assert w[0, 0] == w[0, 1] == w[0, 2]
    assert abs(float(w[0].sum()) - 1.0) < 1e-6


def test_route_weights_invariants():
    T, E, k = 256, 256, 8
    logits = inputs.router_logits(T, E).numpy()
    ids, w = oracle.route(logits, k)
    for t in range(T):
        assert len(set(ids[t])) == k
        assert np.all(np.diff(w[t].astype(np.float64)) <= 0)
        s = float(np.sum(w[t].astype(np.float64)))
        assert abs(s - 1.0) <= 8 * 2.0 ** -24 * k
    # softmax restricted to the selected logits, FP64 reference
    sel = np.take_along_axis(logits, ids, 1).astype(np.float64)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(w - ref)) < 4e-7


def test_route_k_equals_e_is_plain_softmax():
    T, E = 32, 16
    logits = inputs.router_logits(T, E, seed=11).numpy()
    ids, w = oracle.route(logits, E)
    full = torch.softmax(torch.tensor(logits, dtype=torch.float64), dim=1).numpy()
    got = np.zeros_like(full)
    np.put_along_axis(got, ids, w.astype(np.float64), 1)
    assert np.max(np.abs(got - full)) < 4e-7


# ------------------------------------------------------------------ permutation

@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (300, 256, 8), (5, 64, 3), (1, 4, 4)])
def test_permute_is_stable_counting_sort(T, E, k):
    logits = inputs.router_logits(T, E, seed=T + E).numpy()
    ids, _ = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    # library stable sort by expert of the expanded index
    ref = np.argsort(flat, kind="stable")
    assert np.array_equal(p2e, ref)
    assert np.array_equal(e2p[p2e], np.arange(T * k))
    assert np.array_equal(p2e[e2p], np.arange(T * k))
    hist = np.bincount(flat, minlength=E)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(hist)]))


def test_zipf_logits_skew_expert_load():
    T, E, k = 1024, 256, 8
    logits = inputs.router_logits(T, E, zipf_s=1.1).numpy()
    ids, _ = oracle.route(logits, k)
    load = np.sort(np.bincount(ids.reshape(-1), minlength=E))[::-1]
    assert load[0] > 4 * (T * k / E)      # the most popular expert is far above uniform
    assert load.sum() == T * k


# ------------------------------------------------------------------ GEMM

def _quant_weights(E, N, K, seed_base):
    w = inputs.expert_weights(E, N, K, seed_base).numpy()
    return oracle.quantize_weights(w)


def _dequant_np(codes, sf):
    """Independent numpy dequantisation (grid table + torch float8 decode)."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float64)
    lo = grid[codes & 15]
    hi = grid[codes >> 4]
    vals = np.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    scale = torch.tensor(sf).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(scale, 16, axis=-1)


def test_grouped_gemm_matches_numpy_fp64_matmul():
    E, N, K = 4, 64, 128
    rng = np.random.default_rng(0)
    counts = np.array([3, 0, 17, 9])
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = rng.standard_normal((int(offs[-1]), K)).astype(np.float32)
    a_codes, a_sf, a_s = oracle.quantize_dynamic(x)
    b_codes, b_sf, b_s = _quant_weights(E, N, K, 40)
    got = oracle.grouped_gemm(a_codes, a_sf, a_s, b_codes, b_sf, b_s, offs, N, K)
    A = _dequant_np(a_codes, a_sf) * a_s
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        B = _dequant_np(b_codes[e], b_sf[e]) * np.float64(b_s[e])
        ref = A[r0:r1] @ B.T
        assert np.allclose(got[r0:r1], ref, rtol=1e-12, atol=1e-12)
    # one element through the single-element path
    r, n, e = 5, 7, 2
    el = oracle.gemm_element(a_codes[r], a_sf[r], a_s, b_codes[e, n], b_sf[e, n], b_s[e])
    assert abs(el - got[r, n]) <= 1e-12 * max(1.0, abs(got[r, n]))


def test_identity_expert_reproduces_its_input():
    K = 64
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    rng = np.random.default_rng(1)
    x = grid[rng.integers(0, 8, (10, K))] * rng.choice([-1, 1], (10, K)).astype(np.float32)
    x[:, ::16] = 6.0  # every block's amax is 6 -> block scale 1 under s = 1
    a_codes, a_sf = oracle.quantize(x, 1.0)
    # the identity expert: code 2 (= 1.0) on the diagonal, every scale 1.0 (e4m3 0x38)
    b_codes = np.zeros((1, K, K // 2), np.uint8)
    for n in range(K):
        b_codes[0, n, n // 2] = 2 if n % 2 == 0 else 2 << 4
    b_sf = np.full((1, K, K // 16), 0x38, np.uint8)
    assert oracle.e4m3_decode(0x38) == 1.0
    y = oracle.grouped_gemm(a_codes, a_sf, 1.0, b_codes, b_sf, np.ones(1, np.float32),
                            np.array([0, 10], np.int32), K, K)
    assert np.array_equal(y, x.astype(np.float64))


# ------------------------------------------------------------------ SiLU-mul / FINALIZE

def test_silu_mul_closed_forms():
    y1 = np.array([[0.0, 5.0, 3.0, 2.0], [40.0, -40.0, 1.5, 1.0]], np.float64)
    h = oracle.silu_mul(y1)
    assert h[0, 0] == 0.0                                 # silu(0) = 0
    assert abs(h[0, 1] - 5.0 / (1 + math.exp(-5.0)) * 2.0) < 1e-15
    assert abs(h[1, 0] - 40.0 * 1.5) < 1e-12              # silu(g) -> g for large g
    assert abs(h[1, 1]) < 1e-15                            # silu(g) -> 0 for very negative g
    ref = torch.nn.functional.silu(torch.tensor(y1[:, :2])) * torch.tensor(y1[:, 2:])
    assert np.allclose(h, ref.numpy(), rtol=1e-15, atol=0)


def test_finalize_k1_is_inverse_permutation_gather():
    T, H = 9, 6
    rng = np.random.default_rng(2)
    y = rng.standard_normal((T, H))
    perm = rng.permutation(T).astype(np.int32)
    w = np.ones((T, 1), np.float32)
    out = oracle.finalize(y, w, perm[:, None].copy())
    assert np.array_equal(out, y[perm])


def test_finalize_identity_experts_recover_input():
    T, E, k, H = 12, 4, 3, 32
    logits = inputs.router_logits(T, E, seed=3).numpy()
    ids, w = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    x = np.random.default_rng(4).standard_normal((T, H))
    y = x[p2e // k]                                       # identity experts
    out = oracle.finalize(y, w, e2p)
    wsum = w.astype(np.float64).sum(1, keepdims=True)
    assert np.allclose(out, x * wsum, rtol=0, atol=1e-14)
    assert np.allclose(out, x, atol=1e-6 * np.abs(x).max())


# ------------------------------------------------------------------ full layer

def _layer_numpy_fp64(x, logits, k, w13, w2, h_scale):
    """The layer restated from its definitions with numpy, FP64 sums, no permutation."""
    T, H = x.shape
    order = [sorted(range(logits.shape[1]), key=lambda e: (-logits[t, e], e))[:k] for t in range(T)]
    xc, xs, xsc = oracle.quantize_dynamic(x)
    X = _dequant_np(xc, xs) * xsc
    c13, s13, sc13 = w13
    c2, s2, sc2 = w2
    I = c13.shape[1] // 2
    out = np.zeros((T, H))
    ids, w = oracle.route(logits, k)
    for t in range(T):
        assert list(ids[t]) == order[t]
        for j, e in enumerate(order[t]):
            W13 = _dequant_np(c13[e], s13[e]) * np.float64(sc13[e])
            y1 = W13 @ X[t]
            g, u = y1[:I], y1[I:]
            h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
            hc, hs = oracle.quantize(h[None, :], h_scale)
            Hq = _dequant_np(hc, hs)[0] * h_scale
            W2 = _dequant_np(c2[e], s2[e]) * np.float64(sc2[e])
            out[t] += np.float64(w[t, j]) * (W2 @ Hq)
    return out


def test_full_layer_c1_against_fp64_restatement():
    T, E, k, H, I = 16, 8, 2, 256, 128
    x = inputs.activations(T, H).float().numpy()
    logits = inputs.router_logits(T, E).numpy()
    w13 = _quant_weights(E, 2 * I, H, inputs.gate_up_seed_base())
    w2 = _quant_weights(E, H, I, inputs.down_seed_base(E))
    res = oracle.moe_layer(x, logits, w13, w2, k)
    h_scale = oracle.tensor_scale_from_amax(oracle.amax(res.h.astype(np.float32)))
    ref = _layer_numpy_fp64(x, logits, k, w13, w2, h_scale)
    # FP64 on both sides; the only difference is summation order (and the same
    # FP32 h decides the same codes), so agreement is to FP64 rounding.
    assert np.allclose(res.out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    assert np.abs(ref).max() > 0


# ------------------------------------------------------------------ router logits (reading R8)

def _bf16_round(a):
    """Round float32 values to bf16 (nearest even) and back, so they are exact bf16 values."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def test_router_logits_one_hot_gate_selects_columns():
    """Expert e's gate row is the unit vector of hidden index j(e): logits are the selected x columns, exactly."""
    rng = np.random.default_rng(5)
    T, H, E = 7, 96, 12
    x = _bf16_round(rng.standard_normal((T, H)).astype(np.float32))
    cols = rng.choice(H, E, replace=False)
    w = np.zeros((E, H), np.float32)
    w[np.arange(E), cols] = 1.0
    assert np.array_equal(oracle.router_logits(x, w), x[:, cols])


def test_router_logits_constant_inputs_closed_form():
    """x = 1 everywhere, gate row e constant c_e: logit = H * c_e (exact in FP32 for these c_e)."""
    T, H, E = 3, 640, 5
    c = np.array([0.5, -0.25, 1.5, 0.0, -3.0], np.float32)
    x = np.ones((T, H), np.float32)
    w = np.repeat(c[:, None], H, axis=1)
    assert np.array_equal(oracle.router_logits(x, w), np.tile(H * c, (T, 1)).astype(np.float32))


def test_router_logits_brute_force_small_integers():
    """Small integer inputs: every product and sum is exact, checked against plain Python loops."""
    rng = np.random.default_rng(9)
    T, H, E = 4, 9, 6
    x = rng.integers(-8, 9, (T, H)).astype(np.float32)
    w = rng.integers(-8, 9, (E, H)).astype(np.float32)
    ref = [[sum(int(x[t, h]) * int(w[e, h]) for h in range(H)) for e in range(E)] for t in range(T)]
    assert np.array_equal(oracle.router_logits(x, w), np.array(ref, np.float32))


def test_router_logits_single_rounding_to_fp32():
    """The sum is formed in FP64 and rounded once: 1 + 2^-30 - 1 keeps the 2^-30 an FP32 running sum would lose."""
    x = np.array([[1.0, 2.0 ** -15, -1.0]], np.float32)
    w = np.array([[1.0, 2.0 ** -15, 1.0]], np.float32)
    assert oracle.router_logits(x, w)[0, 0] == np.float32(2.0 ** -30)
