"""Parity at the workloads' full sizes, in the launch configuration the benchmark times.

The GPU computes every output; the oracle recomputes sampled outputs one by
one (single GEMM elements for the grouped GEMM, whole token rows for the
layer) from the same seeded inputs.  Routing and quantisation are compared
bit for bit over the full batch.
"""
import numpy as np
import pytest
import torch

import nvfp4_moe_grouped_gb300 as moe
import oracle
from nvfp4_moe_grouped_gb300 import inputs
from tests._helpers import bf16_to_np, counts_to_offsets, padded_rows_of_items, tol_check, untile_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
E, K_TOP, H, I = 256, 8, 6144, 2048


def _expert_host(e, N, K, seed_base):
    """Oracle copy of one expert: the same device draw, copied to the host and quantised by the oracle."""
    w = inputs.expert_weight(e, N, K, seed_base, device=DEV).cpu().numpy()
    return oracle.quantize_dynamic(w)


# ------------------------------------------------------------------ C2: one grouped GEMM

def test_c2_grouped_gemm_none_full_size_sampled():
    N, K, rows = 2048, 6144, 32
    counts = [rows] * E
    offs = counts_to_offsets(counts)
    R = int(offs[-1])
    x = inputs.activations(R, K)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    pad = oracle.padded_offsets(offs)
    e_of_row = np.repeat(np.arange(E), counts)
    dst = (pad[e_of_row] + (np.arange(R) - offs[e_of_row])).astype(np.int32)
    alloc = int(pad[-1])
    codes, sf, s = moe.nvfp4_quantize(x.to(DEV), None, dst_row=torch.from_numpy(dst).to(DEV),
                                      sf_layout=moe.SF_TILED, dst_rows_alloc=alloc)
    assert np.array_equal(codes.cpu().numpy()[dst], xc)
    assert np.array_equal(untile_rows(sf, dst, K), xs)
    wf = inputs.expert_weights(E, N, K, 100, device=DEV)
    pw = moe.prepare_expert_weights(wf, gate_up=False)
    del wf
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_NONE)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    got = bf16_to_np(out)
    rng = np.random.default_rng(0)
    for e in [0, 1, 77, 128, 255]:
        wc, wsf, wsc = _expert_host(e, N, K, 100)
        assert np.float32(wsc) == pw.scale[e].item()
        rs = rng.choice(np.arange(offs[e], offs[e + 1]), 6, replace=False)
        ns = rng.choice(N, 64, replace=False)
        ref = np.array([[oracle.gemm_element(xc[r], xs[r], xsc, wc[n], wsf[n], wsc) for n in ns] for r in rs])
        tol_check(got[dst[rs]][:, ns], ref, f"C2 expert {e}")
    # every routed row of every expert was written (no row left at the zero fill)
    assert np.count_nonzero(np.abs(got[dst]).sum(1) == 0) == 0


# ------------------------------------------------------------------ dense NVFP4 GEMM (the bench's dense workload)

def test_dense_gemm_full_size_sampled():
    """M = N = K = 16384 through dense_gemm_nvfp4 (one group), as `bench.py --workload dense` times it."""
    M = N = K = 16384
    x = inputs.activations(M, K, seed=0, device=DEV)
    codes, sf, s = moe.nvfp4_quantize(x, None, sf_layout=moe.SF_TILED, dst_rows_alloc=M)
    rng = np.random.default_rng(3)
    rs = np.sort(rng.choice(M, 8, replace=False))
    xh = x.cpu().float().numpy()          # exact widening of the bf16 draw, on the host
    del x
    wf = inputs.expert_weights(1, N, K, 900, device=DEV)
    pw = moe.prepare_expert_weights(wf, gate_up=False)
    wh = wf[0].cpu().numpy()
    del wf
    torch.cuda.empty_cache()
    out = moe.dense_gemm_nvfp4(codes, sf, s, pw, M)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    # oracle: per-tensor multipliers from the host copies, then the sampled rows quantised with them
    ns = np.sort(rng.choice(N, 48, replace=False))
    xsc = oracle.tensor_scale_from_amax(oracle.amax(xh))
    wsc = oracle.tensor_scale_from_amax(oracle.amax(wh))
    assert np.float32(xsc) == s.item() and np.float32(wsc) == pw.scale[0].item()
    xc, xsf = oracle.quantize(xh[rs], xsc)
    wc, wsf = oracle.quantize(wh[ns], wsc)
    del xh, wh
    assert np.array_equal(codes[torch.from_numpy(rs).to(DEV)].cpu().numpy(), xc)
    ref = np.array([[oracle.gemm_element(xc[i], xsf[i], xsc, wc[j], wsf[j], wsc) for j in range(len(ns))]
                    for i in range(len(rs))])
    got = bf16_to_np(out[torch.from_numpy(rs).to(DEV)])[:, ns]
    tol_check(got, ref, "dense GEMM 16384^3")
    assert np.count_nonzero(np.abs(bf16_to_np(out[:M:1024])).sum(1) == 0) == 0


# ------------------------------------------------------------------ C3/C4/C5: the layer

@pytest.fixture(scope="module")
def weights():
    w13f = inputs.expert_weights(E, 2 * I, H, inputs.gate_up_seed_base(), device=DEV)
    pw13 = moe.prepare_expert_weights(w13f, gate_up=True)
    del w13f
    w2f = inputs.expert_weights(E, H, I, inputs.down_seed_base(E), device=DEV)
    pw2 = moe.prepare_expert_weights(w2f, gate_up=False)
    del w2f
    torch.cuda.empty_cache()
    return pw13, pw2


def _expert_pair(e, cache):
    if e not in cache:
        cache[e] = (_expert_host(e, 2 * I, H, inputs.gate_up_seed_base()),
                    _expert_host(e, H, I, inputs.down_seed_base(E)))
    return cache[e]


def _oracle_tokens(x, logits, toks, h_scale, cache):
    """Oracle output rows of the chosen tokens (the layer in the method's order) and their h codes."""
    k = K_TOP
    ids, w = oracle.route(logits[toks], k)
    xsc = oracle.tensor_scale_from_amax(oracle.amax(x))
    xc, xsf = oracle.quantize(x[toks], xsc)
    out = np.zeros((len(toks), H))
    hq = {}
    one = np.array([0, 1], np.int32)
    for a, t in enumerate(toks):
        for j in range(k):
            (c13, s13, sc13), (c2, s2, sc2) = _expert_pair(int(ids[a, j]), cache)
            y1 = oracle.grouped_gemm(xc[a:a + 1], xsf[a:a + 1], xsc, c13[None], s13[None],
                                     np.array([sc13], np.float32), one, 2 * I, H)
            h = oracle.silu_mul(y1).astype(np.float32)
            hc, hs = oracle.quantize(h, h_scale)
            hq[(t, j)] = (hc, hs)
            y2 = oracle.grouped_gemm(hc, hs, h_scale, c2[None], s2[None], np.array([sc2], np.float32), one, H, I)
            out[a] += np.float64(w[a, j]) * y2[0]
    return out, hq


def _staged_down_finalize(toks, ids, w, rows, hcodes, hsf_t, h_scale, cache):
    """Oracle down GEMM + FINALIZE of the chosen tokens fed the GPU's own requantised h (codes and scales
    read back from the layer's workspace): the layer's last two steps checked on their own, free of the
    one-grid-step h flips an FP32-vs-FP64 difference before requantisation may cause."""
    one = np.array([0, 1], np.int32)
    out = np.zeros((len(toks), H))
    for a, t in enumerate(toks):
        for j in range(K_TOP):
            _, (c2, s2, sc2) = _expert_pair(int(ids[t, j]), cache)
            r = int(rows[t * K_TOP + j])
            y2 = oracle.grouped_gemm(hcodes[r:r + 1], untile_rows(hsf_t, [r], I), h_scale, c2[None], s2[None],
                                     np.array([sc2], np.float32), one, H, I)
            out[a] += np.float64(w[t, j]) * y2[0]
    return out


def _sample_tokens(T, ids, offs, p2e, n_sample, rng):
    """At least n_sample distinct tokens: the first and the last; for the two busiest experts, the tokens
    owning their routed rows at every 64-row boundary and their last row (the later tiles of a hot
    expert); tokens past T/2; the rest at random."""
    picks = {0, T - 1}
    counts = np.diff(offs)
    for e in np.argsort(-counts, kind="stable")[:2]:
        m = int(counts[e])
        pos = sorted({p for b in range(0, m, 64) for p in (b - 1, b) if 0 <= p < m} | {m - 1})
        picks.update(int(p2e[offs[e] + p]) // K_TOP for p in pos)
    upper = np.arange(T // 2, T)
    picks.update(rng.choice(upper, min(len(upper), 8), replace=False).tolist())
    rest = np.setdiff1d(np.arange(T), np.fromiter(picks, np.int64))
    need = max(0, n_sample - len(picks))
    picks.update(rng.choice(rest, min(need, len(rest)), replace=False).tolist())
    return np.array(sorted(picks))


def _run_layer_case(weights, T, zipf, n_sample, cache):
    pw13, pw2 = weights
    x = inputs.activations(T, H)
    logits = inputs.router_logits(T, E, zipf_s=zipf)
    xf, lf = x.float().numpy(), logits.numpy()
    ids, w = oracle.route(lf, K_TOP)
    offs, p2e, e2p = oracle.permute(ids, E)
    rng = np.random.default_rng(T)
    toks = _sample_tokens(T, ids, offs, p2e, n_sample, rng)
    # static scale of h: the oracle's amax over the first sampled token with a 2x margin (an input both sides share)
    _, hq0 = _oracle_tokens(xf, lf, toks[:1], 1.0, cache)
    fwd = moe.MoeForward(T, E, K_TOP, H, I)
    amax = 0.0
    for (t, j), (hc, hs) in hq0.items():
        amax = max(amax, float(np.abs(oracle.dequantize(hc, hs)).max()))
    h_scale = float(np.float32(2.0 * amax / 2688.0))
    ref, hq = _oracle_tokens(xf, lf, toks, h_scale, cache)
    out = fwd(x.to(DEV), logits.to(DEV), pw13, pw2, h_scale)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    R = T * K_TOP
    # full-batch bit-exact routing, permutation and quantised activations
    assert np.array_equal(fwd.view("topk_id", torch.int32, (T, K_TOP)).cpu().numpy(), ids)
    assert np.array_equal(fwd.view("topk_w", torch.float32, (T, K_TOP)).cpu().numpy(), w)
    assert np.array_equal(fwd.view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy(), offs)
    assert np.array_equal(fwd.view("perm_to_expanded", torch.int32, (R,)).cpu().numpy(), p2e)
    rows = padded_rows_of_items(offs.astype(np.int64), ids.reshape(-1), e2p)
    assert np.array_equal(fwd.view("expanded_to_row", torch.int32, (R,)).cpu().numpy(), rows)
    P = fwd.layout.padded_rows
    xcodes = fwd.view("x_codes", torch.uint8, (P, H // 2)).cpu().numpy()
    xc, xsf, _ = oracle.quantize_dynamic(xf)
    tok_of_item = np.arange(R) // K_TOP
    assert np.array_equal(xcodes[rows], xc[tok_of_item])
    assert np.array_equal(untile_rows(fwd.view("x_sf", torch.uint8, (P * H // 16,)), rows, H), xsf[tok_of_item])
    # sampled token rows of the layer output
    got = bf16_to_np(out)[toks]
    hcodes = fwd.view("h_codes", torch.uint8, (P, I // 2)).cpu().numpy()
    hsf_t = fwd.view("h_sf", torch.uint8, (P * I // 16,))
    # h: decoded GPU codes against the oracle's; a code may differ by one grid step only where the FP32
    # value before requantisation sits at a rounding boundary (rate bounded below)
    flips = 0
    for (t, j), (hc, hs) in hq.items():
        r = rows[t * K_TOP + j]
        g = oracle.dequantize(hcodes[r:r + 1], untile_rows(hsf_t, [r], I))
        flips += int(np.count_nonzero(g != oracle.dequantize(hc, hs)))
    n_h = len(hq) * I
    rate = flips / n_h
    # down GEMM + FINALIZE from the GPU's own h: elementwise on every sampled row
    staged = _staged_down_finalize(toks, ids, w, rows, hcodes, hsf_t, h_scale, cache)
    worst = tol_check(got, staged, f"layer T={T} zipf={zipf}: down+FINALIZE from the GPU's h")
    # the independent end-to-end comparison: relative Frobenius error, elementwise when no h code flipped
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    print(f"\nlayer T={T} zipf={zipf}: {len(toks)} tokens sampled, h code flips {flips}/{n_h} = {rate:.2e}, "
          f"staged worst |err|/bound-scale {worst:.2e}, end-to-end relative Frobenius {rel:.2e}")
    assert rate < 2e-3, rate
    assert rel < 1e-2, rel
    if flips == 0:
        tol_check(got, ref, f"layer T={T}")
    return rel, flips


@pytest.fixture(scope="module")
def oracle_cache():
    return {}


@pytest.mark.parametrize("T,zipf", [(1024, None), (1024, 1.1), (128, None), (128, 1.1), (256, None), (256, 1.1),
                                    (512, None), (512, 1.1)])
def test_layer_decode_sweep_full_size_sampled(weights, oracle_cache, T, zipf):
    """The decode sweep T in {128, 256, 512, 1024} x {uniform, Zipf(1.1)}; T=1024 uniform is the 1024-token
    layer.  At least 32 tokens per case."""
    _run_layer_case(weights, T, zipf, 32, oracle_cache)


def test_layer_prefill_full_size_sampled(weights, oracle_cache):
    """The 16384-token prefill layer: at least 32 tokens, including tokens at every 64-row boundary of the two
    busiest experts and tokens past T/2; each sampled row covers every FINALIZE column chunk."""
    _run_layer_case(weights, 16384, None, 32, oracle_cache)
