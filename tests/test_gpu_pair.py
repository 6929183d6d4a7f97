"""Parity of the CTA-pair grouped GEMM (the prefill-regime kernel) against the oracle.

Launches whose routed-row allocation implies more than 48 rows per expert and whose N is a multiple of 256
run on CTA pairs: 256 weight rows x up to 192 routed rows per unit, M = 256 MMAs over two SMs.  The row
counts below put experts on every edge of that tiling: 1-row experts, 31/32/33 rows (MMA N rounding), 96
and 128 (half and full one-CTA tiles), 191/192/193 (one full pair unit and a one-row second unit), 250-500
(units that start 64 rows into a 128-row scale block).  Each case is also run with debug flag bit 1, which
keeps the one-CTA 128-row tile, so the two kernels are checked on the same input.
"""
import numpy as np
import pytest
import torch

import nvfp4_moe_grouped_gb300 as moe
import oracle
from nvfp4_moe_grouped_gb300 import inputs
from tests._helpers import bf16_to_np, counts_to_offsets, tol_check, untile_rows
from tests.test_gpu_kernels import _assert_rare_adjacent_flips, _routed_operand, _silu_case

pytestmark = pytest.mark.gpu
DEV = "cuda"

EDGE_COUNTS = [1, 31, 32, 33, 64, 96, 127, 128, 129, 191, 192, 193, 250, 256, 300, 384, 385, 500, 0, 160]


def _pair_regime(offs):
    pad = oracle.padded_offsets(offs.astype(np.int64))
    E = len(offs) - 1
    alloc = ((max(128, int(pad[-1])) + 127) // 128) * 128
    return (alloc - 127 * E) // E > 48


def _both_kernels(launch):
    """(pair kernel result, one-CTA kernel result) of `launch`, each checked for device errors."""
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    a = launch()
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    moe.debug_set_flags(2)
    try:
        b = launch()
        torch.cuda.synchronize()
    finally:
        moe.debug_set_flags(0)
    assert moe.device_error() == (0, 0)
    return a, b


@pytest.mark.parametrize("counts,N,K", [(EDGE_COUNTS, 512, 512), ([129, 191, 192, 193, 250, 1], 256, 320),
                                        ([700, 3, 1000], 768, 1024)])
def test_pair_none_matches_oracle(counts, N, K):
    E = len(counts)
    offs = counts_to_offsets(counts)
    assert _pair_regime(offs)
    R = int(offs[-1])
    x = inputs.activations(R, K, seed=R + K + 1)
    w = inputs.expert_weights(E, N, K, 300 + N)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *oracle.quantize_weights(w.numpy()), offs, N, K)
    codes, sf, s, dst = _routed_operand(x, offs)
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=False)
    o = torch.from_numpy(offs).to(DEV)
    pair, one = _both_kernels(lambda: moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, o, moe.EPI_NONE))
    tol_check(bf16_to_np(pair)[dst], ref, "pair NONE")
    tol_check(bf16_to_np(one)[dst], ref, "one-CTA NONE")


@pytest.mark.parametrize("counts,I,H", [(EDGE_COUNTS, 256, 512), ([193, 64, 385], 128, 320)])
def test_pair_silu_mul_quant(counts, I, H):
    offs, x, w13, h_ref, h_scale = _silu_case(counts, I, H, 21 + I)
    assert _pair_regime(offs)
    codes, sf, s, dst = _routed_operand(x, offs)
    pw = moe.prepare_expert_weights(w13.to(DEV), gate_up=True)
    o = torch.from_numpy(offs).to(DEV)

    def launch():
        h_f32 = torch.zeros(codes.shape[0], I, dtype=torch.float32, device=DEV)
        hs_out = torch.zeros(1, dtype=torch.float32, device=DEV)
        hc, hsf = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, o, moe.EPI_SILU_MUL_QUANT, h_scale=h_scale,
                                             h_f32=h_f32, h_scale_out=hs_out)
        return h_f32, hc, hsf, hs_out

    for name, (h_f32, hc, hsf, hs_out) in zip(("pair", "one-CTA"), _both_kernels(launch)):
        assert hs_out.item() == np.float32(h_scale)
        tol_check(h_f32.cpu().numpy()[dst], h_ref, f"{name} SiLU-mul h")
        hc_ref, hs_ref = oracle.quantize(h_ref.astype(np.float32), h_scale)
        got = oracle.dequantize(hc.cpu().numpy()[dst], untile_rows(hsf, dst, I))
        _assert_rare_adjacent_flips(got, oracle.dequantize(hc_ref, hs_ref))
        # the GPU's codes are exactly the oracle's requantisation of the GPU's own FP32 h
        hc_own, hs_own = oracle.quantize(h_f32.cpu().numpy()[dst], h_scale)
        assert np.array_equal(hc.cpu().numpy()[dst], hc_own), name
        assert np.array_equal(untile_rows(hsf, dst, I), hs_own), name


@pytest.mark.parametrize("T,E,k,H,I", [(1000, 8, 2, 512, 256), (3000, 16, 4, 768, 128), (20000, 4, 2, 1024, 64)])
def test_pair_finalize_matches_oracle(T, E, k, H, I):
    """FINALIZE on pairs; T = 20000 at H = 1024 takes the column-chunked unit order (two 256-column pairs
    per chunk keep the live accumulator within 64 MiB)."""
    logits = inputs.router_logits(T, E, seed=T + 3).numpy()
    ids, w = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    assert _pair_regime(offs)
    g = torch.Generator().manual_seed(T + 1)
    h = (torch.randn(T * k, I, generator=g) * 0.3).numpy()
    hc, hs, hsc = oracle.quantize_dynamic(h)
    w2 = inputs.expert_weights(E, H, I, 800)
    ref = oracle.finalize(oracle.grouped_gemm(hc, hs, hsc, *oracle.quantize_weights(w2.numpy()), offs, H, I), w, e2p)
    codes, sf, s, dst = _routed_operand(torch.from_numpy(h), offs.astype(np.int64))
    pw = moe.prepare_expert_weights(w2.to(DEV), gate_up=False)
    o, p, wt = torch.from_numpy(offs).to(DEV), torch.from_numpy(p2e).to(DEV), torch.from_numpy(w).to(DEV)
    pair, one = _both_kernels(lambda: moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, o, moe.EPI_FINALIZE,
                                                                 perm_to_expanded=p, topk_w=wt, T=T, k=k))
    tol_check(bf16_to_np(pair), ref, "pair FINALIZE")
    tol_check(bf16_to_np(one), ref, "one-CTA FINALIZE")


def test_pair_timeout_path_reports_and_recovers():
    """A stage the producers never fill, on a pair launch: both CTAs' bounded waits give up, the launch
    reports MOE_ERR_TIMEOUT, and the next launch on the same context is correct."""
    counts = [200, 150, 300]
    N, K = 256, 512
    offs = counts_to_offsets(counts)
    assert _pair_regime(offs)
    x = inputs.activations(int(offs[-1]), K, seed=2)
    w = inputs.expert_weights(len(counts), N, K, 4)
    codes, sf, s, dst = _routed_operand(x, offs)
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=False)
    o = torch.from_numpy(offs).to(DEV)
    torch.cuda.synchronize()
    moe.device_error()
    moe.set_wait_timeout_ns(50_000_000)
    moe.debug_set_flags(1)
    try:
        moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, o, moe.EPI_NONE)
        code, _ = moe.device_error()
    finally:
        moe.debug_set_flags(0)
        moe.set_wait_timeout_ns(0)
    assert code == 6  # MOE_ERR_TIMEOUT
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, o, moe.EPI_NONE)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *oracle.quantize_weights(w.numpy()), offs, N, K)
    tol_check(bf16_to_np(out)[dst], ref, "pair after timeout")
