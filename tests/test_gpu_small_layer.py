"""The single-launch path for small layers (T * k <= 64, E <= 64, H <= 1024, I <= 512, E * I <= 4096).

moe_forward runs such a layer as one kernel, one cluster of CTAs: each CTA routes every token itself;
gate_up, SiLU and the h requantisation are dealt out in (expert, 32 h columns) units; after the cluster
barrier each CTA runs down and the slot sum for its share of the output columns.  It must give what the
staged kernels give: routing, permutation and quantised x bit for bit (the same rule, the same quantiser
arithmetic), h and the output within the layer tolerances (only the order of the FP32 sums differs), all
against the oracle too.  Debug flag bit 2 runs the staged kernels on the same input for the comparison.
"""
import numpy as np
import pytest
import torch

import nvfp4_moe_grouped_gb300 as moe
import oracle
from nvfp4_moe_grouped_gb300 import inputs
from tests._helpers import bf16_to_np, padded_rows_of_items, tol_check, untile_rows
from tests.test_gpu_kernels import _assert_rare_adjacent_flips, _check_layer, _layer_case

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [
    (16, 8, 2, 256, 128),     # the 16-token, 8-expert, top-2 layer
    (64, 8, 1, 1024, 512),    # T * k, H, I and E * I at their limits
    (64, 64, 1, 256, 64),     # E at its limit, I one unit pair
    (32, 4, 2, 384, 64),      # partial 256-element K tiles in both weight matrices
    (8, 2, 2, 256, 128),      # every expert selected (k = E)
    (5, 1, 1, 128, 64),       # one expert
    (21, 16, 3, 512, 192),    # ragged: 63 items, I not a multiple of 128
]


def _run(fwd, x, logits, pw13, pw2, h_scale, staged):
    moe.debug_set_flags(4 if staged else 0)
    try:
        out = fwd(x, logits, pw13, pw2, h_scale)
        torch.cuda.synchronize()
    finally:
        moe.debug_set_flags(0)
    assert moe.device_error() == (0, 0)
    return out.clone(), fwd.ws.clone()


def _intermediates(fwd, ws, T, E, k, H, I):
    L = fwd.layout
    P = L.padded_rows
    R = T * k

    def v(name, dtype, shape):
        off = getattr(L, name)
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + n].view(dtype).view(shape).cpu().numpy()
    return {
        "topk_id": v("topk_id", torch.int32, (T, k)), "topk_w": v("topk_w", torch.float32, (T, k)),
        "offs": v("expert_offsets", torch.int32, (E + 1,)), "p2e": v("perm_to_expanded", torch.int32, (R,)),
        "e2p": v("expanded_to_perm", torch.int32, (R,)), "e2r": v("expanded_to_row", torch.int32, (R,)),
        "x_scale": v("x_scale", torch.float32, (1,)), "h_scale": v("h_scale", torch.float32, (1,)),
        "x_codes": v("x_codes", torch.uint8, (P, H // 2)), "x_sf": ws[L.x_sf:L.x_sf + P * H // 16],
        "h_codes": v("h_codes", torch.uint8, (P, I // 2)), "h_sf": ws[L.h_sf:L.h_sf + P * I // 16],
    }


@pytest.mark.parametrize("T,E,k,H,I", SHAPES)
def test_small_layer_matches_oracle_and_staged_path(T, E, k, H, I):
    assert moe.forward_kernel_count(T, E, k, H, I) == 1
    x, logits, w13f, w2f = _layer_case(T, E, k, H, I)
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits.numpy(), w13, w2, k)
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I)
    xd, ld = x.to(DEV), logits.to(DEV)
    small, ws_small = _run(fwd, xd, ld, pw13, pw2, h_scale, staged=False)
    # against the oracle: every intermediate as the staged layer is checked
    _check_layer(fwd, small, ref, h_scale, T, E, k, H, I)
    staged, ws_staged = _run(fwd, xd, ld, pw13, pw2, h_scale, staged=True)
    a = _intermediates(fwd, ws_small, T, E, k, H, I)
    b = _intermediates(fwd, ws_staged, T, E, k, H, I)
    # the same routing, permutation, multipliers and quantised x rows, bit for bit
    for name in ("topk_id", "topk_w", "offs", "p2e", "e2p", "e2r", "x_scale", "h_scale"):
        assert np.array_equal(a[name], b[name]), name
    rows = padded_rows_of_items(ref.expert_offsets.astype(np.int64), ref.topk_id.reshape(-1), ref.expanded_to_perm)
    perm_rows = rows[ref.perm_to_expanded]
    assert np.array_equal(a["x_codes"][perm_rows], b["x_codes"][perm_rows])
    assert np.array_equal(untile_rows(a["x_sf"], perm_rows, H), untile_rows(b["x_sf"], perm_rows, H))
    # h: the two paths sum in different orders, so a code may sit one grid step apart, rarely
    ha = oracle.dequantize(a["h_codes"][perm_rows], untile_rows(a["h_sf"], perm_rows, I))
    hb = oracle.dequantize(b["h_codes"][perm_rows], untile_rows(b["h_sf"], perm_rows, I))
    flips = _assert_rare_adjacent_flips(ha, hb)
    got, other = bf16_to_np(small), bf16_to_np(staged)
    assert np.linalg.norm(got - other) / np.linalg.norm(other) < 1e-2
    if not flips.any():
        tol_check(got, other, "single-launch vs staged")


def test_small_layer_hot_expert_takes_several_passes():
    """Every token routed to the same two experts: 32 rows each, four passes of eight rows in each of their
    units, the other experts' units idle; every CTA still writes its output columns."""
    T, E, k, H, I = 32, 16, 2, 256, 128
    x, _, w13f, w2f = _layer_case(T, E, k, H, I)
    logits = inputs.router_logits(T, E, seed=5)
    logits[:, 3] += 50.0
    logits[:, 11] += 40.0
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits.numpy(), w13, w2, k)
    assert np.bincount(ref.topk_id.reshape(-1), minlength=E)[[3, 11]].tolist() == [32, 32]
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I)
    out = fwd(x.to(DEV), logits.to(DEV), pw13, pw2, h_scale)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    _check_layer(fwd, out, ref, h_scale, T, E, k, H, I)


def test_small_layer_graph_replays():
    """Replays of the captured single-launch layer rewrite the whole output every time (no state carries
    from one launch to the next); refilled inputs give the eager result on them."""
    T, E, k, H, I = 16, 8, 2, 256, 128
    x, logits, w13f, w2f = _layer_case(T, E, k, H, I)
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits.numpy(), w13, w2, k)
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I)
    xd, ld = x.to(DEV), logits.to(DEV)
    g = fwd.graph(xd, ld, pw13, pw2, h_scale, stage_events=False)
    for _ in range(3):
        out = g.launch()
        torch.cuda.synchronize()
        _check_layer(fwd, out, ref, h_scale, T, E, k, H, I)
    # the output buffer cleared between replays is rewritten by the next one
    out.zero_()
    out = g.launch()
    torch.cuda.synchronize()
    assert np.linalg.norm(bf16_to_np(out) - ref.out) / np.linalg.norm(ref.out) < 1e-2
    x2 = inputs.activations(T, H, seed=77)
    l2 = inputs.router_logits(T, E, seed=78)
    xd.copy_(x2.to(DEV))
    ld.copy_(l2.to(DEV))
    out = g.launch()
    torch.cuda.synchronize()
    ref2 = oracle.moe_layer(x2.float().numpy(), l2.numpy(), w13, w2, k, h_scale=h_scale)
    assert np.linalg.norm(bf16_to_np(out) - ref2.out) / np.linalg.norm(ref2.out) < 1e-2
    g.close()
    assert moe.device_error() == (0, 0)
