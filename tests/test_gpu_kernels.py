"""GPU parity of every kernel against the CPU oracle, through the C ABI.

Integer and byte work (routing ids, router weights, permutation, NVFP4 codes
and scales) must match bit for bit; GEMM, SiLU and FINALIZE outputs must stay
within |gpu - ref| <= 1e-2 (|ref| + 1e-3 rms(ref)) elementwise.  Sizes span
several tiles, ragged expert counts (0, 1, 31, 33, 128, 129, ...) and the
partial last K tile.
"""
import numpy as np
import pytest
import torch

import nvfp4_moe_grouped_gb300 as moe
import oracle
from nvfp4_moe_grouped_gb300 import inputs
from tests._helpers import (bf16_to_np, counts_to_offsets, padded_rows_of_items, tol_check, unblock_weights,
                            untile_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tie_logits(T, E, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 6, (T, E), generator=g).float() * 0.5).numpy()


def _signed_zero_logits(T, E, seed):
    """Mostly -0.0 and +0.0 (equal logits: the lower index goes first, whatever the sign), some -inf and a few
    0.5, so the selected sets mix zeros of both signs and the weights see differences of zeros."""
    g = torch.Generator().manual_seed(seed)
    vals = torch.tensor([-float("inf"), -0.0, 0.0, 0.5])
    pick = torch.multinomial(torch.tensor([0.3, 0.33, 0.33, 0.04]), T * E, replacement=True, generator=g)
    return vals[pick].view(T, E).numpy()


# ------------------------------------------------------------------ routing / permutation

@pytest.mark.parametrize("T,E,k,kind", [(16, 8, 2, "normal"), (300, 256, 8, "normal"), (1024, 256, 8, "zipf"),
                                        (5, 64, 3, "normal"), (1, 4, 4, "normal"), (777, 256, 8, "ties"),
                                        (64, 1000, 32, "normal"), (4096, 256, 8, "normal"),
                                        (500, 256, 8, "zeros"), (100, 1000, 32, "zeros"), (40, 1000, 4, "zeros"),
                                        (3000, 96, 1, "normal"), (257, 33, 5, "ties")])
def test_route_permute_bitexact(T, E, k, kind):
    if kind == "zipf":
        logits = inputs.router_logits(T, E, zipf_s=1.1).numpy()
    elif kind == "ties":
        logits = _tie_logits(T, E, 9)
    elif kind == "zeros":
        logits = _signed_zero_logits(T, E, 11)
        assert (np.signbit(logits) & (logits == 0)).any() and ((~np.signbit(logits)) & (logits == 0)).any()
    else:
        logits = inputs.router_logits(T, E, seed=T * 7 + E).numpy()
    ids, w = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    r = moe.moe_route_permute(torch.from_numpy(logits).to(DEV), k)
    torch.cuda.synchronize()
    assert np.array_equal(r.topk_id.cpu().numpy(), ids)
    assert np.array_equal(r.topk_w.cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r.expert_offsets.cpu().numpy(), offs)
    assert np.array_equal(r.perm_to_expanded.cpu().numpy(), p2e)
    assert np.array_equal(r.expanded_to_perm.cpu().numpy(), e2p)
    rows = padded_rows_of_items(offs.astype(np.int64), ids.reshape(-1), e2p)
    assert np.array_equal(r.expanded_to_row.cpu().numpy(), rows)


def test_route_permute_is_deterministic():
    T, E, k = 2048, 256, 8
    logits = torch.from_numpy(inputs.router_logits(T, E, seed=5).numpy()).to(DEV)
    a = moe.moe_route_permute(logits, k)
    b = moe.moe_route_permute(logits, k)
    for f in ("topk_id", "topk_w", "expert_offsets", "perm_to_expanded", "expanded_to_perm", "expanded_to_row"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


# ------------------------------------------------------------------ quantisation

@pytest.mark.parametrize("rows,K", [(1, 16), (37, 256), (300, 6144), (128, 2048)])
def test_quantize_linear_bf16_bitexact(rows, K):
    x = inputs.activations(rows, K, seed=rows + K)
    codes_ref, sf_ref, s_ref = oracle.quantize_dynamic(x.float().numpy())
    codes, sf, s = moe.nvfp4_quantize(x.to(DEV))
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    assert s.cpu().numpy()[0] == np.float32(s_ref)


@pytest.mark.parametrize("dtype,groups,rows,K", [(torch.float32, 1, 96, 512), (torch.bfloat16, 4, 200, 320),
                                                  (torch.float32, 3, 129, 1024), (torch.bfloat16, 5, 5, 64)])
def test_quantize_dynamic_per_group_linear_bitexact(dtype, groups, rows, K):
    """Dynamic decode multipliers per group of rows (each group's own amax) in the linear layout, from FP32
    and bf16 input: every group's codes, scales and multiplier as the oracle quantises that group alone.
    One group is all zeros (multiplier 1, zero codes and scales)."""
    x = inputs.activations(rows * groups, K, seed=rows + groups).float() * 3.0
    if groups > 1:
        x[rows:2 * rows] = 0.0
    x = x.to(dtype)
    codes, sf, s = moe.nvfp4_quantize(x.to(DEV), None, groups=groups)
    codes, sf, s = codes.cpu().numpy(), sf.cpu().numpy(), s.cpu().numpy()
    for g in range(groups):
        xr = x[g * rows:(g + 1) * rows].float().numpy()
        c_ref, sf_ref, s_ref = oracle.quantize_dynamic(xr)
        assert s[g] == np.float32(s_ref), g
        assert np.array_equal(codes[g * rows:(g + 1) * rows], c_ref), g
        assert np.array_equal(sf[g * rows:(g + 1) * rows], sf_ref), g


def test_quantize_static_scale_and_zero_rows():
    x = inputs.activations(64, 512, seed=3).float()
    x[5] = 0.0
    x[7, :16] = 1e-30
    s = 0.01
    codes_ref, sf_ref = oracle.quantize(x.numpy(), s)
    codes, sf, _ = moe.nvfp4_quantize(x.to(DEV), torch.tensor([s], dtype=torch.float32, device=DEV))
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)


def test_quantize_rounding_boundaries_bitexact():
    """Every e2m1 rounding boundary (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5), one FP32 step either side of it,
    the grid values, signed zeros, tiny and subnormal values and products above 6 (saturation), in blocks
    whose decoded scale is exactly 1 (block max 6 at s = 1) or rounds below the block max (6.2, 7.5)."""
    f32 = np.float32
    bounds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    probes = []
    for b in bounds:
        b = f32(b)
        probes += [b, np.nextafter(b, f32(0)), np.nextafter(b, f32(np.inf))]
    probes += [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 0.0, 1e-30, 1e-40, 1e-45, 0.2499, 5.999]
    probes = np.array(probes, dtype=f32)
    probes = np.concatenate([probes, -probes, np.array([-0.0], dtype=f32)])
    blocks = []
    for anchor in (6.0, 6.2, 7.5):
        vals = probes * f32(anchor / 6.0) if anchor != 6.0 else probes
        vals = np.concatenate([vals, np.array([anchor * 0.99, -anchor * 0.999], dtype=f32)])
        for i in range(0, len(vals), 15):
            blk = np.zeros(16, dtype=f32)
            chunk = vals[i:i + 15]
            pos = i // 15 % 16                       # the anchor at varying positions
            rest = [j for j in range(16) if j != pos]
            blk[pos] = anchor if (i // 15) % 2 == 0 else -anchor
            blk[rest[:len(chunk)]] = chunk
            blocks.append(blk)
    while len(blocks) % 16:
        blocks.append(np.zeros(16, dtype=f32))
    x = np.stack(blocks).reshape(-1, 256)
    codes_ref, sf_ref = oracle.quantize(x, 1.0)
    codes, sf, _ = moe.nvfp4_quantize(torch.from_numpy(x).to(DEV), torch.tensor([1.0], dtype=torch.float32,
                                                                                device=DEV))
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
    # and through bf16 input (the activations' type): the values that bf16 holds exactly
    xb = torch.from_numpy(x).to(torch.bfloat16)
    codes_ref, sf_ref = oracle.quantize(xb.float().numpy(), 1.0)
    codes, sf, _ = moe.nvfp4_quantize(xb.to(DEV), torch.tensor([1.0], dtype=torch.float32, device=DEV))
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    assert np.array_equal(codes.cpu().numpy(), codes_ref)


@pytest.mark.parametrize("gate_up,K", [(True, 320), (False, 512), (False, 128)])
def test_quantize_weights_grouped_blocked_bitexact(gate_up, K):
    E, N = 3, 256
    w = inputs.expert_weights(E, N, K, 77)
    c_ref, s_ref, sc_ref = oracle.quantize_weights(w.numpy())
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=gate_up)
    torch.cuda.synchronize()
    assert np.array_equal(pw.scale.cpu().numpy(), sc_ref)
    rowmap = moe.gate_up_row_map(N, "cpu").numpy() if gate_up else np.arange(N)
    codes, sf = unblock_weights(pw.blocked, E * N, K)
    for e in range(E):
        assert np.array_equal(codes[e * N + rowmap], c_ref[e])
        assert np.array_equal(sf[e * N + rowmap], s_ref[e])


def test_quantize_gather_into_padded_tiled_rows():
    T, E, k, H = 50, 16, 4, 256
    x = inputs.activations(T, H, seed=4)
    logits = inputs.router_logits(T, E, seed=8).numpy()
    ids, _ = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    rows = padded_rows_of_items(offs.astype(np.int64), ids.reshape(-1), e2p)
    alloc = moe.padded_rows_max(T * k, E)
    codes, sf, s = moe.nvfp4_quantize(x.to(DEV), None, n_items=T * k, src_div=k,
                                      dst_row=torch.from_numpy(rows.astype(np.int32)).to(DEV),
                                      sf_layout=moe.SF_TILED, dst_rows_alloc=alloc)
    tok = np.arange(T * k) // k
    assert np.array_equal(codes.cpu().numpy()[rows], xc[tok])
    assert np.array_equal(untile_rows(sf, rows, H), xs[tok])
    assert s.item() == np.float32(xsc)


# ------------------------------------------------------------------ finalize

@pytest.mark.parametrize("T,k,N", [(16, 2, 256), (333, 8, 1024), (1, 1, 8)])
def test_finalize_matches_oracle(T, k, N):
    R = T * k
    g = torch.Generator().manual_seed(T + N)
    y = torch.randn(R + 7, N, generator=g).to(torch.bfloat16)
    w = torch.rand(T, k, generator=g)
    w = w / w.sum(1, keepdim=True)
    rows = torch.randperm(R + 7, generator=g)[:R].to(torch.int32)
    ref = oracle.finalize(bf16_to_np(y), w.numpy(), rows.numpy())
    out = moe.moe_finalize(y.to(DEV), w.to(DEV), rows.to(DEV))
    tol_check(bf16_to_np(out), ref, "finalize")


# ------------------------------------------------------------------ router (logits GEMM + routing)

# the router kernel's K splits per 128-token tile (a cluster of that many CTAs): 4 (16, 200 and 2000 tokens),
# 8 (129 and 100 tokens), 16 where the GPU holds every tile's 16-CTA cluster at once, else 8 (300, 256 and 1024
# tokens; 256 tokens with E = 200 and 8 K blocks per split), 2 (6144 tokens: 48 tiles); E = 40 and E = 200 leave a
# partial 32-expert lane group; k = 32 makes
# 8-token chunks (two per owner CTA at 8 splits, one at 16), k = 1 one chunk per owner
@pytest.mark.parametrize("T,E,k,H", [(16, 8, 2, 256), (129, 40, 4, 512), (300, 256, 8, 1024), (1024, 256, 8, 6144),
                                     (6144, 256, 8, 512), (100, 256, 32, 512), (256, 256, 32, 1024),
                                     (256, 200, 6, 2048), (200, 64, 1, 256), (2000, 200, 6, 256)])
def test_router_matches_oracle(T, E, k, H):
    """Logits within the FP32 summation-order bound of the oracle's FP64 sums; the routing is exactly the
    oracle's routing of the GPU's logits, and agrees with the oracle's own logits except at near-ties."""
    x = inputs.activations(T, H, seed=T)
    wg = inputs.router_gate(E, H)
    xs = torch.zeros(1, dtype=torch.float32, device=DEV)
    r, lg = moe.moe_router(x.to(DEV), wg.to(DEV), k, x_scale=xs)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    xf, wf = x.float().numpy(), wg.float().numpy()
    # x's NVFP4 decode multiplier, from the GEMM's pass over x: exactly the oracle's
    assert np.float32(oracle.tensor_scale_from_amax(oracle.amax(xf))) == xs.item()
    ref = oracle.router_logits(xf, wf)
    got = lg.cpu().numpy()
    bound = 4.0 * H * 2.0 ** -24 * (np.abs(xf).astype(np.float64) @ np.abs(wf).astype(np.float64).T)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    ids, w = oracle.route(got, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    assert np.array_equal(r.topk_id.cpu().numpy(), ids)
    assert np.array_equal(r.topk_w.cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r.expert_offsets.cpu().numpy(), offs)
    assert np.array_equal(r.perm_to_expanded.cpu().numpy(), p2e)
    assert np.array_equal(r.expanded_to_perm.cpu().numpy(), e2p)
    # against the oracle's logits: a token may select differently only where its k-th and (k+1)-th
    # oracle logits are closer than the summation bound allows to separate
    ids_ref, _ = oracle.route(ref, k)
    for t in np.nonzero(np.any(np.sort(ids, 1) != np.sort(ids_ref, 1), axis=1))[0]:
        srt = np.sort(ref[t])[::-1]
        assert srt[k - 1] - srt[k] <= 2 * bound[t].max(), t


def test_router_one_split_without_logits_output():
    """With 80 or more 128-token tiles each tile gets one K split, and without a logits output the owner CTA
    routes straight from its drained accumulator (no split sum pass): the routing must be the one of the call
    that also writes the logits, which is the oracle's routing of those logits."""
    T, E, k, H = 10240, 64, 4, 256
    x = inputs.activations(T, H, seed=11)
    wg = inputs.router_gate(E, H)
    xd, wgd = x.to(DEV), wg.to(DEV)
    xs1 = torch.zeros(1, dtype=torch.float32, device=DEV)
    xs2 = torch.zeros(1, dtype=torch.float32, device=DEV)
    r1, lg = moe.moe_router(xd, wgd, k, x_scale=xs1)
    r2, none = moe.moe_router(xd, wgd, k, want_logits=False, x_scale=xs2)
    torch.cuda.synchronize()
    assert none is None
    assert moe.device_error() == (0, 0)
    ids, w = oracle.route(lg.cpu().numpy(), k)
    assert np.array_equal(r1.topk_id.cpu().numpy(), ids)
    assert np.array_equal(r1.topk_w.cpu().numpy().view(np.uint32), w.view(np.uint32))
    for f in ("topk_id", "topk_w", "expert_offsets", "perm_to_expanded", "expanded_to_perm", "expanded_to_row"):
        assert torch.equal(getattr(r1, f), getattr(r2, f)), f
    assert xs1.item() == xs2.item() == np.float32(oracle.tensor_scale_from_amax(oracle.amax(x.float().numpy())))


def test_router_timeout_path_reports_and_recovers():
    """The router's first CTA never fills its first stage: its bounded waits give up, the launch reports
    MOE_ERR_TIMEOUT, and that CTA's tile is void in every CTA of its cluster, so the tile's tokens go to
    experts 0..k-1 with weight 0 (a valid routing the scan and scatter place). The other tiles route as a
    clean call does, and the next call is exact."""
    T, E, k, H = 300, 64, 4, 1024
    x = inputs.activations(T, H, seed=T)
    wg = inputs.router_gate(E, H)
    xd, wgd = x.to(DEV), wg.to(DEV)
    got = {}

    def launch():
        got["r"], _ = moe.moe_router(xd, wgd, k)
        torch.cuda.synchronize()
    code, _ = _run_with_timeout_hook(launch)
    assert code == 6  # MOE_ERR_TIMEOUT
    rv = got["r"]
    ids_v, w_v = rv.topk_id.cpu().numpy(), rv.topk_w.cpu().numpy()
    r, lg = moe.moe_router(xd, wgd, k)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    ids, w = oracle.route(lg.cpu().numpy(), k)
    assert np.array_equal(r.topk_id.cpu().numpy(), ids)
    assert np.array_equal(r.topk_w.cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(ids_v[:128], np.tile(np.arange(k), (128, 1)))
    assert not w_v[:128].any()
    assert np.array_equal(ids_v[128:], ids[128:])
    assert np.array_equal(w_v[128:].view(np.uint32), w[128:].view(np.uint32))
    offs, p2e, e2p = oracle.permute(ids_v, E)
    assert np.array_equal(rv.expert_offsets.cpu().numpy(), offs)
    assert np.array_equal(rv.perm_to_expanded.cpu().numpy(), p2e)
    assert np.array_equal(rv.expanded_to_perm.cpu().numpy(), e2p)


# ------------------------------------------------------------------ grouped GEMM

def _routed_operand(x_bf16, offs):
    """Quantise routed rows (unpadded, expert-grouped) into the padded tiled layout on the GPU."""
    R = x_bf16.shape[0]
    pad = oracle.padded_offsets(offs)
    e_of_row = np.repeat(np.arange(len(offs) - 1), np.diff(offs))
    dst = (pad[e_of_row] + (np.arange(R) - offs[e_of_row])).astype(np.int32)
    alloc = max(128, int(pad[-1]))
    alloc = ((alloc + 127) // 128) * 128
    codes, sf, s = moe.nvfp4_quantize(x_bf16.to(DEV), None, dst_row=torch.from_numpy(dst).to(DEV),
                                      sf_layout=moe.SF_TILED, dst_rows_alloc=alloc)
    return codes, sf, s, dst


GEMM_CASES = [
    ([3, 0, 17, 9], 128, 256),
    ([32] * 8, 256, 512),
    ([1, 31, 33, 64, 65, 128, 129, 200, 0, 255], 256, 320),
    ([40, 7], 384, 128),
    ([300], 128, 1024),
]


@pytest.mark.parametrize("counts,N,K", GEMM_CASES)
def test_grouped_gemm_none_matches_oracle(counts, N, K):
    E = len(counts)
    offs = counts_to_offsets(counts)
    R = int(offs[-1])
    x = inputs.activations(R, K, seed=R + K)
    w = inputs.expert_weights(E, N, K, 100 + N)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    wq = oracle.quantize_weights(w.numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *wq, offs, N, K)
    codes, sf, s, dst = _routed_operand(x, offs)
    assert np.array_equal(codes.cpu().numpy()[dst], xc)
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=False)
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_NONE)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    tol_check(bf16_to_np(out)[dst], ref, "grouped GEMM NONE")


def test_grouped_gemm_none_max_experts():
    """E = 1024 (the largest expert count a launch takes), 0-3 rows per expert, one partial K stage."""
    rng = np.random.default_rng(1024)
    counts = rng.integers(0, 4, 1024).tolist()
    E, N, K = 1024, 128, 64
    offs = counts_to_offsets(counts)
    R = int(offs[-1])
    x = inputs.activations(R, K, seed=5)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    w = inputs.expert_weights(E, N, K, 700)
    wq = oracle.quantize_weights(w.numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *wq, offs, N, K)
    codes, sf, s, dst = _routed_operand(x, offs.astype(np.int64))
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=False)
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_NONE)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    tol_check(bf16_to_np(out)[dst], ref, "E=1024")


def test_grouped_gemm_identity_expert_is_exact():
    """W = identity (e2m1 1.0, scales 1), inputs on the e2m1 grid: the output is the input, exactly."""
    K = N = 256
    R = 40
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    rng = np.random.default_rng(1)
    x = grid[rng.integers(0, 8, (R, K))] * rng.choice([-1, 1], (R, K)).astype(np.float32)
    x[:, ::16] = 6.0  # every block's amax is the tensor amax: block scale 448, codes = x
    xt = torch.from_numpy(x).to(torch.bfloat16)
    xf = xt.float().numpy()
    codes, sf, s, dst = _routed_operand(xt, counts_to_offsets([R]))
    eye = torch.eye(K, dtype=torch.float32)[None] * 1.0
    pw = moe.prepare_expert_weights(eye.to(DEV), gate_up=False)
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(counts_to_offsets([R])).to(DEV))
    got = bf16_to_np(out)[dst]
    xc, xs, xsc = oracle.quantize_dynamic(xf)
    wq = oracle.quantize_weights(eye.numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *wq, counts_to_offsets([R]), N, K)
    assert np.allclose(ref, xf, rtol=1e-6, atol=0)  # exact up to the FP32 rounding of the scales
    assert np.array_equal(got, xf.astype(np.float64))


def _assert_rare_adjacent_flips(got, ref):
    """Decoded NVFP4 values of a requantised FP32 tensor whose FP32 inputs differ by rounding:
    a value may differ only near a rounding boundary (rare) and then by at most one e2m1 step
    of its block (2/6 of the block maximum, plus the e4m3 scale's own rounding)."""
    mism = got != ref
    assert mism.mean() < 2e-3, mism.mean()
    if mism.any():
        blk = np.abs(ref).reshape(ref.shape[0], -1, 16).max(-1)
        bound = np.repeat(blk, 16, axis=1) * (2.0 / 6.0) * 1.07 + 1e-30
        assert np.all(np.abs(got - ref)[mism] <= bound[mism])
    return mism


def _silu_case(counts, I, H, seed):
    E = len(counts)
    offs = counts_to_offsets(counts)
    R = int(offs[-1])
    x = inputs.activations(R, H, seed=seed)
    w13 = inputs.expert_weights(E, 2 * I, H, seed + 1)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    w13q = oracle.quantize_weights(w13.numpy())
    y1 = oracle.grouped_gemm(xc, xs, xsc, *w13q, offs, 2 * I, H)
    h = oracle.silu_mul(y1)
    h_scale = oracle.tensor_scale_from_amax(oracle.amax(h.astype(np.float32)))
    return offs, x, w13, h, h_scale


@pytest.mark.parametrize("counts,I,H", [([3, 0, 17, 9], 64, 256), ([1, 33, 129, 64], 128, 320), ([32] * 4, 256, 512)])
def test_grouped_gemm_silu_mul_quant(counts, I, H):
    offs, x, w13, h_ref, h_scale = _silu_case(counts, I, H, 11 + I)
    codes, sf, s, dst = _routed_operand(x, offs)
    pw = moe.prepare_expert_weights(w13.to(DEV), gate_up=True)
    alloc = codes.shape[0]
    h_f32 = torch.zeros(alloc, I, dtype=torch.float32, device=DEV)
    hs_out = torch.zeros(1, dtype=torch.float32, device=DEV)
    hc, hsf = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_SILU_MUL_QUANT,
                                         h_scale=h_scale, h_f32=h_f32, h_scale_out=hs_out)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    assert hs_out.item() == np.float32(h_scale)
    # (i) the FP32 SiLU-mul output against the oracle's FP64 one
    tol_check(h_f32.cpu().numpy()[dst], h_ref, "SiLU-mul h")
    # (ii) the requantised codes: the oracle's own codes of its own h, compared
    # as decoded values; a code may differ only where h sits on a rounding
    # boundary, by one grid step, and such flips must be rare.
    hc_ref, hs_ref = oracle.quantize(h_ref.astype(np.float32), h_scale)
    got = oracle.dequantize(hc.cpu().numpy()[dst], untile_rows(hsf, dst, I))
    ref = oracle.dequantize(hc_ref, hs_ref)
    _assert_rare_adjacent_flips(got, ref)


def test_grouped_gemm_silu_quant_exact_inputs():
    """Inputs chosen so every value on the way is exact in FP32 and FP64: power-of-two tensor
    scales (amax = 2688 * 2^j), e4m3-exact block scales, gate values so large that silu(g) = g in
    both precisions, products of 441 * 2^a.  The requantised codes and scales are then fully
    determined: compare them bit for bit."""
    I, H, R = 64, 256, 48
    # x row r: 10.5 (= 2688 * 2^-8) in column (r % 4) * 64, zero elsewhere
    x = torch.zeros(R, H)
    for r in range(R):
        x[r, (r % 4) * 64] = 10.5
    rng = np.random.default_rng(5)
    mags = np.array([21.0, 42.0, 84.0, 168.0], np.float32)   # 168 = 2688 * 2^-4; block scales 56..448
    w = np.zeros((1, 2 * I, H), np.float32)
    for c in range(4):
        w[0, :I, c * 64] = rng.choice(mags, I)                                  # gate > 0: silu(g) = g
        w[0, I:, c * 64] = rng.choice(mags, I) * rng.choice([-1.0, 1.0], I)     # up
    w[0, 0, 0] = 168.0
    wt = torch.from_numpy(w)
    offs = counts_to_offsets([R])
    xc, xs, xsc = oracle.quantize_dynamic(x.numpy())
    assert xsc == 2.0 ** -8
    wq = oracle.quantize_weights(w)
    assert wq[2][0] == 2.0 ** -4
    y1 = oracle.grouped_gemm(xc, xs, xsc, *wq, offs, 2 * I, H)
    h = oracle.silu_mul(y1)
    assert np.all(h.astype(np.float32) == h)  # exact in FP32
    h_scale = oracle.tensor_scale_from_amax(oracle.amax(h.astype(np.float32)))
    hc_ref, hs_ref = oracle.quantize(h.astype(np.float32), h_scale)
    codes, sf, s, dst = _routed_operand(x.to(torch.bfloat16), offs)
    pw = moe.prepare_expert_weights(wt.to(DEV), gate_up=True)
    h_f32 = torch.zeros(codes.shape[0], I, dtype=torch.float32, device=DEV)
    hc, hsf = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_SILU_MUL_QUANT,
                                         h_scale=h_scale, h_f32=h_f32)
    torch.cuda.synchronize()
    assert np.array_equal(h_f32.cpu().numpy()[dst], h.astype(np.float32))
    assert np.array_equal(hc.cpu().numpy()[dst], hc_ref)
    assert np.array_equal(untile_rows(hsf, dst, I), hs_ref)


@pytest.mark.parametrize("T,E,k,H,I", [(16, 8, 2, 256, 128), (200, 32, 4, 384, 256), (64, 256, 8, 256, 64)])
def test_grouped_gemm_finalize_matches_oracle(T, E, k, H, I):
    logits = inputs.router_logits(T, E, seed=T + E).numpy()
    ids, w = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    R = T * k
    g = torch.Generator().manual_seed(T)
    h = (torch.randn(R, I, generator=g) * 0.3).numpy()
    hc, hs, hsc = oracle.quantize_dynamic(h)
    w2 = inputs.expert_weights(E, H, I, 500)
    w2q = oracle.quantize_weights(w2.numpy())
    y2 = oracle.grouped_gemm(hc, hs, hsc, *w2q, offs, H, I)
    ref = oracle.finalize(y2, w, e2p)
    # GPU: the oracle's h (FP32 values) quantised on the GPU into padded rows
    codes, sf, s, dst = _routed_operand(torch.from_numpy(h), offs.astype(np.int64))
    assert np.array_equal(codes.cpu().numpy()[dst], hc)
    pw = moe.prepare_expert_weights(w2.to(DEV), gate_up=False)
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_FINALIZE,
                                     perm_to_expanded=torch.from_numpy(p2e).to(DEV),
                                     topk_w=torch.from_numpy(w).to(DEV), T=T, k=k)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    tol_check(bf16_to_np(out), ref, "FINALIZE")


@pytest.mark.parametrize("T,E,k,H,I,mode", [(20000, 4, 2, 1024, 64, "chunked"), (132000, 2, 1, 128, 64, "rows")])
def test_grouped_gemm_finalize_large_T_modes(T, E, k, H, I, mode):
    """FINALIZE past an L2-sized accumulator: column-chunked atomics, and per-item rows summed in slot order."""
    ws = moe._lib.load().moe_grouped_gemm_workspace_size(moe.EPI_FINALIZE, T, k, H)
    assert ws == (T * H * 4 if mode == "chunked" else T * k * H * 4)
    logits = inputs.router_logits(T, E, seed=7).numpy()
    ids, w = oracle.route(logits, k)
    offs, p2e, e2p = oracle.permute(ids, E)
    g = torch.Generator().manual_seed(11)
    h = (torch.randn(T * k, I, generator=g) * 0.3).numpy()
    hc, hs, hsc = oracle.quantize_dynamic(h)
    w2 = inputs.expert_weights(E, H, I, 600)
    w2q = oracle.quantize_weights(w2.numpy())
    ref = oracle.finalize(oracle.grouped_gemm(hc, hs, hsc, *w2q, offs, H, I), w, e2p)
    codes, sf, s, dst = _routed_operand(torch.from_numpy(h), offs.astype(np.int64))
    pw = moe.prepare_expert_weights(w2.to(DEV), gate_up=False)
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV), moe.EPI_FINALIZE,
                                     perm_to_expanded=torch.from_numpy(p2e).to(DEV),
                                     topk_w=torch.from_numpy(w).to(DEV), T=T, k=k)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    tol_check(bf16_to_np(out), ref, "FINALIZE " + mode)


# ------------------------------------------------------------------ fused layer

def _layer_case(T, E, k, H, I, zipf=None):
    x = inputs.activations(T, H)
    logits = inputs.router_logits(T, E, zipf_s=zipf)
    w13f = inputs.expert_weights(E, 2 * I, H, inputs.gate_up_seed_base())
    w2f = inputs.expert_weights(E, H, I, inputs.down_seed_base(E))
    return x, logits, w13f, w2f


@pytest.mark.parametrize("T,E,k,H,I,zipf", [(16, 8, 2, 256, 128, None), (96, 64, 6, 512, 192, None),
                                            (128, 32, 4, 256, 128, 1.1),
                                            # degenerate shapes: one token and one expert; every expert
                                            # selected (k = E); one token over mostly empty experts with a
                                            # single partial K stage in the down GEMM (I = 64)
                                            (1, 1, 1, 256, 128, None), (40, 4, 4, 256, 128, None),
                                            (1, 256, 8, 256, 64, None), (33, 3, 2, 384, 64, None)])
def test_moe_forward_matches_oracle(T, E, k, H, I, zipf):
    x, logits, w13f, w2f = _layer_case(T, E, k, H, I, zipf)
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits.numpy(), w13, w2, k)
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I)
    out = fwd(x.to(DEV), logits.to(DEV), pw13, pw2, h_scale)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    _check_layer(fwd, out, ref, h_scale, T, E, k, H, I)


def _check_layer(fwd, out, ref, h_scale, T, E, k, H, I):
    R = T * k
    # routing, permutation and the quantised activations: bit-exact
    assert np.array_equal(fwd.view("topk_id", torch.int32, (T, k)).cpu().numpy(), ref.topk_id)
    assert np.array_equal(fwd.view("topk_w", torch.float32, (T, k)).cpu().numpy(), ref.topk_w)
    assert np.array_equal(fwd.view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(fwd.view("perm_to_expanded", torch.int32, (R,)).cpu().numpy(), ref.perm_to_expanded)
    rows = padded_rows_of_items(ref.expert_offsets.astype(np.int64), ref.topk_id.reshape(-1), ref.expanded_to_perm)
    P = fwd.layout.padded_rows
    xcodes = fwd.view("x_codes", torch.uint8, (P, H // 2)).cpu().numpy()
    perm_rows = rows[ref.perm_to_expanded]
    assert np.array_equal(xcodes[perm_rows], ref.x_codes)
    assert np.array_equal(untile_rows(fwd.view("x_sf", torch.uint8, (P * H // 16,)), perm_rows, H), ref.x_sf)
    # the requantised intermediate: rare one-step flips only
    hcodes = fwd.view("h_codes", torch.uint8, (P, I // 2)).cpu().numpy()[perm_rows]
    hsf = untile_rows(fwd.view("h_sf", torch.uint8, (P * I // 16,)), perm_rows, I)
    href_c, href_s = oracle.quantize(ref.h.astype(np.float32), h_scale)
    flips = _assert_rare_adjacent_flips(oracle.dequantize(hcodes, hsf), oracle.dequantize(href_c, href_s))
    got = bf16_to_np(out)
    rel = np.linalg.norm(got - ref.out) / np.linalg.norm(ref.out)
    assert rel < 1e-2, rel
    if not flips.any():
        tol_check(got, ref.out, "moe_forward")


@pytest.mark.parametrize("T,E,k,H,I", [(16, 8, 2, 256, 128), (300, 64, 6, 512, 192), (129, 40, 4, 256, 128)])
def test_moe_forward_gated_matches_oracle(T, E, k, H, I):
    """The router in front of the layer: the oracle's layer on the GPU router's logits (the logits themselves
    are checked against the oracle's FP64 sums in test_router_matches_oracle), x's decode multiplier from
    the router's GEMM, everything else as moe_forward."""
    x, _, w13f, w2f = _layer_case(T, E, k, H, I)
    wg = inputs.router_gate(E, H)
    _, lg = moe.moe_router(x.to(DEV), wg.to(DEV), k)
    logits = lg.cpu().numpy()
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits, w13, w2, k)
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I, gated=True)
    out = fwd.gated(x.to(DEV), wg.to(DEV), pw13, pw2, h_scale)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    assert np.float32(oracle.tensor_scale_from_amax(oracle.amax(x.float().numpy()))) == \
        fwd.view("x_scale", torch.float32, (1,)).item()
    _check_layer(fwd, out, ref, h_scale, T, E, k, H, I)


def _run_with_timeout_hook(launch):
    """Runs `launch` with the first pipeline stage never filled and a 50 ms wait bound; returns the error."""
    torch.cuda.synchronize()
    moe.device_error()
    moe.set_wait_timeout_ns(50_000_000)
    moe.debug_set_flags(1)
    try:
        launch()
        return moe.device_error()
    finally:
        moe.debug_set_flags(0)
        moe.set_wait_timeout_ns(0)


@pytest.mark.parametrize("counts", [[32, 32], [200, 150]])   # the 64-row (decode) and 128-row tile
def test_timeout_path_reports_and_recovers(counts):
    """A pipeline stage that is never filled: the bounded waits give up, the kernel reports
    MOE_ERR_TIMEOUT and returns; the context stays usable."""
    N, K = 128, 512
    offs = counts_to_offsets(counts)
    x = inputs.activations(int(offs[-1]), K, seed=1)
    w = inputs.expert_weights(2, N, K, 3)
    codes, sf, s, dst = _routed_operand(x, offs)
    pw = moe.prepare_expert_weights(w.to(DEV), gate_up=False)
    code, _ = _run_with_timeout_hook(lambda: moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV)))
    assert code == 6  # MOE_ERR_TIMEOUT
    out = moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw, torch.from_numpy(offs).to(DEV))
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    xc, xs, xsc = oracle.quantize_dynamic(x.float().numpy())
    ref = oracle.grouped_gemm(xc, xs, xsc, *oracle.quantize_weights(w.numpy()), offs, N, K)
    tol_check(bf16_to_np(out)[dst], ref, "after timeout")


@pytest.mark.parametrize("epi", ["silu", "finalize"])
def test_timeout_path_128_row_epilogues(epi):
    """The same at the 128-row tile with the SiLU epilogue and with FINALIZE (two epilogue warp groups)."""
    T, E, k, H, I = 512, 4, 2, 256, 128
    x, logits, w13f, w2f = _layer_case(T, E, k, H, I)
    fwd = moe.MoeForward(T, E, k, H, I)
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    ids, w = oracle.route(logits.numpy(), k)
    offs, p2e, e2p = oracle.permute(ids, E)
    pad = oracle.padded_offsets(offs.astype(np.int64))
    assert (int(pad[-1]) - 127 * E) // E > 48  # the kernel picks its 128-row tile above 48 rows per expert
    if epi == "silu":
        codes, sf, s, dst = _routed_operand(torch.repeat_interleave(x, k, 0)[p2e], offs.astype(np.int64))

        def launch():
            moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw13, torch.from_numpy(offs).to(DEV), moe.EPI_SILU_MUL_QUANT,
                                       h_scale=0.01)
    else:
        h = (torch.randn(T * k, I, generator=torch.Generator().manual_seed(2)) * 0.3)
        codes, sf, s, dst = _routed_operand(h, offs.astype(np.int64))

        def launch():
            moe.moe_grouped_gemm_nvfp4(codes, sf, s, pw2, torch.from_numpy(offs).to(DEV), moe.EPI_FINALIZE,
                                       perm_to_expanded=torch.from_numpy(p2e).to(DEV),
                                       topk_w=torch.from_numpy(w).to(DEV), T=T, k=k)
    code, _ = _run_with_timeout_hook(launch)
    assert code == 6  # MOE_ERR_TIMEOUT
    # the context still works: the layer runs and matches the oracle
    out = fwd(x.to(DEV), logits.to(DEV), pw13, pw2, 0.01)
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("stage_events,staged", [(True, True), (False, True), (True, False), (False, False)])
def test_forward_graph_replays_the_layer(stage_events, staged):
    """moe_forward captured as one CUDA graph: the replay matches the oracle, and refilling the
    inputs in place then relaunching matches an eager moe_forward on the new inputs.  Without stage
    events the staged graph runs the amax pass beside the routing and clears the FINALIZE accumulator
    beside the gate_up GEMM: every intermediate is checked as for the eager layer.  `staged` captures
    the staged kernels (debug flag bit 2) instead of the single-launch path this size takes."""
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
    moe.debug_set_flags(4 if staged else 0)
    try:
        g = fwd.graph(xd, ld, pw13, pw2, h_scale, stage_events=stage_events)
    finally:
        moe.debug_set_flags(0)
    for _ in range(2):  # a replay after a replay (the accumulator cleared again)
        out = g.launch()
    torch.cuda.synchronize()
    assert moe.device_error() == (0, 0)
    got = bf16_to_np(out)
    assert np.linalg.norm(got - ref.out) / np.linalg.norm(ref.out) < 1e-2
    _check_layer(fwd, out, ref, h_scale, T, E, k, H, I)
    if stage_events:
        ms = g.stage_ms()
        # the single-launch layer's time is all in the first stage
        assert (all(m > 0 for m in ms) if staged else ms[0] > 0 and all(m >= 0 for m in ms))
        assert abs(sum(ms[:4]) - ms[4]) < 1e-3 * max(1.0, ms[4]) + 1e-3
    # new inputs, same buffers
    x2 = inputs.activations(T, H, seed=123)
    l2 = inputs.router_logits(T, E, seed=456)
    xd.copy_(x2.to(DEV))
    ld.copy_(l2.to(DEV))
    out = g.launch()
    torch.cuda.synchronize()
    eager = moe.moe_forward(x2.to(DEV), l2.to(DEV), pw13, pw2, k, h_scale)
    torch.cuda.synchronize()
    ref2 = oracle.moe_layer(x2.float().numpy(), l2.numpy(), w13, w2, k, h_scale=h_scale)
    a, b = bf16_to_np(out), bf16_to_np(eager)
    assert np.linalg.norm(a - ref2.out) / np.linalg.norm(ref2.out) < 1e-2
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-3
    g.close()
    assert moe.device_error() == (0, 0)


def test_fp4_mma_probes_run_and_report_rates():
    """Both dense FP4 MMA-rate probes (one CTA per SM, M = 128; CTA pairs, M = 256) finish without a device
    error and report a rate in the range a GB300's tensor cores can give."""
    one = moe.fp4_mma_peak_tflops(iters=2000, reps=2)
    pair = moe.fp4_mma_peak_tflops(iters=2000, reps=2, pair=True)
    assert moe.device_error() == (0, 0)
    for rate in (one, pair):
        assert 1000.0 < rate < 20000.0, (one, pair)


@pytest.mark.parametrize("T,E,k,H,I", [(16, 8, 2, 256, 128), (96, 64, 6, 512, 192)])
def test_forward_graph_run_host_from_and_to_host_buffers(T, E, k, H, I):
    """moe_forward_graph_run_host: host inputs copied in, the graph replayed, the output copied back, on one
    stream; the host result equals the device replay's on the same inputs, and new host inputs give the
    layer on them."""
    x, logits, w13f, w2f = _layer_case(T, E, k, H, I)
    w13 = oracle.quantize_weights(w13f.numpy())
    w2 = oracle.quantize_weights(w2f.numpy())
    ref = oracle.moe_layer(x.float().numpy(), logits.numpy(), w13, w2, k)
    h_scale = float(oracle.tensor_scale_from_amax(oracle.amax(ref.h.astype(np.float32))))
    pw13 = moe.prepare_expert_weights(w13f.to(DEV), gate_up=True)
    pw2 = moe.prepare_expert_weights(w2f.to(DEV), gate_up=False)
    fwd = moe.MoeForward(T, E, k, H, I)
    xd, ld = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV), torch.zeros(T, E, device=DEV)
    g = fwd.graph(xd, ld, pw13, pw2, h_scale, stage_events=False)
    out_h = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    st = torch.cuda.Stream()
    g.run_host(x.contiguous().pin_memory(), logits.contiguous().pin_memory(), out_h, stream=st)
    st.synchronize()
    assert moe.device_error() == (0, 0)
    got = bf16_to_np(out_h)
    assert np.linalg.norm(got - ref.out) / np.linalg.norm(ref.out) < 1e-2
    # the device buffers hold what was copied in: a plain replay gives the same output
    dev_out = g.launch()
    torch.cuda.synchronize()
    assert np.linalg.norm(bf16_to_np(dev_out) - got) / np.linalg.norm(got) < 1e-3
    x2 = inputs.activations(T, H, seed=31)
    l2 = inputs.router_logits(T, E, seed=32)
    g.run_host(x2.pin_memory(), l2.pin_memory(), out_h, stream=st)
    st.synchronize()
    ref2 = oracle.moe_layer(x2.float().numpy(), l2.numpy(), w13, w2, k, h_scale=h_scale)
    assert np.linalg.norm(bf16_to_np(out_h) - ref2.out) / np.linalg.norm(ref2.out) < 1e-2
    g.close()
