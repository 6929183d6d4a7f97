"""Shared helpers of the GPU parity tests: the tolerance rule and layout views.

The tolerance for floating-point outputs is the one the method states:
    |gpu - ref| <= 1e-2 * (|ref| + 1e-3 * rms(ref))
elementwise, with ref the oracle's FP64 result.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def tol_check(got: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = 1e-2 * (np.abs(ref) + 1e-3 * rms)
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} bound {bound[tuple(i)]!r}")
    return float((err / np.maximum(np.abs(ref) + 1e-3 * rms, 1e-300)).max()) if ref.size else 0.0


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def untile_rows(sf_tiled: torch.Tensor, rows, K: int) -> np.ndarray:
    return oracle.untile_sf(sf_tiled.cpu().numpy().reshape(-1), np.asarray(rows), K)


def padded_rows_of_items(expert_offsets: np.ndarray, topk_id_flat: np.ndarray, expanded_to_perm: np.ndarray):
    """Padded routed row of every expanded item, from the layout's written definition."""
    pad = oracle.padded_offsets(expert_offsets)
    e = topk_id_flat.astype(np.int64)
    return pad[e] + (expanded_to_perm.astype(np.int64) - expert_offsets[e])


def counts_to_offsets(counts) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def unblock_weights(blocked: torch.Tensor, rows: int, K: int):
    """Linear codes [rows, K/2] and scales [rows, K/16] out of a blocked weight buffer.

    Written from the blocked layout's definition: per 128 rows x 256 K-elements an
    18432-byte block, codes row rr at rr*128 with 16-byte chunk c stored at chunk
    c ^ (rr % 8), then four 512-byte scale atoms.
    """
    b = blocked.cpu().numpy().reshape(-1)
    KT = (K + 255) // 256
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    r = np.arange(rows)
    rr = r % 128
    for kt in range(KT):
        base = ((r // 128) * KT + kt) * 18432
        for c in range(8):
            if kt * 128 + 16 * c >= K // 2:
                break
            src = base + rr * 128 + ((c ^ (rr % 8)) * 16)
            codes[:, kt * 128 + 16 * c:kt * 128 + 16 * c + 16] = b[src[:, None] + np.arange(16)[None, :]]
        for cc in range(16):
            col = kt * 16 + cc
            if col >= K // 16:
                break
            src = base + 16384 + (cc // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc % 4
            sf[:, col] = b[src]
    return codes, sf
