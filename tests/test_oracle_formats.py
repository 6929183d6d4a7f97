"""Pins of the oracle's number formats and quantiser against things other than itself.

e2m1/e4m3 decode: the published FP4 grid and torch's float8_e4m3fn type (a
library routine).  Encoders: exhaustive rounding-boundary sweeps and the
golden tie table.  Quantiser: properties the NVFP4 definition fixes (block
amax maps onto the top of the e2m1 range, codes are the nearest grid points,
re-quantising a quantised block is the identity).
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def next_up(x):
    return float(np.nextafter(np.float32(x), np.float32(np.inf)))


def next_down(x):
    return float(np.nextafter(np.float32(x), np.float32(-np.inf)))


def test_e2m1_decode_matches_published_grid():
    for c in range(8):
        assert oracle.e2m1_decode(c) == E2M1_GRID[c]
        assert oracle.e2m1_decode(c | 8) == -E2M1_GRID[c]


def test_e4m3_decode_matches_torch_float8_e4m3fn_exhaustively():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def _e4m3_values():
    return sorted({oracle.e4m3_decode(c) for c in range(0x7F)})


def test_e4m3_encode_matches_torch_on_every_midpoint_and_neighbour():
    vals = _e4m3_values()
    probes = []
    for a, b in zip(vals[:-1], vals[1:]):
        mid = f32((a + b) / 2)
        probes += [a, b, mid, next_up(mid), next_down(mid), next_up(a), next_down(b)]
    probes = [p for p in probes if 0 <= p <= 448.0]
    t = torch.tensor(probes, dtype=torch.float32)
    ref = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for p, r in zip(probes, ref):
        assert oracle.e4m3_encode(p) == r, (p, oracle.e4m3_encode(p), r)


def test_e4m3_encode_saturates_and_handles_zero():
    for v in [448.0, 449.0, 463.9, 464.0, 500.0, 1e30, float("inf")]:
        assert oracle.e4m3_encode(v) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0
    assert oracle.e4m3_encode(2.0 ** -11) == 0          # below half the smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10) == 0          # exact tie with 0 -> even code 0
    assert oracle.e4m3_encode(next_up(2.0 ** -10)) == 1


def test_e2m1_encode_golden_table():
    n = 0
    with open(os.path.join(GOLDEN, "e2m1_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            x, code = line.split()
            assert oracle.e2m1_encode(float(x)) == int(code, 16), (x, code)
            n += 1
    assert n >= 25


def test_e2m1_encode_is_nearest_even_on_every_boundary():
    grid = E2M1_GRID
    for i in range(7):
        a, b = grid[i], grid[i + 1]
        mid = (a + b) / 2
        even = i if i % 2 == 0 else i + 1
        assert oracle.e2m1_encode(mid) == even
        assert oracle.e2m1_encode(next_down(mid)) == i
        assert oracle.e2m1_encode(next_up(mid)) == i + 1
        assert oracle.e2m1_encode(-next_up(mid)) == (i + 1) | 8


def test_tensor_scale_definition():
    assert oracle.tensor_scale_from_amax(0.0) == 1.0
    assert oracle.tensor_scale_from_amax(2688.0) == 1.0
    assert oracle.tensor_scale_from_amax(6.0) == np.float32(6.0) / np.float32(2688.0)


def _decode_row(codes, sf, s):
    vals = oracle.dequantize(codes[None, :], sf[None, :])[0]
    return vals * s


def test_quantize_block_max_lands_on_six_and_codes_are_nearest():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 64)).astype(np.float32) * 3.0
    codes, sf, s = oracle.quantize_dynamic(x)
    # tensor amax sits in some block: its scale is exactly 448 and its code is +-6
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, c // 16] == 0x7E
    byte = codes[r, c // 2]
    q = (byte >> 4) if c % 2 else (byte & 15)
    assert q & 7 == 7
    # every code is the nearest grid point of x / (e4m3(sf) * s), from the definition
    for row in range(0, 64, 7):
        for blk in range(4):
            d = np.float32(oracle.e4m3_decode(int(sf[row, blk]))) * np.float32(s)
            for i in range(16):
                kk = blk * 16 + i
                v = np.float32(x[row, kk]) * (np.float32(1.0) / d)
                byte = codes[row, kk // 2]
                q = (byte >> 4) if kk % 2 else (byte & 15)
                mag = E2M1_GRID[q & 7]
                dist = abs(abs(float(v)) - mag)
                assert all(dist <= abs(abs(float(v)) - g) + 1e-12 for g in E2M1_GRID)


def test_requantising_a_quantised_tensor_is_identity():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    codes, sf, s = oracle.quantize_dynamic(x)
    xq = (oracle.dequantize(codes, sf) * s).astype(np.float32)
    codes2, sf2 = oracle.quantize(xq, s)
    assert np.array_equal(codes, codes2)
    assert np.array_equal(sf, sf2)


def test_zero_block_and_packing_order():
    x = np.zeros((1, 32), np.float32)
    x[0, 16] = 6.0 * 448 * 0.5    # second block only; element 16 -> low nibble of byte 8
    x[0, 17] = -6.0 * 448 * 0.25  # element 17 -> high nibble of byte 8
    codes, sf = oracle.quantize(x, 0.5)
    assert sf[0, 0] == 0 and np.all(codes[0, :8] == 0)
    assert sf[0, 1] == 0x7E
    assert codes[0, 8] & 15 == 7          # 6.0
    assert codes[0, 8] >> 4 == (5 | 8)    # -3.0


def test_smem_model_matches_pages_table():
    n = 0
    with open(os.path.join(GOLDEN, "smem_model_sm120.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            M, N, K, st, dflt, fin = map(int, line.split())
            assert round(oracle.smem_model_bytes(M, N, K, st, False) / 1024) == dflt
            assert round(oracle.smem_model_bytes(M, N, K, st, True) / 1024) == fin
            n += 1
    assert n == 4
    assert oracle.smem_model_bytes(128, 256, 128, 1, False) - 128 * 256 * 2 == 27648


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-5, 5, 2000),
                        [0.0, -0.0, 1.0, 65504.0, 3.0e38]])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    got = oracle.f64_to_bf16_bits(v)
    assert np.array_equal(got.view(np.int16), ref)


@pytest.mark.parametrize("x", [0.0, -1e-3, -0.5, -1.0, -3.7, -10.0, -20.0, -50.0, -85.9, 0.3, 2.0])
def test_exp_close_to_libm(x):
    got = oracle.exp32(x)
    ref = math.exp(np.float32(x))
    assert abs(got - ref) <= 2 * abs(float(np.spacing(np.float32(ref))))


def test_exp_sweep_within_two_ulp():
    xs = np.linspace(-86.0, 0.0, 20001, dtype=np.float32)
    worst = 0.0
    for x in xs:
        got = oracle.exp32(float(x))
        ref = math.exp(float(x))
        ulp = float(np.spacing(np.float32(ref)))
        worst = max(worst, abs(got - ref) / ulp)
    assert worst <= 2.0, worst
    assert oracle.exp32(-86.5) == 0.0
    assert oracle.exp32(0.0) == 1.0
