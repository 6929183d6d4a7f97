"""The routing entry point for callers that cannot allocate device memory.

moe_route_permute_static takes no workspace (its scratch is a fixed array in
the library's device memory) and must give exactly what moe_route_permute
gives with a caller-allocated workspace, on consecutive calls that reuse the
shared scratch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_moe_grouped_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(T, E, k):
    R = T * k
    return [torch.full((T, k), -1, dtype=torch.int32, device=DEV), torch.full((T, k), -1.0, device=DEV),
            torch.full((E + 1,), -1, dtype=torch.int32, device=DEV)] + \
           [torch.full((R,), -1, dtype=torch.int32, device=DEV) for _ in range(3)]


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _with_workspace(L, logits, k):
    T, E = logits.shape
    outs = _outputs(T, E, k)
    wsb = L.moe_route_permute_workspace_size(T, E, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    assert L.moe_route_permute(_p(logits), T, E, k, *[_p(o) for o in outs], _p(ws), wsb, _stream()) == 0
    return outs


def _static(L, logits, k):
    T, E = logits.shape
    outs = _outputs(T, E, k)
    assert L.moe_route_permute_static(_p(logits), T, E, k, *[_p(o) for o in outs], _stream()) == 0
    return outs


@pytest.mark.parametrize("T,E,k,zipf", [(1024, 256, 8, None), (512, 256, 8, 1.1), (16, 8, 2, None)])
def test_static_scratch_matches_workspace_version_twice(T, E, k, zipf):
    L = _lib.load()
    assert L.moe_route_permute_static_scratch_bytes() == 1 << 20
    la = inputs.router_logits(T, E, zipf_s=zipf).to(DEV)
    lb = inputs.router_logits(T, E, seed=77).to(DEV)
    ref_a = _with_workspace(L, la, k)
    ref_b = _with_workspace(L, lb, k)
    got_a = _static(L, la, k)       # first call (sets up the scratch address on this device)
    got_b = _static(L, lb, k)       # second call reuses the scratch left by the first
    torch.cuda.synchronize()
    for ref, got in ((ref_a, got_a), (ref_b, got_b)):
        for r, g in zip(ref, got):
            assert torch.equal(r, g)
    # the routing weights are bit-identical, not just close
    assert np.array_equal(ref_a[1].cpu().numpy().view(np.uint32), got_a[1].cpu().numpy().view(np.uint32))


def test_static_scratch_rejects_oversized_problems():
    L = _lib.load()
    T, E, k = 65536, 1024, 8   # needs far more than 1 MiB of scratch
    assert L.moe_route_permute_workspace_size(T, E, k) > L.moe_route_permute_static_scratch_bytes()
    # Null pointers everywhere: the size check answers first (MOE_ERR_WORKSPACE).  Were it ever to let
    # the call through, the null-pointer check behind it would still stop it on the host before any launch.
    assert L.moe_route_permute_static(None, T, E, k, *([None] * 6), None) == 7  # MOE_ERR_WORKSPACE
    # shapes the routing kernels do not implement get MOE_ERR_UNSUPPORTED, as from moe_route_permute,
    # however large their workspace would be
    assert L.moe_route_permute_static(None, 65536, 2048, 8, *([None] * 6), None) == 3
    assert L.moe_route_permute_static(None, 65536, 256, 33, *([None] * 6), None) == 3
