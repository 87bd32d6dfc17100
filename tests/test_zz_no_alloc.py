"""moe_sort_noalloc: the expert sort for callers that cannot allocate device
memory (a serving engine whose pool owns the GPU memory, a decode loop that
must not trigger an allocation's device synchronisation, a router with no
moe_ctx). Called through the C ABI with caller-owned output buffers and
checked against moe_sort's output; the two are integer data, so the check is
exact. Two calls in a row on different routings show that the shared scratch
array keeps no stale state between calls. This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import quantized_moe_expert_sort_gb300 as moe
from quantized_moe_expert_sort_gb300 import inputs

pytestmark = pytest.mark.gpu


def _noalloc_sort(ids, E, tile_m):
    L = moe.lib()
    L.moe_sort_noalloc.restype = ctypes.c_int
    L.moe_sort_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int] + \
        [ctypes.c_void_p] * 7
    T, K = ids.shape
    n = T * K
    rows = n + min(E, n) * (tile_m - 1)
    dev = ids.device
    out = dict(sorted_ids=torch.full((max(rows, 1),), -7, dtype=torch.int32, device=dev),
               block_expert=torch.full((max(rows // tile_m + 1, 1),), -7, dtype=torch.int32, device=dev),
               expert_count=torch.empty(E, dtype=torch.int32, device=dev),
               expert_offset=torch.empty(E + 1, dtype=torch.int32, device=dev),
               active_experts=torch.empty(E, dtype=torch.int32, device=dev),
               meta=torch.full((4,), -1, dtype=torch.int32, device=dev))
    st = L.moe_sort_noalloc(ctypes.c_void_p(ids.data_ptr()), T, K, E, tile_m,
                            *[ctypes.c_void_p(out[k].data_ptr()) for k in
                              ("sorted_ids", "block_expert", "expert_count", "expert_offset", "active_experts",
                               "meta")],
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.moe_last_error_message().decode()
    torch.cuda.synchronize()
    meta = out["meta"].cpu().numpy()
    nb, na, nr = int(meta[0]), int(meta[1]), int(meta[2])
    return dict(sorted_ids=out["sorted_ids"][:nr].cpu().numpy(), block_expert=out["block_expert"][:nb].cpu().numpy(),
                expert_count=out["expert_count"].cpu().numpy(), expert_offset=out["expert_offset"].cpu().numpy(),
                active_experts=out["active_experts"][:na].cpu().numpy(), flags=int(meta[3]))


@pytest.mark.parametrize("T,K,E,tile_m,kind", [(4096, 16, 896, 16, "uniform"), (64, 16, 896, 8, "uniform")])
def test_noalloc_sort_matches_moe_sort_twice(T, K, E, tile_m, kind):
    ctx = moe.MoE(128, 128, E, K, T)
    for seed in (11, 12):  # two calls in a row on different routings
        ids, _ = inputs.make_routing(T, E, K, kind, seed=seed)
        ids = ids.clone()
        ids[5, 3] = E + 9  # dropped pair, must be flagged in meta[3]
        ids = ids.cuda()
        got = _noalloc_sort(ids, E, tile_m)
        ref = ctx.sort(ids, tile_m)
        for key in ("sorted_ids", "block_expert", "expert_count", "expert_offset", "active_experts"):
            assert np.array_equal(got[key], ref[key].cpu().numpy()), key
        assert got["flags"] & moe.DEVERR_BAD_EXPERT
        ctx.get_error()


def test_noalloc_sort_rejects_oversize_problem():
    L = moe.lib()
    L.moe_sort_noalloc.restype = ctypes.c_int
    L.moe_sort_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int] + \
        [ctypes.c_void_p] * 7
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    # 1M pairs x 4096 experts needs far more than the scratch array holds
    st = L.moe_sort_noalloc(p, 65536, 16, 4096, 16, p, p, p, p, p, p, None)
    assert st == 1
    assert "scratch" in L.moe_last_error_message().decode()
