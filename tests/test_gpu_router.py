"""GPU parity of the top-k softmax router (moe_route) against the oracle:
expert ids bit-exact (selection compares logits exactly on both sides), weights
within 2e-6 of the oracle's fp64 values (fp32 exp and sum on the GPU)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_sort_gb300 as moe
from quantized_moe_expert_sort_gb300 import inputs

pytestmark = pytest.mark.gpu


def _route(logits, K):
    ids, w = moe.route(logits.cuda(), K)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)


def test_router_on_the_small_workload_logits():
    T, E, K, seed = 16, 8, 2, 0
    logits = inputs.make_router_logits(T, E, seed)
    ids, w = _route(logits, K)
    rid, rw = oracle.route(logits.numpy(), K)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= 2e-6
    ids_in, _ = inputs.make_routing(T, E, K, "softmax_topk", seed)
    assert np.array_equal(ids, ids_in.numpy())


@pytest.mark.parametrize("T,E,K,grid", [(4096, 896, 16, None), (3000, 112, 16, None), (513, 896, 16, 0.25),
                                        (100, 4096, 32, None), (77, 33, 32, 1.0), (1, 8, 1, None)])
def test_router_ids_bit_exact(T, E, K, grid):
    g = torch.Generator().manual_seed(T + E + K)
    logits = torch.randn(T, E, generator=g)
    if grid:  # many equal logits: ties go to the lower expert id
        logits = torch.round(logits / grid) * grid
    ids, w = _route(logits, K)
    rid, rw = oracle.route(logits.numpy(), K)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= 2e-6


def test_router_neg_inf_and_empty():
    logits = torch.randn(64, 112)
    logits[:, :50] = float("-inf")
    ids, w = _route(logits, 16)
    rid, rw = oracle.route(logits.numpy(), 16)
    assert np.array_equal(ids, rid) and np.all(ids >= 50)
    assert np.max(np.abs(w - rw)) <= 2e-6
    e_ids, e_w = moe.route(torch.empty((0, 112), device="cuda"), 16)
    assert e_ids.shape == (0, 16)
    with pytest.raises(moe.MoEError):
        moe.route(torch.zeros((4, 8), device="cuda"), 9)
