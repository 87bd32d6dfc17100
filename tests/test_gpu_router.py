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


@pytest.mark.parametrize("E,K", [(200, 8), (255, 16), (500, 32), (512, 4), (1000, 16), (1023, 32), (1024, 1)])
def test_router_every_register_width(E, K):
    # E <= 1024 runs the register-resident kernel (4, 8, 16 or 32 logits per lane;
    # 16-byte loads when E % 4 == 0); half the rows carry a coarse grid of ties
    g = torch.Generator().manual_seed(E * 31 + K)
    logits = torch.randn(300, E, generator=g)
    logits[1::2] = torch.round(logits[1::2] * 2) / 2
    ids, w = _route(logits, K)
    rid, rw = oracle.route(logits.numpy(), K)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= 2e-6


def test_router_all_equal_and_candidate_overflow():
    # all logits equal: every element passes the lane-maximum threshold, so the
    # exact fallback selection runs; ids are 0..K-1, weights 1/K
    ids, w = _route(torch.full((5, 896), 0.5), 16)
    assert np.array_equal(ids, np.tile(np.arange(16, dtype=np.int32), (5, 1)))
    assert np.max(np.abs(w - 1.0 / 16)) <= 2e-6
    # one block of 200 equal logits on top of noise: more candidates than the
    # rank step takes on some rows, few on others
    g = torch.Generator().manual_seed(7)
    logits = torch.randn(257, 4096, generator=g) * 0.1
    logits[::2, 1000:1200] = 3.0
    ids, w = _route(logits, 32)
    rid, rw = oracle.route(logits.numpy(), 32)
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
