"""Pins for the oracle's top-k softmax router (the routing of the small parity
workload: softmax over the E logits of a token, the K largest probabilities,
renormalised over the K; equal logits take the lower expert id first).

Checked against: a brute-force selection written independently (numpy's stable
lexicographic sort); the softmax carried out in 40-digit arithmetic (mpmath) in
the order the routing states it (softmax over E, pick, renormalise); closed
forms (K = E, equal logits, shift invariance); and the seeded routing of
quantized_moe_expert_sort_gb300.inputs, which draws the same logits.
"""
import numpy as np
import pytest

import oracle
from quantized_moe_expert_sort_gb300 import inputs

mpmath = pytest.importorskip("mpmath")


def _brute_ids(logits, K):
    T, E = logits.shape
    out = np.zeros((T, K), np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))  # by -logit, then id
        out[t] = order[:K]
    return out


def _mp_weights(logits, ids):
    mpmath.mp.dps = 40
    T, K = ids.shape
    w = np.zeros((T, K))
    for t in range(T):
        ex = [mpmath.exp(mpmath.mpf(float(v))) for v in logits[t]]
        tot = mpmath.fsum(ex)
        p = [v / tot for v in ex]
        sel = [p[int(e)] for e in ids[t]]
        s = mpmath.fsum(sel)
        w[t] = [float(v / s) for v in sel]
    return w


@pytest.mark.parametrize("T,E,K,grid", [(64, 8, 2, None), (32, 112, 16, None), (16, 896, 16, None),
                                        (64, 9, 4, 0.5), (40, 33, 7, 1.0)])
def test_router_ids_and_weights(T, E, K, grid):
    rng = np.random.default_rng(T * E + K)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if grid:  # coarse grid: many equal logits, ties broken by the lower id
        logits = (np.round(logits / grid) * grid).astype(np.float32)
    ids, w = oracle.route(logits, K)
    assert np.array_equal(ids, _brute_ids(logits, K))
    assert np.max(np.abs(w - _mp_weights(logits, ids))) <= 1e-15
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_router_closed_forms():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((5, 6)).astype(np.float32)
    # K = E: every expert, weights = the full softmax
    ids, w = oracle.route(logits, 6)
    z = np.exp(logits.astype(np.float64) - logits.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    assert np.allclose(np.take_along_axis(p, ids.astype(np.int64), 1), w, rtol=1e-15, atol=0)
    # equal logits: ids 0..K-1 and weights 1/K
    ids, w = oracle.route(np.zeros((3, 10), np.float32), 4)
    assert np.array_equal(ids, np.tile(np.arange(4), (3, 1)))
    assert np.all(w == 0.25)
    # adding a constant to every logit changes nothing (logits on a 2^-12 grid, so
    # that the shifted values are exact in fp32)
    lg = (np.round(logits * 4096) / 4096).astype(np.float32)
    ids0, w0 = oracle.route(lg, 3)
    ids1, w1 = oracle.route(lg + np.float32(8.0), 3)
    assert np.array_equal(ids0, ids1) and np.allclose(w0, w1, rtol=1e-14, atol=0)
    # -inf logits are never chosen while a finite one is left
    l2 = logits.copy()
    l2[:, :3] = -np.inf
    ids2, w2 = oracle.route(l2, 3)
    assert np.all(ids2 >= 3) and np.allclose(w2.sum(axis=1), 1.0)
    with pytest.raises(ValueError):
        oracle.route(logits, 7)


def test_router_matches_the_seeded_softmax_topk_routing():
    T, E, K, seed = 16, 8, 2, 0
    logits = inputs.make_router_logits(T, E, seed).numpy()
    ids_ref, w_ref = inputs.make_routing(T, E, K, "softmax_topk", seed)
    ids, w = oracle.route(logits, K)
    assert np.array_equal(ids, ids_ref.numpy())
    assert np.max(np.abs(w - w_ref.numpy().astype(np.float64))) <= 1e-6
