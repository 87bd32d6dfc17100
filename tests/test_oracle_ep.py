"""Pins for the oracle's expert-parallel forward (ranks own equal expert slices;
each rank's share of a token crosses an fp8 1x32 combine wire; shares are summed).

(1) without the wire, the shares add up to the single-rank forward (1e-12);
(2) with one rank, the result is the single-rank forward held in fp32 and sent
    through the pinned MX quantiser (e4m3, 32 along H), composed in numpy;
(3) any number of ranks with the wire stays within the fp8 quantisation error of
    the single-rank forward, and moving experts between ranks changes only that;
(4) a token whose pairs all live on one rank gets exactly one wire round trip.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_sort_gb300 import inputs


def _case(T=12, H=256, I=128, E=8, K=3, seed=1):
    x = inputs.make_x(T, H, seed)
    ids, w = inputs.make_routing(T, E, K, "uniform", seed)
    w13 = torch.stack([inputs.expert_w13(e, H, I, seed) for e in range(E)]).numpy()
    w2 = torch.stack([inputs.expert_w2(e, H, I, seed) for e in range(E)]).numpy()
    c13, s13 = oracle.quantize_weights(w13)
    c2, s2 = oracle.quantize_weights(w2)
    return dict(x=x.view(torch.int16).numpy().astype(np.uint16), ids=ids.numpy(), w=w.numpy(),
                w13=c13, w13s=s13, w2=c2, w2s=s2)


def _fwd(c, **kw):
    return oracle.moe_forward(c["x"], c["ids"], c["w"], c["w13"], c["w13s"], c["w2"], c["w2s"], "situv2", 4.0, 25.0,
                              kw.get("adt", "bf16"))


def _ep(c, R, wire=True, adt="bf16", subset=None):
    return oracle.ep_forward(c["x"], c["ids"], c["w"], c["w13"], c["w13s"], c["w2"], c["w2s"], R, "situv2", 4.0, 25.0,
                             adt, wire=wire, subset=subset)


@pytest.mark.parametrize("R", [1, 2, 4, 8])
@pytest.mark.parametrize("adt", ["bf16", "fp8"])
def test_shares_add_up_without_the_wire(R, adt):
    c = _case()
    full, _, _, _ = _fwd(c, adt=adt)
    ep, _ = _ep(c, R, wire=False, adt=adt)
    assert np.max(np.abs(ep - full)) <= 1e-12 * np.max(np.abs(full))


def test_one_rank_is_one_wire_round_trip_of_the_forward():
    c = _case()
    full, _, _, _ = _fwd(c)
    f32 = full.astype(np.float32).astype(np.float64)
    codes, scales = oracle.mx_quantize(f32, "e4m3")
    want = oracle.mx_dequantize(codes, scales, "e4m3")
    ep, ep16 = _ep(c, 1)
    assert np.array_equal(ep, want)
    assert np.array_equal(ep16, np.array([[oracle.bf16_from_f64(v) for v in row] for row in want], np.uint16))


@pytest.mark.parametrize("R", [2, 4, 8])
def test_wire_error_is_the_fp8_quantisation(R):
    c = _case(T=16, H=512, E=16, K=4)
    full, _, _, _ = _fwd(c)
    ep, _ = _ep(c, R)
    rel = np.linalg.norm(ep - full, axis=1) / np.linalg.norm(full, axis=1)
    # e4m3 has 3 mantissa bits: per-value error below 2^-4 relative, ~1-3% in L2
    assert rel.max() < 0.05 and rel.max() > 1e-3
    # a subset of tokens gives the same rows
    sub = np.array([3, 0, 15], np.int32)
    ep_s, _ = _ep(c, R, subset=sub)
    assert np.array_equal(ep_s, ep[sub])


def test_token_on_one_rank_gets_one_round_trip():
    c = _case(T=4, E=8, K=2)
    c["ids"] = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32)  # with R=4 each token lives on one rank
    full, _, _, _ = _fwd(c)
    f32 = full.astype(np.float32).astype(np.float64)
    codes, scales = oracle.mx_quantize(f32, "e4m3")
    ep, _ = _ep(c, 4)
    assert np.array_equal(ep, oracle.mx_dequantize(codes, scales, "e4m3"))
