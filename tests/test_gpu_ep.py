"""GPU parity of the expert-parallel emulation (moe_ep_*: dispatch to per-rank
receive buffers, per-rank forward on the rank's expert slice, fp8 1x32 combine
wire) against the oracle's expert-parallel forward: every sampled token's bf16
output within relL2 1e-2 (the combine wire's e4m3 codes may round the other way
where the GPU's fp32 share lies on a rounding boundary), the per-rank token
counts exact."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_sort_gb300 as moe
from _cases import bits_to_f64, gpu_f64, make_case, to_dev, token_rel_l2

pytestmark = pytest.mark.gpu


def _run(case, ranks, a_dtype, subset=None):
    d = to_dev(case)
    ep = moe.MoEEP(case["H"], case["I"], case["E"] // ranks, ranks, case["K"], case["T"])
    out = ep.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], "situv2", 4.0, 25.0, a_dtype)
    torch.cuda.synchronize()
    ids = case["ids"].numpy()
    El = case["E"] // ranks
    want_counts = [int(((ids >= r * El) & (ids < (r + 1) * El)).any(axis=1).sum()) for r in range(ranks)]
    assert ep.counts() == want_counts
    assert ep.get_error() == (0, 0)
    _, ref16 = oracle.ep_forward(case["x_bits"], ids, case["w"].numpy(), case["w13"], case["w13s"], case["w2"],
                                 case["w2s"], ranks, "situv2", 4.0, 25.0, a_dtype, subset=subset)
    got = gpu_f64(out) if subset is None else gpu_f64(out)[subset]
    return token_rel_l2(got, bits_to_f64(ref16))


@pytest.mark.parametrize("a_dtype", ["bf16", "fp8", "fp4"])
@pytest.mark.parametrize("ranks", [1, 4])
def test_ep_small_all_tokens(a_dtype, ranks):
    case = make_case(48, 512, 256, 16, 4, "uniform", 61, experts_all=True)
    assert _run(case, ranks, a_dtype) <= 1e-2


def test_ep8_kimi_layout_sampled():
    """EP8 with 112 experts per rank (896 global), top-16: the layout of the A8W4
    MegaMoE page, at the TP8 expert shape (hidden 3584, inter 384) and a8."""
    case = make_case(96, 3584, 384, 896, 16, "uniform", 62)
    assert _run(case, 8, "fp8", subset=np.array([0, 33, 95], np.int32)) <= 1e-2


def test_ep_token_without_local_pairs_and_dropped_ids():
    case = make_case(16, 256, 128, 8, 2, "uniform", 63, experts_all=True)
    ids = case["ids"].clone()
    ids[5, :] = -1  # no expert at all: zeros, and a dropped pair is flagged
    case["ids"] = ids
    d = to_dev(case)
    ep = moe.MoEEP(256, 128, 2, 4, 2, 16)
    out = ep.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], "silu", 4.0, 25.0, "bf16")
    torch.cuda.synchronize()
    assert torch.all(out[5] == 0)
    st, flags = ep.get_error()
    assert st == 5 and flags & moe.DEVERR_BAD_EXPERT
    _, ref16 = oracle.ep_forward(case["x_bits"], ids.numpy(), case["w"].numpy(), case["w13"], case["w13s"],
                                 case["w2"], case["w2s"], 4, "silu", 4.0, 25.0, "bf16")
    assert token_rel_l2(gpu_f64(out), bits_to_f64(ref16)) <= 1e-2
