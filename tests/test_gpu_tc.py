"""GPU parity of the tensor-core (tcgen05 block-scaled) path against the CPU oracle.

The path is chosen when the mean number of routed rows per active expert
reaches the context's threshold (MOE_TC_MIN_ROWS at moe_create, default 32);
the tests force it either way to run both paths on the same inputs.
Bar: outputs within relL2 <= 1e-2 of the oracle; intermediate codes decoded and
compared row by row in the sorted order.
"""
import os

import numpy as np
import pytest
import torch

import quantized_moe_expert_sort_gb300 as moe
from _cases import decode_codes, decode_intermediate, make_case, oracle_forward, rel_l2, to_dev

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _ctx(case, min_rows):
    old = os.environ.get("MOE_TC_MIN_ROWS")
    os.environ["MOE_TC_MIN_ROWS"] = str(min_rows)
    try:
        return moe.MoE(case["H"], case["I"], case["E"], case["K"], case["T"])
    finally:
        if old is None:
            del os.environ["MOE_TC_MIN_ROWS"]
        else:
            os.environ["MOE_TC_MIN_ROWS"] = old


def _run(case, ctx, act, a_dtype):
    d = to_dev(case)
    out = ctx.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], act, 4.0, 25.0, a_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("a_dtype", ["fp8", "fp4"])
@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_tc_small_full_output_and_intermediate(a_dtype, act):
    case = make_case(256, 1024, 256, 4, 2, "uniform", 21, experts_all=True)
    ctx = _ctx(case, 1)
    got = _run(case, ctx, act, a_dtype)
    assert ctx.last_sort()["tile_m"] == 128
    ref64, _, inter, _ = oracle_forward(case, act, a_dtype, want_inter=True)
    r = rel_l2(got, ref64)
    assert r <= TOL, r
    st, flags = ctx.get_error()
    assert st == 0 and flags == 0
    srt = ctx.last_sort()
    codes, scales, fmt = ctx.intermediate(srt["num_rows"], a_dtype)
    dec = decode_intermediate(codes.cpu().numpy(), scales.cpu().numpy(), fmt)
    sid = srt["sorted_ids"].cpu().numpy()
    valid = sid < case["T"] * case["K"]
    assert rel_l2(dec[valid], inter[sid[valid]]) <= TOL


@pytest.mark.parametrize("a_dtype", ["fp8", "fp4"])
def test_tc_and_decode_paths_agree(a_dtype):
    case = make_case(192, 512, 384, 6, 4, "uniform", 22, experts_all=True)
    a = _run(case, _ctx(case, 1), "situv2", a_dtype)
    b = _run(case, _ctx(case, 0), "situv2", a_dtype)
    ref64, _, _, _ = oracle_forward(case, "situv2", a_dtype)
    assert rel_l2(a, ref64) <= TOL and rel_l2(b, ref64) <= TOL
    assert rel_l2(a, b) <= TOL


def test_tc_tp8_a8_4096_sampled():
    case = make_case(4096, 3584, 384, 896, 16, "uniform", 123, experts_all=True)
    ctx = _ctx(case, 32)
    got = _run(case, ctx, "situv2", "fp8")
    assert ctx.last_sort()["tile_m"] == 128
    sub = np.array([0, 1, 999, 2048, 4095], np.int32)
    ref64, _, _, _ = oracle_forward(case, "situv2", "fp8", subset=sub)
    assert rel_l2(got[sub], ref64) <= TOL


def test_tc_ep_wide_inter_2048_sampled():
    case = make_case(2048, 3584, 3072, 112, 16, "uniform", 7, experts_all=True)
    ctx = _ctx(case, 32)
    got = _run(case, ctx, "situv2", "fp8")
    assert ctx.last_sort()["tile_m"] == 128
    sub = np.array([0, 77, 2047], np.int32)
    ref64, _, _, _ = oracle_forward(case, "situv2", "fp8", subset=sub)
    assert rel_l2(got[sub], ref64) <= TOL


@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_tc_a4_zipf_8192_sampled(act):
    case = make_case(8192, 3584, 384, 896, 16, "zipf", 42, experts_all=True)
    ctx = _ctx(case, 8)
    got = _run(case, ctx, act, "fp4")
    assert ctx.last_sort()["tile_m"] == 128
    ids = case["ids"].numpy()
    counts = np.bincount(ids.ravel(), minlength=896)
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0][:6]
    sub = np.unique(np.concatenate([np.array([0, 4095, 8191]), hot_tokens])).astype(np.int32)
    ref64, _, _, _ = oracle_forward(case, act, "fp4", subset=sub)
    assert rel_l2(got[sub], ref64) <= TOL
