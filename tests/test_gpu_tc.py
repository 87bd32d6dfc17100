"""GPU parity of the many-rows tensor-core path (tcgen05 block-scaled, 128 sorted
rows x 128 weight rows per tile) against the CPU oracle.

The path is chosen when the mean number of routed rows per active expert
reaches the context's threshold (MOE_TC_MIN_ROWS at moe_create, default 32).
The small cases force it either way to run both paths on the same inputs; the
full-size workloads run with the default selection. Bar: every sampled token's
bf16 output within relL2 <= 1e-2 of the oracle's; requantised intermediates
checked code by code (_cases.check_requant_rows).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_sort_gb300 as moe
from _cases import bits_to_f64, check_requant_rows, gpu_f64, make_case, oracle_forward, to_dev, token_rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _ctx(case, min_rows=None):
    old = os.environ.get("MOE_TC_MIN_ROWS")
    if min_rows is not None:
        os.environ["MOE_TC_MIN_ROWS"] = str(min_rows)
    elif old is not None:
        del os.environ["MOE_TC_MIN_ROWS"]
    try:
        return moe.MoE(case["H"], case["I"], case["E"], case["K"], case["T"])
    finally:
        if old is None:
            os.environ.pop("MOE_TC_MIN_ROWS", None)
        else:
            os.environ["MOE_TC_MIN_ROWS"] = old


def _run(case, ctx, act, a_dtype):
    d = to_dev(case)
    out = ctx.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], act, 4.0, 25.0, a_dtype)
    torch.cuda.synchronize()
    return gpu_f64(out)


def _check_tokens(got, case, act, a_dtype, subset=None):
    _, ref16, _, _ = oracle_forward(case, act, a_dtype, subset=subset)
    g = got if subset is None else got[np.asarray(subset)]
    r = token_rel_l2(g, bits_to_f64(ref16))
    assert r <= TOL, r
    return r


def _check_expert_rows(ctx, case, act, a_dtype, expert, max_rows=None):
    """The requantised stage-1 output of every routed row of one expert (or the
    first max_rows of them), element by element."""
    T, K = case["T"], case["K"]
    srt = ctx.last_sort()
    off = srt["expert_offset"].cpu().numpy()
    cnt = int(srt["expert_count"].cpu().numpy()[expert])
    n = cnt if max_rows is None else min(cnt, max_rows)
    rows = np.arange(off[expert], off[expert] + n)
    pid = srt["sorted_ids"].cpu().numpy()[rows]
    assert np.all(pid < T * K) and np.all(np.diff(pid) > 0)  # ascending pair ids inside an expert
    codes, scales, fmt = ctx.intermediate(srt["num_rows"], a_dtype)
    y32, _ = oracle.expert_stage1(case["x_bits"], pid // K, case["w13"][expert], case["w13s"][expert], act, 4.0, 25.0,
                                  a_dtype)
    return check_requant_rows(codes.cpu().numpy()[rows], scales.cpu().numpy()[rows], y32, a_dtype)


@pytest.mark.parametrize("a_dtype", ["fp8", "fp4"])
@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_tc_small_full_output_and_intermediate(a_dtype, act):
    case = make_case(256, 1024, 256, 4, 2, "uniform", 21, experts_all=True)
    ctx = _ctx(case, 1)
    got = _run(case, ctx, act, a_dtype)
    assert ctx.last_sort()["tile_m"] == 128
    _check_tokens(got, case, act, a_dtype)
    st, flags = ctx.get_error()
    assert st == 0 and flags == 0
    for e in range(4):
        cd, sd = _check_expert_rows(ctx, case, act, a_dtype, e)
        assert cd < 0.01 and sd < 0.01


@pytest.mark.parametrize("a_dtype", ["fp8", "fp4"])
def test_tc_and_decode_paths_agree(a_dtype):
    case = make_case(192, 512, 384, 6, 4, "uniform", 22, experts_all=True)
    a = _run(case, _ctx(case, 1), "situv2", a_dtype)
    b = _run(case, _ctx(case, 0), "situv2", a_dtype)
    _check_tokens(a, case, "situv2", a_dtype)
    _check_tokens(b, case, "situv2", a_dtype)
    assert token_rel_l2(a, b) <= 2 * TOL


@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_tp8_a8_4096_default_path(act):
    case = make_case(4096, 3584, 384, 896, 16, "uniform", 123, experts_all=True)
    ctx = _ctx(case)
    got = _run(case, ctx, act, "fp8")
    assert ctx.last_sort()["tile_m"] == 128
    _check_tokens(got, case, act, "fp8", subset=np.array([0, 1, 999, 2048, 4095], np.int32))
    _check_expert_rows(ctx, case, act, "fp8", expert=int(case["ids"][0, 0]))


def test_ep_wide_inter_2048_forced_and_8192_default():
    case = make_case(2048, 3584, 3072, 112, 16, "uniform", 7, experts_all=True)
    got = _run(case, _ctx(case, 32), "situv2", "fp8")
    _check_tokens(got, case, "situv2", "fp8", subset=np.array([0, 77, 2047], np.int32))
    case = make_case(8192, 3584, 3072, 112, 16, "uniform", 7, experts_all=True)
    ctx = _ctx(case)
    got = _run(case, ctx, "situv2", "fp8")
    assert ctx.last_sort()["tile_m"] == 128
    _check_tokens(got, case, "situv2", "fp8", subset=np.array([0, 4096, 8191], np.int32))
    _check_expert_rows(ctx, case, "situv2", "fp8", expert=int(case["ids"][8191, 3]), max_rows=256)
    st, flags = ctx.get_error()
    assert st == 0 and flags == 0


@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_a4_zipf_32768_default_path(act):
    """The largest workload: Zipf(1.1) routing concentrates pairs on few experts.
    Every routed row of the most loaded expert is checked element by element, plus
    the full output of sampled tokens, including tokens of that expert."""
    case = make_case(32768, 3584, 384, 896, 16, "zipf", 42, experts_all=True)
    ctx = _ctx(case)
    got = _run(case, ctx, act, "fp4")
    assert ctx.last_sort()["tile_m"] == 128
    ids = case["ids"].numpy()
    counts = np.bincount(ids.ravel(), minlength=896)
    hot = int(np.argmax(counts))
    cd, sd = _check_expert_rows(ctx, case, act, "fp4", hot)
    assert cd < 1e-3 and sd < 1e-3
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0]
    cold = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    cold_tokens = np.nonzero((ids == cold).any(axis=1))[0][:4]
    sub = np.unique(np.concatenate([np.array([0, 16383, 32767]), hot_tokens[:: max(1, len(hot_tokens) // 12)][:12],
                                    cold_tokens])).astype(np.int32)
    _check_tokens(got, case, act, "fp4", subset=sub)
    st, flags = ctx.get_error()
    assert st == 0 and flags == 0


@pytest.mark.parametrize("act", ["silu", "situv2"])
def test_tc_a4_zipf_8192_forced(act):
    case = make_case(8192, 3584, 384, 896, 16, "zipf", 42, experts_all=True)
    ctx = _ctx(case, 8)
    got = _run(case, ctx, act, "fp4")
    assert ctx.last_sort()["tile_m"] == 128
    ids = case["ids"].numpy()
    counts = np.bincount(ids.ravel(), minlength=896)
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0][:6]
    sub = np.unique(np.concatenate([np.array([0, 4095, 8191]), hot_tokens])).astype(np.int32)
    _check_tokens(got, case, act, "fp4", subset=sub)
