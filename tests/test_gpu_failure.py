"""Failure detection on the GPU, with no GPU fault involved.

- The bounded wait every pipeline stage uses runs out on a barrier nothing
  completes (a short limit, a self-test kernel): the kernel returns, the device
  error word reports MOE_ERR_TIMEOUT, and the context stays usable.
- An allocation failure injected on the host makes moe_create release what it
  had allocated and return MOE_ERR_OOM.
"""
import pytest
import torch

import quantized_moe_expert_sort_gb300 as moe
from _cases import bits_to_f64, make_case, oracle_forward, to_dev, token_rel_l2, gpu_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_survives():
    case = make_case(16, 256, 128, 8, 2, "softmax_topk", 0)
    ctx = moe.MoE(256, 128, 8, 2, 16)
    ctx.selftest_wait(1_000_000, complete=False)  # 1 ms on a barrier nobody completes
    st, flags = ctx.get_error()
    assert st == 6 and flags & moe.DEVERR_TIMEOUT
    ctx.selftest_wait(1_000_000_000, complete=True)
    assert ctx.get_error() == (0, 0)
    d = to_dev(case)
    out = ctx.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], "situv2", 4.0, 25.0, "bf16")
    _, ref16, _, _ = oracle_forward(case, "situv2", "bf16")
    assert token_rel_l2(gpu_f64(out), bits_to_f64(ref16)) <= 2e-3
    assert ctx.get_error() == (0, 0)


@pytest.mark.parametrize("n", [0, 5, 12])
def test_injected_allocation_failure_frees_and_reports_oom(n):
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    moe.debug_inject_alloc_failure(n)
    with pytest.raises(moe.MoEError) as e:
        moe.MoE(3584, 384, 896, 16, 4096)
    assert e.value.status == 4 and "injected" in str(e.value)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (64 << 20)  # nothing of the failed context stays allocated
    ctx = moe.MoE(3584, 384, 896, 16, 64)   # one-shot: the next creation succeeds
    ctx.close()
