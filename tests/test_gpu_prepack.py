"""Prepacked stage-2 weights (moe_prepack): the packed bytes are a pure
rearrangement of w2 / w2_scale (checked against numpy, bit for bit), and the
forward pass reading them matches the oracle like the plain layout does."""
import numpy as np
import pytest
import torch

import quantized_moe_expert_sort_gb300 as moe
from _cases import bits_to_f64, gpu_f64, make_case, oracle_forward, to_dev, token_rel_l2

pytestmark = pytest.mark.gpu


def _numpy_pack(w2, w2s, swizzled):
    E, H, Ih = w2.shape
    I = 2 * Ih
    HT, KC = H // 128, I // 128
    blocks = w2.reshape(E, HT, 128, KC, 4, 16).transpose(0, 1, 3, 2, 4, 5)  # [e, ht, kc, r, chunk, 16]
    if swizzled:  # chunk c of row r stored at c ^ ((r / 2) % 4)
        r = np.arange(128)[:, None]
        c = np.arange(4)[None, :]
        dst = c ^ ((r >> 1) & 3)
        out = np.empty_like(blocks)
        out[:, :, :, r, dst, :] = blocks[:, :, :, r, c, :]
        blocks = out
    codes = blocks.reshape(-1)
    s = w2s.reshape(E, HT, 4, 32, KC, 4)            # [e, ht, r/32, r%32, kc, b]
    scales = s.transpose(0, 1, 4, 3, 2, 5).reshape(-1)  # [e, ht, kc, r%32, r/32, b]
    return np.concatenate([codes, scales])


@pytest.mark.parametrize("a_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("H,I,E", [(3584, 384, 16), (384, 256, 5)])
def test_prepack_is_a_rearrangement(H, I, E, a_dtype):
    g = torch.Generator().manual_seed(H + I)
    w2 = torch.randint(0, 256, (E, H, I // 2), generator=g, dtype=torch.uint8)
    w2s = torch.randint(100, 140, (E, H, I // 32), generator=g, dtype=torch.uint8)
    ctx = moe.MoE(H, I, E, 4, 8)
    packed = ctx.prepack(w2.cuda(), w2s.cuda(), a_dtype)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), _numpy_pack(w2.numpy(), w2s.numpy(), a_dtype != "fp8"))


@pytest.mark.parametrize("a_dtype,T,H,I,E,K", [("bf16", 1, 3584, 384, 896, 16), ("bf16", 64, 3584, 384, 896, 16),
                                               ("fp8", 64, 3584, 384, 896, 16), ("fp4", 16, 3584, 384, 896, 16),
                                               ("bf16", 16, 384, 128, 8, 2), ("fp8", 16, 384, 128, 8, 2)])
def test_forward_with_prepacked_w2(a_dtype, T, H, I, E, K):
    case = make_case(T, H, I, E, K, "uniform", 321, experts_all=E <= 8)
    d = to_dev(case)
    ctx = moe.MoE(H, I, E, K, T)
    plain = ctx.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], "situv2", 4.0, 25.0, a_dtype)
    ctx.prepack(d["w2"], d["w2s"], a_dtype)
    packed = ctx.forward(d["x"], d["ids"], d["w"], d["w13"], d["w13s"], d["w2"], d["w2s"], "situv2", 4.0, 25.0,
                         a_dtype)
    torch.cuda.synchronize()
    assert ctx.last_sort()["tile_m"] == 1  # the few-rows path
    _, ref16, _, _ = oracle_forward(case, "situv2", a_dtype)
    bar = 2e-3 if a_dtype == "bf16" else 1e-2
    assert token_rel_l2(gpu_f64(packed), bits_to_f64(ref16)) <= bar
    # the same products, summed in another order by the combine: equal to rounding
    assert token_rel_l2(gpu_f64(packed), gpu_f64(plain)) <= bar
    assert ctx.get_error() == (0, 0)
    ctx.unbind_prepacked()
