"""bench.py's roofline arithmetic (CPU): a kernel against the slower of its bytes at
the HBM peak and its FLOPs at the tensor peak; a call against its roofline time."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_hbm_bound_kernel():
    # TP8 a16w4 decode T = 64, stage 1: 608 active experts' w13 + x + intermediate
    r = bench.kernel_roofline(890306560, 5637144576.0, 0.15815, 6773.9, "measured", 1937.8, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(890306560 / 0.15815e-3 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(0.8311, abs=1e-4)


def test_tensor_bound_kernel():
    # EP-shard a8w4 T = 8192, stage 1: 4 H I flops per routed pair at the fp8 peak (2 x bf16)
    flops = 4.0 * 131072 * 3584 * 3072
    r = bench.kernel_roofline(1.43e9, flops, 3.446, 6773.9, "m", 2 * 1937.8, "m")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(flops / 3.446e-3 / 1e12, abs=0.05)
    assert 0.42 < r["frac"] < 0.44


def test_call_fraction():
    bound, frac = bench.call_roofline(1336079360, 6.0 * 1024 * 3584 * 384, 0.28496, 6773.9, 1937.8)
    assert bound == "hbm"
    assert frac == pytest.approx(1336079360 / 6773.9e9 / 0.28496e-3, abs=1e-4)
    bound, _ = bench.call_roofline(1.0e6, 1.0e12, 1.0, 6773.9, 1937.8)
    assert bound == "tensor"


def test_algorithmic_bytes_of_the_decode_call():
    bench.select_config("tp8_decode")
    ab = bench.algo_bytes(64, 608, 1024)
    assert ab["stage1"] == 890306560
    assert ab["call"] == ab["stage1"] + ab["stage2"]  # the intermediate is written by one, read by the other
    assert ab["call"] == 608 * 2 * 384 * (1792 + 112) + 608 * 3584 * (192 + 12) + 64 * 3584 * 2 * 2 + 2 * 1024 * 384 * 2
