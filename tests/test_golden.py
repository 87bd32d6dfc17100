"""Pins against values the pages print (fixtures under tests/golden/, each citing
its page and section).
"""
import math
import os
import re

import numpy as np

import oracle
from quantized_moe_expert_sort_gb300 import inputs
from _cases import make_case, oracle_forward

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n").split("\t") for ln in f if ln.strip() and not ln.startswith("#")]


def _tag_float(s):
    # "0x1d9000000000000pp4" -> "0x1.9000000000000p4"
    m = re.fullmatch(r"0x1d([0-9a-f]+)pp(-?\d+)", s)
    assert m, s
    return float.fromhex("0x1.%sp%s" % (m.group(1), m.group(2)))


def test_module_tags_decode_to_the_labelled_betas():
    """The pages' module tags encode the beta pair exactly; the Kimi-K3 pair is the
    one every workload here runs with."""
    seen = {}
    for label, tag in _rows("situv2_module_tags.txt"):
        m = re.fullmatch(r"_situv2_sb(\S+)_slb(\S+)", tag)
        assert m, tag
        b, lb = _tag_float(m.group(1)), _tag_float(m.group(2))
        lm = re.fullmatch(r"situv2 b(\d+)/l(\d+)", label)
        assert (b, lb) == (float(lm.group(1)), float(lm.group(2)))
        seen[label] = (b, lb)
    k3 = seen["situv2 b4/l25"]
    for name, cfg in inputs.CONFIGS.items():
        if "situv2" in cfg.acts:
            assert (cfg.beta, cfg.linear_beta) == k3, name


def test_linear_term_saturates_where_the_page_says():
    """|lbeta * tanh(u / lbeta)| at lbeta = 25 is within the stated margin of 25 for
    |u| at and above the page's ~100, read through the oracle's SiTUv2 at g = 200
    (where sigmoid(g) and tanh(g / beta) are exactly 1 in fp64)."""
    for u, bound in _rows("situv2_saturation.txt"):
        u, bound = float(u), float(bound)
        for s in (1.0, -1.0):
            up = oracle.act("situv2", 200.0, s * u, 4.0, 25.0) / 4.0
            assert s * up >= bound and abs(up) <= 25.0
    # below the stated range the term is visibly not saturated
    assert oracle.act("situv2", 200.0, 25.0, 4.0, 25.0) / 4.0 < 20.0


def test_a8w4_error_is_of_the_pages_order():
    """a8w4 (fp8 1x32 activations and intermediate) against the same dequantised
    weights with unquantised activations, at the Kimi-K3 TP8 shape: the same order
    of magnitude as the pages' relL2 for their fused a8w4 op."""
    (page,), = _rows("a8w4_relL2.txt")
    page = float(page)
    c = make_case(6, 3584, 384, 4, 2, "uniform", 3)
    a8, _, _, _ = oracle_forward(c, "situv2", "fp8")
    a16, _, _, _ = oracle_forward(c, "situv2", "bf16")
    rel = float(np.linalg.norm(a8 - a16) / np.linalg.norm(a16))
    assert page / 10 < rel < 2 * page, (rel, page)
    assert math.isfinite(rel)
