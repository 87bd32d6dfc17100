"""Pins for the oracle's expert sort and activation functions.

Sort: invariants, numpy's stable argsort (the same ordering written a second
way) and brute-force enumeration on tiny cases. Activations: mpmath at 40
digits, the closed-form values the SiTUv2 definition gives, and its limits.
"""
import math

import mpmath as mp
import numpy as np
import pytest

import oracle

mp.mp.dps = 40


def _sort_ref_numpy(ids, E, tile_m):
    """Second formulation: stable argsort on expert id, then padding."""
    flat = ids.ravel()
    n = flat.size
    valid = (flat >= 0) & (flat < E)
    p = np.arange(n)[valid]
    e = flat[valid]
    order = np.argsort(e, kind="stable")
    out = []
    block_expert = []
    for ex in range(E):
        sel = p[order][e[order] == ex]
        if sel.size == 0:
            continue
        pad = -sel.size % tile_m
        out.extend(sel.tolist() + [n] * pad)
        block_expert.extend([ex] * ((sel.size + pad) // tile_m))
    return np.array(out, dtype=np.int32), np.array(block_expert, dtype=np.int32)


@pytest.mark.parametrize("T,K,E,tile_m", [(16, 2, 8, 16), (64, 16, 896, 8), (300, 16, 112, 32),
                                          (1, 16, 896, 16), (0, 4, 8, 16), (257, 3, 5, 128)])
def test_sort_invariants_and_second_formulation(T, K, E, tile_m):
    rng = np.random.default_rng(T * 7 + K)
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    if T > 4:
        ids[3, 0] = E + 5   # out of range -> dropped
        ids[4, K - 1] = -1
    s = oracle.sort(ids, E, tile_m)
    ref_ids, ref_be = _sort_ref_numpy(ids, E, tile_m)
    assert np.array_equal(s["sorted_ids"], ref_ids)
    assert np.array_equal(s["block_expert"], ref_be)
    n = T * K
    flat = ids.ravel()
    valid = (flat >= 0) & (flat < E)
    assert s["dropped"] == int((~valid).sum())
    assert np.array_equal(s["expert_count"], np.bincount(flat[valid], minlength=E))
    real = s["sorted_ids"][s["sorted_ids"] < n]
    assert np.array_equal(np.sort(real), np.nonzero(valid)[0])  # each valid pair exactly once
    assert s["sorted_ids"].size == s["num_blocks"] * tile_m
    for b, ex in enumerate(s["block_expert"]):
        rows = s["sorted_ids"][b * tile_m:(b + 1) * tile_m]
        r = rows[rows < n]
        assert np.all(flat[r] == ex)                   # single-expert blocks
        assert np.all(np.diff(r) > 0)                  # ascending pair id
        assert np.all(rows[r.size:] == n)              # padding at the end only
    assert np.all(np.diff(s["expert_offset"]) % tile_m == 0)


def test_sort_brute_force_enumeration():
    """Every routing of T=2, K=2 over E=3 experts (with duplicates), tile 2."""
    E, tile_m = 3, 2
    for a in range(E):
        for b in range(E):
            for c in range(E):
                for d in range(E):
                    ids = np.array([[a, b], [c, d]], dtype=np.int32)
                    s = oracle.sort(ids, E, tile_m)
                    expect = []
                    for ex in range(E):
                        rows = [p for p, v in enumerate([a, b, c, d]) if v == ex]
                        if rows:
                            expect += rows + [4] * (len(rows) % 2)
                    assert s["sorted_ids"].tolist() == expect


def _situ_mp(g, u, b, lb):
    g, u = mp.mpf(g), mp.mpf(u)
    return b * mp.tanh(g / b) / (1 + mp.exp(-g)) * lb * mp.tanh(u / lb)


def _silu_mp(g, u):
    g, u = mp.mpf(g), mp.mpf(u)
    return g / (1 + mp.exp(-g)) * u


def test_situv2_closed_form_values():
    # beta = 4, linear beta = 25 (the Kimi-K3 values, aiter PR 6259 Motivation)
    table = [((1, 1), 0.715817828), ((-1, 2), -0.525828896), ((2, -3), -4.861066551),
             ((0.5, 0.5), 0.154788735)]
    for (g, u), v in table:
        got = oracle.act("situv2", g, u, 4.0, 25.0)
        assert abs(got - v) < 1e-9
    assert oracle.act("situv2", 0.0, 7.0, 4.0, 25.0) == 0.0


def test_act_against_mpmath():
    rng = np.random.default_rng(11)
    for g, u in rng.standard_normal((300, 2)) * rng.choice([0.1, 1, 10, 100], (300, 1)):
        for b, lb in [(4.0, 25.0), (2.0, 1.5), (1.0, 1.0)]:
            ref = float(_situ_mp(g, u, b, lb))
            got = oracle.act("situv2", g, u, b, lb)
            assert math.isclose(got, ref, rel_tol=1e-13, abs_tol=1e-300)
        assert math.isclose(oracle.act("silu", g, u, 4.0, 25.0), float(_silu_mp(g, u)), rel_tol=1e-13, abs_tol=1e-300)


def test_situv2_limits_and_saturation():
    # g -> +inf: situ(g) -> beta, y -> beta * up(u); g -> -inf: y -> 0
    for u in (-3.0, 0.5, 40.0):
        up = 25.0 * math.tanh(u / 25.0)
        assert math.isclose(oracle.act("situv2", 60.0, u, 4.0, 25.0), 4.0 * up, rel_tol=1e-12)
        assert abs(oracle.act("situv2", -60.0, u, 4.0, 25.0)) < 1e-20
    # up(u) = y / situ(g) at g = 200, where tanh(50) and sigmoid(200) are exactly 1 in fp64
    up = lambda u: oracle.act("situv2", 200.0, u, 4.0, 25.0) / 4.0
    assert abs(up(100.0) - 25.0) < 0.02 and abs(up(-100.0) + 25.0) < 0.02
    assert up(1000.0) == 25.0 and up(-1000.0) == -25.0


def test_silu_and_situv2_are_distinguishable():
    """A wrong activation must be visible (aiter PR 4471: cosine 0.9619 vs 0.99998)."""
    rng = np.random.default_rng(2)
    g, u = rng.standard_normal((2, 4096)) * 3
    a = np.array([oracle.act("silu", x, y, 4.0, 25.0) for x, y in zip(g, u)])
    b = np.array([oracle.act("situv2", x, y, 4.0, 25.0) for x, y in zip(g, u)])
    cos = a @ b / np.linalg.norm(a) / np.linalg.norm(b)
    assert cos < 0.99
    # and the beta pair matters: defaults (2.0, 1.5) vs (4.0, 25.0)
    c = np.array([oracle.act("situv2", x, y, 2.0, 1.5) for x, y in zip(g, u)])
    assert np.linalg.norm(b - c) / np.linalg.norm(b) > 0.2
