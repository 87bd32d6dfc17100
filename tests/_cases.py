"""Test-case builder: seeded inputs (quantized_moe_expert_sort_gb300.inputs),
MXFP4 weights quantised by the oracle, and helpers to compare with it.

Parity of outputs is judged per token: the largest relative L2 error of any
token's output row against the oracle's bf16 output (one wrong row cannot hide
in the norm of a large tensor). Requantised codes are judged element by element
against the oracle's fp32-held values: a code must be a nearest grid value of
that value under the scale chosen, and the scale must be the oracle's or, where
the block maximum sits on a power-of-two boundary, its neighbour (the GPU sums
in fp32, so values on a rounding boundary may land on either side)."""
import functools

import numpy as np
import torch

import oracle
from quantized_moe_expert_sort_gb300 import inputs

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def bf16_bits(x):
    return x.contiguous().view(torch.int16).numpy().astype(np.uint16)


def bits_to_f64(bits):
    return torch.tensor(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def token_rel_l2(got, ref):
    """Largest per-row relative L2 error (rows = tokens); a row whose reference is
    zero must be zero."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    r = np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num > 0, np.inf, 0.0))
    return float(r.max()) if r.size else 0.0


def gpu_f64(out):
    return out.float().cpu().numpy().astype(np.float64)


E2M1_GRID = np.unique(np.concatenate([-E2M1, E2M1]))
_E4M3_ALL = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
E4M3_GRID = np.unique(_E4M3_ALL[np.isfinite(_E4M3_ALL)])  # sorted, -0 and +0 as one value


def check_requant_rows(codes, scales, y32, a_dtype, tol=1e-3):
    """Requantised rows (codes [n, I*bytes], e8m0 scales [n, I/32]) against the
    oracle's fp32-held stage-1 output y32 [n, I]. Returns (fraction of elements
    whose value differs from the oracle's requantisation, fraction of scale bytes
    that differ); raises AssertionError on any code that is not a nearest grid
    value or any scale that is not the MX rule's (or its boundary neighbour)."""
    fmt = {"fp8": "e4m3", "fp4": "e2m1"}[a_dtype]
    grid = E4M3_GRID if fmt == "e4m3" else E2M1_GRID
    emax = 8 if fmt == "e4m3" else 2
    n, I = y32.shape
    codes = np.asarray(codes)
    sc = np.asarray(scales).astype(np.int64).reshape(n, I // 32)
    if fmt == "e2m1":
        lo, hi = codes & 15, codes >> 4
        c = np.stack([lo, hi], axis=-1).reshape(n, I)
        q = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
    else:
        q = torch.tensor(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    blk = np.abs(y32).reshape(n, I // 32, 32).max(axis=-1)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(blk > 0, blk, 1.0))
    e_or = np.clip(np.floor(lg) - emax, -127, 127)
    e_gpu = sc - 127
    zero = blk == 0
    assert np.all(sc[zero] == 127), "an all-zero block must get scale 127"
    near_pow2 = np.abs(lg - np.round(lg)) <= 1e-4
    ok_scale = (e_gpu == e_or) | ((np.abs(e_gpu - e_or) == 1) & near_pow2)
    assert np.all(ok_scale | zero), "scale bytes off the MX rule at %s" % (np.argwhere(~(ok_scale | zero))[:5],)
    s_val = y32 * np.repeat(np.exp2(-e_gpu.astype(np.float64)), 32, axis=-1)
    s_clip = np.clip(s_val, grid[0], grid[-1])
    idx = np.clip(np.searchsorted(grid, s_clip), 1, len(grid) - 1)
    best = np.minimum(np.abs(grid[idx] - s_clip), np.abs(grid[idx - 1] - s_clip))
    dist = np.abs(q - s_clip)
    bad = dist > best + tol * np.maximum(1.0, np.abs(s_clip))
    assert not np.any(bad), "codes not nearest at %s" % (np.argwhere(bad)[:5],)
    c_o, s_o = oracle.mx_quantize(np.ascontiguousarray(y32), fmt)
    ref = oracle.mx_dequantize(c_o, s_o, fmt)
    got = q * np.repeat(np.exp2(e_gpu.astype(np.float64)), 32, axis=-1)
    return float(np.mean(got != ref)), float(np.mean(sc != s_o.reshape(n, -1)))


def quantized_experts(experts, H, I, seed, E):
    """Oracle-quantised MXFP4 weights; experts not in `experts` stay zero
    (never read by a routing that does not touch them)."""
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    w13s = np.zeros((E, 2 * I, H // 32), np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    w2s = np.zeros((E, H, I // 32), np.uint8)
    for e in sorted(set(int(v) for v in experts)):
        c, s = oracle.quantize_weights(inputs.expert_w13(e, H, I, seed).numpy())
        w13[e], w13s[e] = c, s
        c, s = oracle.quantize_weights(inputs.expert_w2(e, H, I, seed).numpy())
        w2[e], w2s[e] = c, s
    return w13, w13s, w2, w2s


@functools.lru_cache(maxsize=3)
def _weights_cached(key, H, I, seed, E):
    experts = np.frombuffer(key, dtype=np.int32)
    return quantized_experts(experts, H, I, seed, E)


def make_case(T, H, I, E, K, routing, seed, experts_all=False, x=None):
    x = inputs.make_x(T, H, seed) if x is None else x
    ids, w = inputs.make_routing(T, E, K, routing, seed)
    ids_np = ids.numpy()
    touched = np.arange(E, dtype=np.int32) if experts_all else np.unique(ids_np[(ids_np >= 0) & (ids_np < E)]).astype(np.int32)
    w13, w13s, w2, w2s = _weights_cached(touched.tobytes(), H, I, seed, E)
    return dict(x=x, x_bits=bf16_bits(x), ids=ids, w=w, w13=w13, w13s=w13s, w2=w2, w2s=w2s,
                T=T, H=H, I=I, E=E, K=K)


def oracle_forward(case, act, a_dtype, subset=None, want_inter=False, ids=None, w=None, beta=4.0, lbeta=25.0):
    ids = case["ids"] if ids is None else ids
    w = case["w"] if w is None else w
    return oracle.moe_forward(case["x_bits"], np.asarray(ids), np.asarray(w), case["w13"], case["w13s"],
                              case["w2"], case["w2s"], act, beta, lbeta, a_dtype, tile_m=16,
                              subset=subset, want_inter=want_inter)


def to_dev(case, device="cuda"):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return dict(x=case["x"].to(device), ids=case["ids"].to(device), w=case["w"].to(device),
                w13=t(case["w13"]), w13s=t(case["w13s"]), w2=t(case["w2"]), w2s=t(case["w2s"]))


def decode_intermediate(codes, scales, fmt):
    """Decode the (codes, scales, fmt) triple of MoE.intermediate() to float64."""
    if fmt.startswith("e2m1x"):  # a sum of e2m1 code terms
        n = int(fmt[5:])
        hb, nb = codes.shape[1] // n, scales.shape[1] // n
        return sum(decode_codes(codes[:, t * hb:(t + 1) * hb], scales[:, t * nb:(t + 1) * nb], "fp4") for t in range(n))
    return decode_codes(codes, scales, {"f16": "bf16", "e4m3": "fp8", "e2m1": "fp4"}[fmt])


def decode_codes(codes, scales, a_dtype):
    """Decode GPU activation / intermediate codes to float64 (test-side decoder)."""
    codes = np.asarray(codes)
    scales = np.asarray(scales).astype(np.float64)
    if a_dtype == "bf16":
        v = codes.view(np.float16).astype(np.float64)
    elif a_dtype == "fp8":
        v = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        lo, hi = codes & 15, codes >> 4
        c = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
        v = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
    return v * np.repeat(np.exp2(scales - 127), 32, axis=-1)
