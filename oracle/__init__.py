"""ctypes binding of the CPU fp64 oracle (oracle.c).

TEST INFRASTRUCTURE ONLY. The product path never imports this package; only
tests/, __graft_entry__.smoke() and bench.py's CPU baseline / reference leg
do. Every function here marshals numpy arrays into the C oracle; none of the
method's arithmetic lives in Python.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ACT = {"silu": 0, "situv2": 1}
ADTYPE = {"bf16": 0, "fp8": 1, "fp4": 2}
FMT = {"e2m1": 0, "e4m3": 1}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        d, i32, i64, u16, vp = ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_uint16, ctypes.c_void_p
        L.orc_e2m1_value.restype = d
        L.orc_e2m1_value.argtypes = [i32]
        L.orc_e4m3_value.restype = d
        L.orc_e4m3_value.argtypes = [i32]
        L.orc_e8m0_value.restype = d
        L.orc_e8m0_value.argtypes = [i32]
        L.orc_bf16_value.restype = d
        L.orc_bf16_value.argtypes = [u16]
        L.orc_bf16_from_f64.restype = u16
        L.orc_bf16_from_f64.argtypes = [d]
        L.orc_round_to_format.restype = d
        L.orc_round_to_format.argtypes = [d, i32]
        L.orc_encode.restype = i32
        L.orc_encode.argtypes = [d, i32]
        for name in ("orc_mx_quantize_f64", "orc_mx_quantize_f32", "orc_mx_quantize_bf16"):
            fn = getattr(L, name)
            fn.restype = None
            fn.argtypes = [vp, i64, i32, vp, vp]
        L.orc_mx_dequantize.restype = None
        L.orc_mx_dequantize.argtypes = [vp, vp, i64, i32, vp]
        L.orc_sort.restype = i64
        L.orc_sort.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.orc_act.restype = d
        L.orc_act.argtypes = [i32, d, d, d, d]
        L.orc_moe_forward.restype = i64
        L.orc_moe_forward.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                      i32, d, d, i32, i32, vp, i32, vp, vp, vp]
        L.orc_moe_dense.restype = i64
        L.orc_moe_dense.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                    i32, d, d, i32, vp, vp]
        L.orc_activation_row.restype = None
        L.orc_activation_row.argtypes = [vp, i32, i32, vp]
        L.orc_requantize_intermediate.restype = None
        L.orc_requantize_intermediate.argtypes = [vp, i32, i32, vp]
        L.orc_expert_stage1.restype = i64
        L.orc_expert_stage1.argtypes = [vp, vp, i32, i32, i32, vp, vp, i32, d, d, i32, vp, vp]
        L.orc_ep_forward.restype = i64
        L.orc_ep_forward.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                     i32, d, d, i32, i32, vp, i32, vp, vp]
        L.orc_route.restype = i64
        L.orc_route.argtypes = [vp, i32, i32, i32, vp, vp]
        L.orc_num_threads.restype = i32
        L.orc_num_threads.argtypes = []
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads():
    return lib().orc_num_threads()


def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e4m3_value(byte):
    return lib().orc_e4m3_value(int(byte))


def e8m0_value(byte):
    return lib().orc_e8m0_value(int(byte))


def bf16_value(bits):
    return lib().orc_bf16_value(int(bits))


def bf16_from_f64(v):
    return lib().orc_bf16_from_f64(float(v))


def round_to_format(x, fmt):
    return lib().orc_round_to_format(float(x), FMT[fmt])


def encode(r, fmt):
    return lib().orc_encode(float(r), FMT[fmt])


def mx_quantize(v, fmt):
    """Quantise the last axis (a multiple of 32) of v (float64, float32 or a
    uint16 array of bf16 bits) to MX codes + e8m0 scales."""
    v = np.asarray(v)
    n = v.shape[-1]
    assert n % 32 == 0
    nblocks = v.size // 32
    lead = v.shape[:-1]
    per = 16 if fmt == "e2m1" else 32
    codes = np.zeros(lead + (n // 32 * per,), dtype=np.uint8)
    scales = np.zeros(lead + (n // 32,), dtype=np.uint8)
    if v.dtype == np.uint16:
        lib().orc_mx_quantize_bf16(_p(_c(v, np.uint16)), nblocks, FMT[fmt], _p(codes), _p(scales))
    elif v.dtype == np.float32:
        lib().orc_mx_quantize_f32(_p(_c(v, np.float32)), nblocks, FMT[fmt], _p(codes), _p(scales))
    else:
        lib().orc_mx_quantize_f64(_p(_c(v, np.float64)), nblocks, FMT[fmt], _p(codes), _p(scales))
    return codes, scales


def mx_dequantize(codes, scales, fmt):
    scales = _c(scales, np.uint8)
    codes = _c(codes, np.uint8)
    nblocks = scales.size
    out = np.zeros(scales.shape[:-1] + (scales.shape[-1] * 32,), dtype=np.float64)
    lib().orc_mx_dequantize(_p(codes), _p(scales), nblocks, FMT[fmt], _p(out))
    return out


def sort(ids, E, tile_m):
    """The expert sort. Returns dict with sorted_ids, block_expert, num_blocks,
    expert_count, expert_offset, dropped."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    n = T * K
    cap = n + min(E, n) * (tile_m - 1) + tile_m
    sorted_ids = np.zeros(max(cap, 1), dtype=np.int32)
    block_expert = np.zeros(cap // tile_m + 1, dtype=np.int32)
    nb = np.zeros(1, dtype=np.int32)
    count = np.zeros(E, dtype=np.int32)
    offset = np.zeros(E + 1, dtype=np.int32)
    dropped = lib().orc_sort(_p(ids), T, K, E, tile_m, _p(sorted_ids), _p(block_expert), _p(nb),
                             _p(count), _p(offset))
    rows = int(offset[E])
    return dict(sorted_ids=sorted_ids[:rows].copy(), block_expert=block_expert[:int(nb[0])].copy(),
                num_blocks=int(nb[0]), expert_count=count, expert_offset=offset, dropped=int(dropped))


def act(kind, g, u, beta, lbeta):
    return lib().orc_act(ACT[kind], float(g), float(u), float(beta), float(lbeta))


def moe_forward(x_bf16, ids, w, w13, w13s, w2, w2s, act_kind, beta, lbeta, a_dtype,
                tile_m=16, subset=None, want_inter=False):
    """Grouped oracle forward. x_bf16: uint16 [T,H] (bf16 bits). Returns
    (out_f64 [n,H], out_bf16 uint16 [n,H], inter [n*K,I] or None, dropped)."""
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x_bf16.shape
    K = ids.shape[1]
    E = w13.shape[0]
    I = w13.shape[1] // 2
    sub = None if subset is None else _c(subset, np.int32)
    n = T if sub is None else sub.size
    out_f64 = np.zeros((n, H), dtype=np.float64)
    out_bf16 = np.zeros((n, H), dtype=np.uint16)
    inter = np.zeros((n * K, I), dtype=np.float64) if want_inter else None
    dropped = lib().orc_moe_forward(
        _p(x_bf16), _p(ids), _p(w), T, H, I, E, K,
        _p(_c(w13, np.uint8)), _p(_c(w13s, np.uint8)), _p(_c(w2, np.uint8)), _p(_c(w2s, np.uint8)),
        ACT[act_kind], float(beta), float(lbeta), ADTYPE[a_dtype], int(tile_m),
        _p(sub), n, _p(out_f64), _p(out_bf16), _p(inter))
    if dropped < 0:
        raise ValueError("oracle rejected the arguments")
    return out_f64, out_bf16, inter, int(dropped)


def moe_dense(x_bf16, ids, w, w13, w13s, w2, w2s, act_kind, beta, lbeta, a_dtype):
    """Brute-force per-token oracle (no sort). Returns (out_f64, out_bf16, dropped)."""
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x_bf16.shape
    K = ids.shape[1]
    E = w13.shape[0]
    I = w13.shape[1] // 2
    out_f64 = np.zeros((T, H), dtype=np.float64)
    out_bf16 = np.zeros((T, H), dtype=np.uint16)
    dropped = lib().orc_moe_dense(
        _p(x_bf16), _p(ids), _p(w), T, H, I, E, K,
        _p(_c(w13, np.uint8)), _p(_c(w13s, np.uint8)), _p(_c(w2, np.uint8)), _p(_c(w2s, np.uint8)),
        ACT[act_kind], float(beta), float(lbeta), ADTYPE[a_dtype], _p(out_f64), _p(out_bf16))
    if dropped < 0:
        raise ValueError("oracle rejected the arguments")
    return out_f64, out_bf16, int(dropped)


def activation_row(x_bits_row, a_dtype):
    """The stage-1 activation operand of one token (uint16 bf16 bits [H]) as float64 [H]."""
    x = _c(x_bits_row, np.uint16).reshape(-1)
    out = np.zeros(x.size, dtype=np.float64)
    lib().orc_activation_row(_p(x), x.size, ADTYPE[a_dtype], _p(out))
    return out


def requantize_intermediate(y, a_dtype):
    """One pair's stage-1 output y (float64 [I]) held in fp32 and requantised; float64 [I]."""
    y = _c(y, np.float64).reshape(-1)
    out = np.zeros(y.size, dtype=np.float64)
    lib().orc_requantize_intermediate(_p(y), y.size, ADTYPE[a_dtype], _p(out))
    return out


def expert_stage1(x_bits, tokens, w13e, w13se, act_kind, beta, lbeta, a_dtype):
    """Stage 1 of one expert for token rows `tokens` of x (uint16 bf16 bits [T,H]);
    w13e [2I,H/2], w13se [2I,H/32]. Returns (y32 [n,I], the fp32-held stage-1 output,
    yq [n,I], the requantised intermediate)."""
    x_bits = _c(x_bits, np.uint16)
    tokens = _c(tokens, np.int32).reshape(-1)
    H = x_bits.shape[1]
    I = w13e.shape[0] // 2
    n = tokens.size
    y32 = np.zeros((n, I), dtype=np.float64)
    yq = np.zeros((n, I), dtype=np.float64)
    st = lib().orc_expert_stage1(_p(x_bits), _p(tokens), n, H, I, _p(_c(w13e, np.uint8)), _p(_c(w13se, np.uint8)),
                                 ACT[act_kind], float(beta), float(lbeta), ADTYPE[a_dtype], _p(y32), _p(yq))
    if st != 0:
        raise ValueError("oracle rejected the arguments")
    return y32, yq


def ep_forward(x_bf16, ids, w, w13, w13s, w2, w2s, ranks, act_kind, beta, lbeta, a_dtype, wire=True,
               subset=None):
    """Expert-parallel oracle: `ranks` ranks own equal slices of the E experts; each
    rank's share of a token goes over an fp8 1x32 combine wire (wire=True) and the
    shares are summed. Returns (out_f64 [n,H], out_bf16 uint16 [n,H])."""
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x_bf16.shape
    K = ids.shape[1]
    E = w13.shape[0]
    I = w13.shape[1] // 2
    assert E % ranks == 0
    sub = None if subset is None else _c(subset, np.int32)
    n = T if sub is None else sub.size
    out_f64 = np.zeros((n, H), dtype=np.float64)
    out_bf16 = np.zeros((n, H), dtype=np.uint16)
    st = lib().orc_ep_forward(
        _p(x_bf16), _p(ids), _p(w), T, H, I, E // ranks, ranks, K,
        _p(_c(w13, np.uint8)), _p(_c(w13s, np.uint8)), _p(_c(w2, np.uint8)), _p(_c(w2s, np.uint8)),
        ACT[act_kind], float(beta), float(lbeta), ADTYPE[a_dtype], 1 if wire else 0, _p(sub), n,
        _p(out_f64), _p(out_bf16))
    if st != 0:
        raise ValueError("oracle rejected the arguments")
    return out_f64, out_bf16


def route(logits, K):
    """Top-k softmax router: logits fp32 [T,E] -> (ids int32 [T,K], weights float64 [T,K])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, K), dtype=np.int32)
    w = np.zeros((T, K), dtype=np.float64)
    if lib().orc_route(_p(logits), T, E, K, _p(ids), _p(w)) != 0:
        raise ValueError("oracle rejected the arguments")
    return ids, w


def quantize_weights(w_f32):
    """MXFP4-quantise fp32 weights [..., K] along K: (codes [..., K/2], scales [..., K/32])."""
    return mx_quantize(np.asarray(w_f32, dtype=np.float32), "e2m1")
