"""Pins for the oracle's number formats and its MX 1x32 quantiser.

Each check compares the oracle with something other than itself: the literal
OCP MX e2m1 table, torch's own float8_e4m3fn / bfloat16 conversions, brute-force
nearest-value search over every code, and closed-form properties of the scale rule.
"""
import math

import numpy as np
import pytest
import torch

import oracle

# OCP MX e2m1 magnitudes, codes 0..7 (sign is bit 3).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_decode_ref(codes):
    codes = np.asarray(codes)
    mag = np.array(E2M1_TABLE)[codes & 7]
    return np.where(codes & 8, -mag, mag)


def e4m3_decode_ref(bytes_):
    t = torch.tensor(np.asarray(bytes_, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e2m1_exhaustive_table():
    for c in range(16):
        v = oracle.e2m1_value(c)
        ref = E2M1_TABLE[c & 7] * (-1 if c & 8 else 1)
        assert v == ref, c
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0), c  # signed zero at code 8


def test_e4m3_full_byte_table():
    ref = e4m3_decode_ref(np.arange(256))
    for b in range(256):
        v = oracle.e4m3_value(b)
        if np.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b], b
            assert math.copysign(1.0, v) == math.copysign(1.0, ref[b]), b
    assert oracle.e4m3_value(0x7E) == 448.0


def test_e8m0_full_byte_table():
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_e2m1_decode_times_every_scale():
    """All 16 codes x 255 finite scales through the block dequantiser."""
    codes = np.arange(16, dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)  # 8 bytes = 16 elements
    row = np.concatenate([packed, packed])  # one 32-block
    for s in range(255):
        out = oracle.mx_dequantize(row[None, :], np.array([[s]], dtype=np.uint8), "e2m1")[0]
        ref = np.concatenate([e2m1_decode_ref(codes), e2m1_decode_ref(codes)]) * math.ldexp(1.0, s - 127)
        assert np.array_equal(out, ref), s


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        rng.standard_normal(2000) * 1e-40,  # bf16 subnormals
        np.array([3.3895313892515355e38, 3.3961e38, -3.4e38, 1.0, -2.0, 0.0]),
    ]).astype(np.float32).astype(np.float64)
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_from_f64(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_single_rounding_from_f64():
    # 1 + 2^-8 is the tie between bf16 neighbours 1 and 1 + 2^-7; a double just
    # above it must round up, although its fp32 rounding lands on the tie.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_from_f64(v) == 0x3F81
    assert oracle.bf16_from_f64(1.0 + 2.0 ** -8) == 0x3F80  # exact tie -> even
    assert oracle.bf16_from_f64(1.0 + 3 * 2.0 ** -8) == 0x3F82


def _brute_nearest(x, values, codes):
    """Nearest representable value; ties go to the code whose mantissa LSB is 0."""
    d = np.abs(x[:, None] - values[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & ((codes[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    return values[pick]


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_block_quantizer_rne_brute_force(fmt):
    """Element rounding of the block quantiser vs brute-force nearest search.
    Each block carries an anchor at 2^emax so that its scale is 2^0."""
    rng = np.random.default_rng(7 if fmt == "e2m1" else 8)
    if fmt == "e2m1":
        pos = np.arange(8)
        values, codes, anchor, vmax = e2m1_decode_ref(pos), pos, 4.0, 6.0
    else:
        pos = np.array([b for b in range(128) if b != 0x7F])
        values, codes, anchor, vmax = e4m3_decode_ref(pos), pos, 256.0, 448.0
    nblk = 33000
    x = rng.uniform(-1, 1, (nblk, 31)) * (anchor * 1.999)
    x = x * np.where(rng.random((nblk, 31)) < 0.5, 1.0, rng.uniform(0, 1, (nblk, 31)) ** 4)
    # exact ties between neighbours, too
    mids = (values[1:] + values[:-1]) / 2
    x[:2000, :] = rng.choice(mids, (2000, 31)) * rng.choice([-1, 1], (2000, 31))
    x = np.clip(x, -(anchor * 1.999), anchor * 1.999)  # keep amax in [2^emax, 2^(emax+1))
    blocks = np.concatenate([np.full((nblk, 1), anchor), x], axis=1)
    c, s = oracle.mx_quantize(blocks, fmt)
    assert np.all(s == 127)
    if fmt == "e2m1":
        lo, hi = c & 15, c >> 4
        dec_codes = np.stack([lo, hi], axis=-1).reshape(nblk, 32)
        dec = e2m1_decode_ref(dec_codes)
    else:
        dec = e4m3_decode_ref(c)
    ref_mag = _brute_nearest(np.abs(blocks.ravel()), values, codes).reshape(blocks.shape)
    assert np.array_equal(np.abs(dec), ref_mag)
    nz = ref_mag != 0
    assert np.array_equal(np.sign(dec[nz]), np.sign(blocks[nz]))


@pytest.mark.parametrize("fmt,emax", [("e2m1", 2), ("e4m3", 8)])
def test_scale_rule_floor_log2(fmt, emax):
    rng = np.random.default_rng(3)
    nblk = 4000
    x = rng.standard_normal((nblk, 32)) * np.exp2(rng.integers(-60, 60, (nblk, 1)))
    c, s = oracle.mx_quantize(x, fmt)
    amax = np.abs(x).max(axis=1)
    expect = np.array([math.frexp(a)[1] - 1 - emax + 127 for a in amax])
    assert np.array_equal(s.ravel().astype(int), expect)
    deq = oracle.mx_dequantize(c, s, fmt)
    # with that scale the block maximum lands in the top binade of the format
    top = np.abs(deq).max(axis=1) / np.exp2(s.ravel().astype(float) - 127)
    assert np.all(top >= 2.0 ** emax)


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_zero_block_and_signed_zero(fmt):
    z = np.zeros((1, 32))
    c, s = oracle.mx_quantize(z, fmt)
    assert s[0, 0] == 127 and not c.any()
    v = np.zeros((1, 32))
    v[0, 0] = 1.0
    v[0, 1] = -1e-30  # rounds to zero, keeps its sign
    c, s = oracle.mx_quantize(v, fmt)
    if fmt == "e2m1":
        assert (c[0, 0] >> 4) == 8
    else:
        assert c[0, 1] == 0x80


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_roundtrip_of_representable_values(fmt):
    if fmt == "e2m1":
        vals = e2m1_decode_ref(np.arange(16))
    else:
        vals = e4m3_decode_ref(np.array([b for b in range(256) if b not in (0x7F, 0xFF)]))
    rng = np.random.default_rng(5)
    for E in (-20, -3, 0, 5, 40):
        blk = rng.choice(vals, (200, 32)) * math.ldexp(1.0, E)
        blk[:, 0] = (6.0 if fmt == "e2m1" else 448.0) * math.ldexp(1.0, E)
        c, s = oracle.mx_quantize(blk, fmt)
        assert np.array_equal(oracle.mx_dequantize(c, s, fmt), blk)


def test_quantize_input_precisions_agree():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    xb = torch.tensor(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().astype(np.uint16)
    for fmt in ("e2m1", "e4m3"):
        a = oracle.mx_quantize(bits, fmt)
        b = oracle.mx_quantize(xb.to(torch.float64).numpy(), fmt)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
