"""Pins of the oracle's format decoders and bf16 rounding against library routines
and exact arithmetic (no GPU).

The pages name the formats (uint4b8 in "Marlin MoE kernel occupancy ..." (sglang
PR #31552), test_fused_marlin_moe_large_non_ep_schedule; E2M1 with E8M0 scales in
"SM120 MXFP4 MoE ... Marlin" (sglang PR #28231); E2M1 with float8_e4m3fn scales in
"013-moe-middle-tiles.py", Weights) but do not define them, so the pins are the
public definitions as implemented by torch's float8 types and exact rationals.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch


def exact_rne_bf16(x: float) -> float:
    """Nearest bf16 to x by exact rational comparison (ties to even mantissa)."""
    if x == 0 or math.isnan(x):
        return x
    fx = Fraction(x)
    a = abs(fx)
    e = math.floor(math.log2(a))
    # fix floor(log2) for values near powers of two
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)
    lo = (a // q) * q
    hi = lo + q
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / q) % 2 == 0 else hi
    if r > Fraction(2) ** 127 * (2 - Fraction(1, 128)):
        return math.copysign(math.inf, x)
    return math.copysign(float(r), x)


def test_e2m1_all_codes(orc):
    # the eight E2M1 magnitudes, sign in bit 3
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for code in range(16):
        v = orc.e2m1_value(code)
        expect = mags[code & 7] * (-1 if code & 8 else 1)
        assert v == expect and math.copysign(1, v) == (-1 if code & 8 else 1), code


def test_e4m3_exhaustive_against_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        v = orc.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b], (b, v, ref[b])


def test_e8m0_exhaustive(orc):
    for b in range(256):
        v = orc.e8m0_value(b)
        if b == 255:
            assert math.isnan(v)
        else:
            assert v == math.ldexp(1.0, b - 127), b
    if hasattr(torch, "float8_e8m0fnu"):
        codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
        ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert all(orc.e8m0_value(b) == ref[b] for b in range(255))


def test_int4_uint4b8(orc):
    assert [orc.int4_value(q) for q in range(16)] == [float(q - 8) for q in range(16)]


def test_bf16_value_against_torch(orc):
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits[::13], ref[::13]):
        v = orc.bf16_value(int(b))
        assert (math.isnan(v) and math.isnan(r)) or v == r


def test_bf16_round_fp32_inputs_match_torch(orc):
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 3000),
        # exact ties: bf16 value plus half its quantum
        (np.arange(1, 300, dtype=np.float32) / 128 + 1) + np.float32(2.0 ** -8),
        np.array([1e-40, -3e-39, 1.2e-38, 3.3895e38, 3.4e38, -3.4e38, 0.0, -0.0], dtype=np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, r in zip(vals, ref):
        assert orc.bf16_round(float(v)) == int(r), (v, hex(orc.bf16_round(float(v))), hex(int(r)))


def test_bf16_round_fp64_inputs_exact(orc):
    # direct rounding of doubles (no intermediate fp32 step), checked by exact rationals
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(400) * 10.0 ** rng.integers(-40, 38, 400))
    vals += [1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -40), 2 ** -133,
             2 ** -134, 3 * 2 ** -135, 2 ** -127 * 1.5]
    for v in vals:
        got = orc.bf16_value(orc.bf16_round(v))
        assert got == exact_rne_bf16(v), (v, got, exact_rne_bf16(v))


def test_dequant_nibble_order_and_groups(orc):
    # one row, 8 elements: bytes 0x21, 0xF0, 0x87, 0x0C -> codes 1,2,0,15,7,8,12,0
    codes = np.array([[0x21, 0xF0, 0x87, 0x0C]], dtype=np.uint8)
    # int4, group 4: scales 0.5 (first four), 2.0 (last four) as bf16 bits
    sc = np.array([[0x3F00, 0x4000]], dtype=np.uint16)
    got = orc.dequant("int4", codes, sc, 4)[0]
    assert list(got) == [-3.5, -3.0, -4.0, 3.5, -2.0, 0.0, 8.0, -16.0]
    # mxfp4, group 4: exponents 2^-1 and 2^3
    sc = np.array([[126, 130]], dtype=np.uint8)
    got = orc.dequant("mxfp4", codes, sc, 4)[0]
    assert list(got) == [0.25, 0.5, 0.0, -3.0, 48.0, -0.0, -16.0, 0.0]
    # nvfp4, group 4: e4m3 0x38 = 1.0, 0x3C = 1.5
    sc = np.array([[0x38, 0x3C]], dtype=np.uint8)
    got = orc.dequant("nvfp4", codes, sc, 4)[0]
    assert list(got) == [0.5, 1.0, 0.0, -6.0, 9.0, -0.0, -3.0, 0.0]


@pytest.mark.parametrize("fmt,group", [("int4", 128), ("mxfp4", 32), ("nvfp4", 16)])
def test_dequant_matches_torch_decoders(orc, fmt, group):
    rng = np.random.default_rng(2)
    R, C = 24, 256
    codes = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    q = np.empty((R, C), dtype=np.int64)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    if fmt == "int4":
        s = torch.from_numpy(rng.uniform(0.005, 0.02, (R, C // group)).astype(np.float32)).to(torch.bfloat16)
        sbits = s.view(torch.int16).numpy().view(np.uint16)
        sval = s.to(torch.float64).numpy()
        val = (q - 8).astype(np.float64)
    else:
        e2m1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)
        val = e2m1[torch.from_numpy(q)].numpy()
        if fmt == "mxfp4":
            sbits = rng.integers(119, 124, size=(R, C // group)).astype(np.uint8)
            sval = torch.from_numpy(sbits).view(torch.float8_e8m0fnu).to(torch.float64).numpy() \
                if hasattr(torch, "float8_e8m0fnu") else np.ldexp(1.0, sbits.astype(np.int64) - 127)
        else:
            s = torch.from_numpy(rng.uniform(0.5, 2.0, (R, C // group)).astype(np.float32)).to(torch.float8_e4m3fn)
            sbits = s.view(torch.uint8).numpy()
            sval = s.to(torch.float64).numpy()
    expect = val * np.repeat(sval, group, axis=1)
    got = orc.dequant(fmt, codes, sbits, group)
    np.testing.assert_array_equal(got.astype(np.float64), expect)
    # row_map reads stored rows in the given order (used for interleaved gate/up rows)
    rm = np.array([2 * i for i in range(R // 2)] + [2 * i + 1 for i in range(R // 2)], dtype=np.int32)
    np.testing.assert_array_equal(orc.dequant(fmt, codes, sbits, group, rm), got[rm])
