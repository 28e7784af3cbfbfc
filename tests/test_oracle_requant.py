"""Pins of the oracle's FP8 requantisation (no GPU).

The requantisation is that of "W4AFP8 requant ..." (sglang PR #35760,
_fp8_per_token_quant_to_per_tensor_quant_kernel / _requant_row): each valid
element becomes e4m3(fp32(fp32(x * s) * r)), r = fp32(1 / S) -- the page's two
multiplies per element.  Pins, each independent of the oracle's own code:
  * the E4M3 encoder against every finite code (round trip), against torch's
    float8_e4m3fn cast (round to nearest, ties to even) on random values and on
    every exact midpoint, and against the saturation rule beyond 448;
  * the requantisation against a numpy / torch brute force (float32 products in
    the same order, torch's cast, explicit clamp at 448), in both scale layouts;
  * the identity closed form (s = 1, S = 1 leaves every code unchanged) and
    untouched rows past masked_m.
"""
import numpy as np
import torch

import oracle
from weight_only_bit_moe_gb300 import workloads as wk

FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def e4m3_values(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def torch_encode(v):
    """float32 -> E4M3 byte by torch's cast, after clamping to +-448."""
    t = torch.from_numpy(np.clip(np.asarray(v, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_round_trip_every_code(orc):
    for c in FINITE:
        v = float(e4m3_values([c])[0])
        assert orc.e4m3_encode(v) == c, hex(c)


def test_encode_matches_torch_cast(orc):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000), rng.normal(0, 0.01, 2000),
                        rng.uniform(-2 ** -6, 2 ** -6, 2000)]).astype(np.float32)
    got = np.array([orc.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(got, torch_encode(v))


def test_encode_ties_to_even(orc):
    pos = sorted(FINITE[:0x7F], key=lambda c: float(e4m3_values([c])[0]))
    vals = e4m3_values(pos)
    for lo, hi, a, b in zip(pos, pos[1:], vals, vals[1:]):
        mid = np.float32((np.float64(a) + np.float64(b)) / 2)
        assert float(mid) == (float(a) + float(b)) / 2  # exact in fp32
        want = lo if lo % 2 == 0 else hi
        assert orc.e4m3_encode(float(mid)) == want, (a, b)
        assert orc.e4m3_encode(-float(mid)) == want | 0x80


def test_encode_saturates_and_nan(orc):
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, float("inf")):
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE
    assert orc.e4m3_encode(float("nan")) == 0x7F
    assert orc.e4m3_encode(-0.0) == 0x80 and orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal: ties to 0
    assert orc.e4m3_encode(1.5 * 2.0 ** -10) == 0x01


def brute(x, scale_gm, mm, S, group):
    """numpy brute force: scale_gm [E, G, max_m]; float32 (x * s) * r, clamp, torch cast."""
    E, max_m, K = x.shape
    xv = e4m3_values(x.reshape(-1)).reshape(x.shape)
    s = np.repeat(np.transpose(scale_gm, (0, 2, 1)), group, axis=2)  # [E, max_m, K]
    r = np.float32(1.0) / np.float32(S)
    t = (xv.astype(np.float32) * s.astype(np.float32)).astype(np.float32) * r
    q = torch_encode(t.astype(np.float32).reshape(-1)).reshape(x.shape)
    out = np.zeros_like(x)
    for e in range(E):
        n = min(max(int(mm[e]), 0), max_m)
        out[e, :n] = q[e, :n]
    return out


def test_requant_matches_brute_force_both_layouts(orc):
    wl = wk.RequantWorkload("t", E=5, max_m=7, K=384, rows="random")
    X = wk.make_requant(wl, 3)
    X.masked_m[1] = 0
    X.masked_m[2] = 99  # clamped to max_m
    want = brute(X.x, X.scale, X.masked_m, X.tensor_scale, 128)
    got = orc.requant(X.x, X.scale, X.masked_m, X.tensor_scale)
    np.testing.assert_array_equal(got, want)
    row_major = np.ascontiguousarray(np.transpose(X.scale, (0, 2, 1)))  # [E, max_m, G]
    G = wl.K // 128
    got2 = orc.requant(X.x, row_major, X.masked_m, X.tensor_scale, scale_strides=(wl.max_m * G, 1, G))
    np.testing.assert_array_equal(got2, want)


def test_requant_group_64(orc):
    wl = wk.RequantWorkload("t", E=3, max_m=4, K=256, rows="random", group=64)
    X = wk.make_requant(wl, 5)
    want = brute(X.x, X.scale, X.masked_m, X.tensor_scale, 64)
    np.testing.assert_array_equal(orc.requant(X.x, X.scale, X.masked_m, X.tensor_scale, group=64), want)


def test_requant_identity_and_untouched_rows(orc):
    E, max_m, K = 2, 3, 256
    x = np.array(FINITE * ((E * max_m * K) // len(FINITE) + 1), dtype=np.uint8)[: E * max_m * K].reshape(E, max_m, K)
    ones = np.ones((E, K // 128, max_m), dtype=np.float32)
    mm = np.array([3, 1], dtype=np.int32)
    canvas = np.full_like(x, 0xA5)
    got = orc.requant(x, ones, mm, 1.0, out=canvas)
    np.testing.assert_array_equal(got[0], x[0])
    np.testing.assert_array_equal(got[1, :1], x[1, :1])
    assert np.all(got[1, 1:] == 0xA5)
