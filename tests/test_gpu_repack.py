"""The repacked blob, read back and decoded on the host, against its sources.

moe_repack_weights writes the tile-native layout that the kernels stream: per
expert and 256-row tile a sequence of 64-element K-stages, each a block of
fragment-ordered 4-bit codes with the scale block in front of the stage that
first needs it (INT4 one bf16 per 128, MXFP4 two E8M0 bytes per stage, NVFP4
four E4M3 bytes), then the deinterleaved, zero-padded biases, the per-expert
fp32 epilogue factors and the per-expert scale-exponent shifts.  This test
decodes that layout with numpy, from the layout's description alone, and checks
every code, scale, bias and factor byte for byte against the checkpoint tensors
(after the deinterleave and padding of "SM120 MXFP4 MoE ... Marlin", sglang PR
#28231: deinterleave_moe_mxfp4_w13_for_marlin, _pad_w13 / _pad_w2), so a layout
slip shows here rather than only in downstream parity.
"""
import dataclasses

import numpy as np
import pytest
import torch

from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import GPU_SMALL, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def rup(a, b):
    return (a + b - 1) // b * b


def packed_fmt(W):
    """int4 banks with zero points or groups below 128 pack one (multiplier, zero)
    entry per row and 32-column half stage ("int4x")."""
    if W.fmt == "int4" and (W.zero_kind or 0 < W.group < 128):
        return "int4x"
    return W.fmt


def layout(W):
    """Byte offsets of the blob's sections (the layout the kernels read)."""
    pf = packed_fmt(W)
    int4, nv = pf == "int4", pf == "nvfp4"
    gated = W.gated
    f1 = 128 if gated else 256
    Npad, Kpad2 = rup(W.N, f1), rup(W.K, 256)
    T1, T2, S1, S2 = Npad // f1, Kpad2 // 256, W.K // 64, Npad // 64
    period = 2 if int4 else 1
    scale_bytes = 256 * (8 if pf == "int4x" else (4 if nv else 2))
    period_bytes = scale_bytes + period * 8192
    tile1, tile2 = (S1 // period) * period_bytes, (S2 // period) * period_bytes
    off = 256
    d = dict(Npad=Npad, Kpad2=Kpad2, T1=T1, T2=T2, S1=S1, S2=S2, period=period, scale_bytes=scale_bytes,
             period_bytes=period_bytes, tile1=tile1, tile2=tile2, w13=off)
    off += W.E * T1 * tile1
    d["w2"] = off = rup(off, 256)
    off += W.E * T2 * tile2
    d["b13"] = off = rup(off, 256)
    if W.b13 is not None:
        off += W.E * (2 if gated else 1) * Npad * 2
    d["b2"] = off = rup(off, 256)
    if W.b2 is not None:
        off += W.E * Kpad2 * 2
    d["gs13"] = off = rup(off, 256)
    off += W.E * 4
    d["gs2"] = off = rup(off, 256)
    off += W.E * 4
    d["shift"] = off = rup(off, 256)
    off += 2 * W.E * 4
    d["perm13"] = off = rup(off, 256)
    if W.w13_perm is not None:
        off += W.E * W.K * 4
    d["total"] = rup(off, 256)
    d["fmt"] = pf
    return d


def stage_codes(blob, base, L, s):
    """The 64 codes of each of the 256 rows of stage s of the tile at `base`: uint8 [256, 64]."""
    q, r = divmod(s, L["period"])
    start = base + q * L["period_bytes"] + L["scale_bytes"] + r * 8192
    units = blob[start:start + 8192].view(np.uint32).reshape(2, 256, 4)  # [j][row][word]
    words = np.concatenate([units[0], units[1]], axis=1)                  # [row][v], v = 4j + w
    out = np.zeros((256, 64), dtype=np.uint8)
    int4 = L["fmt"] in ("int4", "int4x")
    for v in range(8):
        t, h = v >> 1, v & 1
        for p in range(4):
            k = 32 * h + 2 * t + 8 * p
            lo_shift, hi_shift = (4 * p, 16 + 4 * p) if int4 else (8 * p, 8 * p + 4)
            out[:, k] = (words[:, v] >> lo_shift) & 15
            out[:, k + 1] = (words[:, v] >> hi_shift) & 15
    return out


def stage_scales(blob, base, L, q):
    """Scale block of chunk q (stage q * period): [256, entries] raw values."""
    start = base + q * L["period_bytes"]
    if L["fmt"] == "int4":
        return blob[start:start + 512].view(np.uint16).reshape(256, 1)
    if L["fmt"] == "int4x":  # (m, x) f16 pairs of both 32-column halves
        return blob[start:start + 2048].view(np.uint16).reshape(256, 4)
    if L["fmt"] == "mxfp4":
        return blob[start:start + 512].reshape(256, 2)
    return blob[start:start + 1024].reshape(256, 4)


def unpack_matrix(blob, L, W, which):
    """Decode one expert matrix bank: codes uint8 [E, rows, red] and scales [E, rows, red/g]
    in the kernels' tile row order (tile rows, before source-row mapping)."""
    T = L["T2"] if which else L["T1"]
    S = L["S2"] if which else L["S1"]
    tile_bytes = L["tile2"] if which else L["tile1"]
    off = L["w2"] if which else L["w13"]
    per_chunk = {"int4": 1, "int4x": 4, "mxfp4": 2, "nvfp4": 4}[L["fmt"]]
    codes = np.zeros((W.E, T * 256, S * 64), dtype=np.uint8)
    scales = np.zeros((W.E, T * 256, S // L["period"] * per_chunk),
                      dtype=np.uint16 if L["fmt"] in ("int4", "int4x") else np.uint8)
    for e in range(W.E):
        for t in range(T):
            base = off + (e * T + t) * tile_bytes
            for s in range(S):
                codes[e, t * 256:(t + 1) * 256, s * 64:(s + 1) * 64] = stage_codes(blob, base, L, s)
            for q in range(S // L["period"]):
                scales[e, t * 256:(t + 1) * 256, q * per_chunk:(q + 1) * per_chunk] = stage_scales(blob, base, L, q)
    return codes, scales


def nibbles(packed):
    q = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    q[..., 0::2] = packed & 15
    q[..., 1::2] = packed >> 4
    return q


def tile_row_sources(W, L, which, e=0):
    """Source row (or -1 for padding) of each tile row of expert e, as the layout
    defines it (act-order banks put w13's features in w2's sort order)."""
    if which:
        return np.array([r if r < W.K else -1 for r in range(L["T2"] * 256)])
    feat = (lambda f: int(W.w2_perm[e, f])) if W.w2_perm is not None else (lambda f: f)
    rows = []
    for t in range(L["T1"]):
        for r in range(256):
            if not W.gated:
                f = t * 256 + r
                rows.append(feat(f) if f < W.N else -1)
                continue
            f, half = t * 128 + (r & 127), r >> 7
            if f >= W.N:
                rows.append(-1)
            else:
                sf = feat(f)
                rows.append(2 * sf + half if W.interleaved else half * W.N + sf)
    return np.array(rows)


def bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bank(W):
    from weight_only_bit_moe_gb300.layer import MoELayer
    layer = MoELayer.from_numpy(W)
    blob = layer.packed.cpu().numpy()
    L = layout(W)
    assert blob.size == L["total"]
    shift = blob[L["shift"]:L["shift"] + 8 * W.E].view(np.int32).reshape(2, W.E)
    assert blob[:4].view(np.uint32)[0] == 0, "window flag set for in-window scales"
    zero_code = 8 if W.fmt == "int4" else 0
    for which in (0, 1):
        codes, scales = unpack_matrix(blob, L, W, which)
        src_codes = nibbles(W.w2 if which else W.w13)
        src_scales = W.w2_s if which else W.w13_s
        src_z = W.w2_z if which else W.w13_z
        perm = W.w2_perm if which else W.w13_perm  # packed column k holds checkpoint column perm[k]
        red = W.N if which else W.K
        ng = 1 if W.group < 0 else red // W.group
        for e in range(W.E):
            cols = perm[e] if perm is not None else np.arange(red)
            for tr, sr in enumerate(tile_row_sources(W, L, which, e)):
                if sr < 0:
                    assert np.all(codes[e, tr] == zero_code), f"padding row {tr} of matrix {which}"
                    continue
                np.testing.assert_array_equal(codes[e, tr, :red], src_codes[e, sr, cols], err_msg=f"codes row {tr}")
                assert np.all(codes[e, tr, red:] == zero_code)
                scale_f = np.ldexp(1.0, shift[which][e])
                if L["fmt"] == "int4x":  # entry of 32-column block b: m = s * 2^d, x = 1024 + z / -z m / 1032
                    nb = red // 32
                    grp = np.arange(nb) * 32 // (red if W.group < 0 else W.group)
                    ent = scales[e, tr, :2 * nb].reshape(nb, 2)
                    s_sh = bf16_f64(src_scales[e, sr, grp]) * scale_f
                    np.testing.assert_array_equal(ent[:, 0], s_sh.astype(np.float16).view(np.uint16))
                    if W.zero_kind == "int":
                        want_x = (1024.0 + src_z[e, sr, grp]).astype(np.float16)
                    elif W.zero_kind == "float":
                        want_x = (-bf16_f64(src_z[e, sr, grp]) * s_sh).astype(np.float32).astype(np.float16)
                    else:
                        want_x = np.full(nb, 1032.0, np.float16)
                    np.testing.assert_array_equal(ent[:, 1], want_x.view(np.uint16), err_msg=f"entries row {tr}")
                elif W.fmt == "int4":  # stored s * 2^d, a power-of-two shift per expert matrix
                    nch = red // 128
                    grp = np.arange(nch) * 128 // (red if W.group < 0 else W.group)
                    np.testing.assert_array_equal(bf16_f64(scales[e, tr, :nch]),
                                                  bf16_f64(src_scales[e, sr, grp]) * scale_f)
                elif W.fmt == "mxfp4":
                    want = src_scales[e, sr].astype(np.int64) + shift[which][e]
                    np.testing.assert_array_equal(scales[e, tr, :ng].astype(np.int64), want)
                else:
                    assert shift[which][e] == 0
                    np.testing.assert_array_equal(scales[e, tr, :ng], src_scales[e, sr])
    # biases: deinterleaved gate | up halves padded to Npad (GEMM1), K padded to Kpad2 (GEMM2)
    if W.b13 is not None:
        halves = 2 if W.gated else 1
        b13 = blob[L["b13"]:L["b13"] + W.E * halves * L["Npad"] * 2].view(np.uint16).reshape(W.E, halves, L["Npad"])
        for e in range(W.E):
            for f in range(L["Npad"]):
                for h in range(halves):
                    if f >= W.N:
                        assert b13[e, h, f] == 0
                        continue
                    sf = int(W.w2_perm[e, f]) if W.w2_perm is not None else f
                    row = (2 * sf + h if W.interleaved else h * W.N + sf) if W.gated else sf
                    assert b13[e, h, f] == W.b13[e, row]
    if W.w13_perm is not None:
        perm13 = blob[L["perm13"]:L["perm13"] + W.E * W.K * 4].view(np.int32).reshape(W.E, W.K)
        np.testing.assert_array_equal(perm13, W.w13_perm)
    if W.b2 is not None:
        b2 = blob[L["b2"]:L["b2"] + W.E * L["Kpad2"] * 2].view(np.uint16).reshape(W.E, L["Kpad2"])
        np.testing.assert_array_equal(b2[:, :W.K], W.b2)
        assert np.all(b2[:, W.K:] == 0)
    # epilogue factors: 2^-d (INT4 and its variants), 256 * 2^-d (MXFP4), 256 * gs (NVFP4)
    gs13 = blob[L["gs13"]:L["gs13"] + 4 * W.E].view(np.float32)
    gs2 = blob[L["gs2"]:L["gs2"] + 4 * W.E].view(np.float32)
    for g, which, src in ((gs13, 0, W.w13_gs), (gs2, 1, W.w2_gs)):
        want = np.ldexp(1.0, -shift[which]) * (256.0 if W.fmt != "int4" else 1.0)
        if W.fmt == "nvfp4":
            want = want * src.astype(np.float64)
        np.testing.assert_array_equal(g.astype(np.float64), want.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("name", ["int4-bias-small", "mxfp4-alpha-small", "nvfp4-ep-small", "int4-relu2-small",
                                  "mxfp4-relu2-small", "tiny-int4"])
def test_repack_round_trip(name):
    wl = GPU_SMALL[name]
    check_bank(wk.make_weights(wl, 7))


def test_repack_round_trip_shifted_scales():
    """Scales outside the fp16 window are stored shifted by a power of two per expert
    matrix (INT4 1e-6 scales, MXFP4 bytes 100..110), and the factor undoes it."""
    wl = dataclasses.replace(GPU_SMALL["int4-bias-small"], E=3)
    W = wk.make_weights(wl, 9)
    rng = np.random.default_rng(9)
    W.w13_s = wk.to_bf16_bits(rng.uniform(1e-6, 2e-6, size=W.w13_s.shape).astype(np.float32))
    check_bank(W)
    wl = dataclasses.replace(GPU_SMALL["mxfp4-alpha-small"], E=3)
    W = wk.make_weights(wl, 10)
    W.w13_s = rng.integers(100, 111, size=W.w13_s.shape).astype(np.uint8)
    check_bank(W)


@pytest.mark.parametrize("variant", ["zp-int-g64", "zp-float-g32", "sym-g32", "channelwise", "actorder-g128",
                                     "actorder-zp-g64"])
def test_repack_round_trip_int4_variants(variant):
    """Zero-point / small-group entries, whole-row groups and act-order
    permutations (columns in sort_indices order, w13 features in w2's order),
    decoded from the blob and compared with the checkpoint tensors."""
    base = dataclasses.replace(GPU_SMALL["int4-bias-small"], E=3, N=256)
    kw = {"zp-int-g64": dict(zero_kind="int", group_size=64), "zp-float-g32": dict(zero_kind="float", group_size=32),
          "sym-g32": dict(group_size=32), "channelwise": dict(group_size=-1), "actorder-g128": dict(act_order=True),
          "actorder-zp-g64": dict(act_order=True, zero_kind="int", group_size=64)}[variant]
    check_bank(wk.make_weights(dataclasses.replace(base, **kw), 12))
