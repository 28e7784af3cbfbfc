"""Pins of the oracle's INT4 variants (no GPU): zero points, act-order and
other group sizes -- the w*_zeros, is_zp_float, g_idx / sort_indices and
group_blocks of fused_marlin_moe and the Marlin template in "Marlin MoE kernel
occupancy ..." (sglang PR #31552).

Readings (the pages name these parameters but do not define their layouts):
  * an integer zero point is a byte 0..15 per (row, group), W = (q - z) * s;
    a float zero point (is_zp_float) is a bf16 value per (row, group), same
    formula; without zero points the codes are uint4b8, W = (q - 8) * s;
  * g_idx[k] is the group of reduction index k (act-order); sort_indices orders
    the indices by group; groups hold group_size indices each;
  * group sizes 32, 64, 128 or one group per row (-1, channelwise).

Pins, each independent of the oracle's loops:
  * dense brute force (numpy decode of every expert with the zeros and g_idx
    gathered by index, numpy matmuls, then routing) for every variant;
  * integer zero points all 8 equal the uint4b8 bank bit for bit;
  * act-order with g_idx = k // g (identity order) equals no act-order bit for
    bit; a random act-order bank equals the bank whose reduction indices are
    stored in sort_indices order with x's columns permuted the same way;
  * closed form: unit scales, every code c, every integer zero z: each weight
    is c - z;
  * channelwise equals group = K.
"""
import dataclasses
import math

import numpy as np
import pytest

from weight_only_bit_moe_gb300 import workloads as wk
from test_oracle_forward import bf16v, rne_bf16

BASE = dataclasses.replace(wk.WORKLOADS["int4-bias"], K=256, N=128, E=4, Ms=(9,))
VARIANTS = {
    "zp-int-g128": dataclasses.replace(BASE, zero_kind="int"),
    "zp-int-g64": dataclasses.replace(BASE, zero_kind="int", group_size=64),
    "zp-float-g32": dataclasses.replace(BASE, zero_kind="float", group_size=32),
    "sym-g32": dataclasses.replace(BASE, group_size=32),
    "sym-g64": dataclasses.replace(BASE, group_size=64),
    "channelwise": dataclasses.replace(BASE, group_size=-1),
    "actorder-g128": dataclasses.replace(BASE, act_order=True),
    "actorder-zp-g64": dataclasses.replace(BASE, act_order=True, zero_kind="int", group_size=64),
    "actorder-zpf-g32-relu2": dataclasses.replace(wk.WORKLOADS["int4-relu2"], K=256, N=128, E=4, Ms=(9,),
                                                  act_order=True, zero_kind="float", group_size=32),
}


def case(name, seed=3):
    wl = VARIANTS[name]
    return wl, wk.make_weights(wl, seed), wk.make_batch(wl, wl.Ms[0], seed + 1)


def decode(codes, scales, zeros, zero_kind, gidx, group):
    """numpy decode of [E, R, C/2] codes: group of index k by gidx or k // group."""
    q = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.int64)
    q[..., 0::2] = codes & 15
    q[..., 1::2] = codes >> 4
    E, R, C = q.shape
    if gidx is None:
        g = np.arange(C) // (C if group < 0 else group)
        g = np.broadcast_to(g, (E, C))
    else:
        g = gidx
    idx = np.broadcast_to(g[:, None, :], (E, R, C))
    s = np.take_along_axis(bf16v(scales), idx, axis=2)
    if zero_kind == "int":
        z = np.take_along_axis(zeros.astype(np.float64), idx, axis=2)
    elif zero_kind == "float":
        z = np.take_along_axis(bf16v(zeros), idx, axis=2)
    else:
        z = 8.0
    w = (q - z) * s
    return w.astype(np.float32).astype(np.float64)  # the oracle keeps weights in binary32


def dense(wl, W, X):
    N, K = W.N, W.K
    W13 = decode(W.w13, W.w13_s, W.w13_z, W.zero_kind, W.w13_gidx, W.group)
    W2 = decode(W.w2, W.w2_s, W.w2_z, W.zero_kind, W.w2_gidx, W.group)
    R = W13.shape[1]
    b13 = bf16v(W.b13) if W.b13 is not None else np.zeros((W.E, R))
    b2 = bf16v(W.b2) if W.b2 is not None else np.zeros((W.E, K))
    x = bf16v(X.x)
    out = np.zeros((x.shape[0], K))
    for t in range(x.shape[0]):
        for j in range(X.topk_ids.shape[1]):
            e = int(X.topk_ids[t, j])
            h = W13[e] @ x[t] + b13[e]
            if W.gated:
                g, u = h[:N], h[N:]
                a = g / (1 + np.exp(-g)) * u
            else:
                a = np.square(np.maximum(h, 0.0))
            out[t] += float(X.topk_weights[t, j]) * (W2[e] @ a + b2[e])
    return out


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_dense_bruteforce(orc, name):
    wl, W, X = case(name)
    bits, acc = orc.forward_workload(wl, W, X, return_acc=True)
    ref = dense(wl, W, X)
    np.testing.assert_allclose(acc, ref, rtol=1e-11, atol=1e-11)
    assert (bf16v(bits) == rne_bf16(ref)).mean() > 0.999
    assert np.abs(ref).max() > 0.0


def test_integer_zero_8_is_uint4b8(orc):
    wl, W, X = case("zp-int-g128")
    sym = dataclasses.replace(W, zero_kind="", w13_z=None, w2_z=None)
    eight = dataclasses.replace(W, w13_z=np.full_like(W.w13_z, 8), w2_z=np.full_like(W.w2_z, 8))
    np.testing.assert_array_equal(orc.forward_workload(wl, eight, X), orc.forward_workload(wl, sym, X))


def test_act_order_identity_equals_plain(orc):
    wl, W, X = case("zp-int-g64")
    ident13 = np.broadcast_to(np.arange(W.K, dtype=np.int32) // 64, (W.E, W.K)).copy()
    ident2 = np.broadcast_to(np.arange(W.N, dtype=np.int32) // 64, (W.E, W.N)).copy()
    A = dataclasses.replace(W, w13_gidx=ident13, w2_gidx=ident2)
    np.testing.assert_array_equal(orc.forward_workload(wl, A, X), orc.forward_workload(wl, W, X))


def _permute_codes(codes, perm):
    """[E, R, C/2] packed codes -> the same with each expert's columns in perm order."""
    q = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    q[..., 0::2] = codes & 15
    q[..., 1::2] = codes >> 4
    q = np.take_along_axis(q, perm[:, None, :].astype(np.int64), axis=2)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def test_act_order_equals_sorted_storage(orc):
    """One expert (so x's columns can follow its order): the act-order bank equals
    the bank stored in sort_indices order, groups contiguous, with x permuted alike;
    w2's order is folded into w13's output rows and w2's columns."""
    wl = dataclasses.replace(VARIANTS["actorder-zp-g64"], E=1, top_k=1)
    W = wk.make_weights(wl, 5)
    X = wk.make_batch(wl, 7, 6)
    p13, p2 = W.w13_perm[0], W.w2_perm[0]
    N = W.N
    rows13 = np.concatenate([p2, N + p2])  # gate and up rows of feature p2[n] to position n
    S = dataclasses.replace(
        W, w13=_permute_codes(W.w13, W.w13_perm)[:, rows13], w13_s=W.w13_s[:, rows13], w13_z=W.w13_z[:, rows13],
        b13=W.b13[:, rows13], w13_gidx=None, w2=_permute_codes(W.w2, W.w2_perm), w2_gidx=None)
    Xs = wk.BatchInputs(np.ascontiguousarray(X.x[:, p13]), X.topk_ids, X.topk_weights, None)
    _, a = orc.forward_workload(wl, W, X, return_acc=True)
    _, b = orc.forward_workload(wl, S, Xs, return_acc=True)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("group", [32, 64, 128, -1])
def test_closed_form_zero_points(orc, group):
    """Unit scales, every code c and every integer zero z: each weight is c - z, so
    with x in {-1/8, 0, 1/8}, h = (c1 - z1) S_t and y = (c2 - z2) N a."""
    K, N, E, M = 256, 128, 2, 5
    c1, z1, c2, z2 = 13, 9, 2, 5
    ng13, ng2 = (1, 1) if group < 0 else (K // group, N // group)
    W = wk.LayerWeights("int4", E, K, N, group, False,
                        np.full((E, 2 * N, K // 2), c1 | (c1 << 4), np.uint8), np.full((E, 2 * N, ng13), 0x3F80, np.uint16),
                        None, None,
                        np.full((E, K, N // 2), c2 | (c2 << 4), np.uint8), np.full((E, K, ng2), 0x3F80, np.uint16),
                        None, None, zero_kind="int",
                        w13_z=np.full((E, 2 * N, ng13), z1, np.uint8), w2_z=np.full((E, K, ng2), z2, np.uint8))
    rng = np.random.default_rng(9)
    xv = rng.integers(-1, 2, size=(M, K)) / 8.0
    X = wk.BatchInputs(wk.to_bf16_bits(xv.astype(np.float32)), np.array([[0, 1]] * M, np.int32),
                       np.full((M, 2), 0.5, np.float32), None)
    _, acc = orc.forward(W, X, return_acc=True)
    for t in range(M):
        h = (c1 - z1) * xv[t].sum()
        a = h / (1 + math.exp(-h)) * h
        np.testing.assert_allclose(acc[t], (c2 - z2) * N * a, rtol=1e-12, atol=1e-300)


def test_channelwise_equals_whole_row_group(orc):
    wl, W, X = case("channelwise")
    # group -1 on both matrices is group K for w13 and group N for w2: equal when K == N
    wl2 = dataclasses.replace(wl, K=128, N=128)
    W2 = wk.make_weights(wl2, 8)
    X2 = wk.make_batch(wl2, 6, 9)
    G = dataclasses.replace(W2, group=128)
    np.testing.assert_array_equal(orc.forward_workload(wl2, W2, X2), orc.forward_workload(wl2, G, X2))
