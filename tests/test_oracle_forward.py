"""Pins of the oracle's layer forward (no GPU).

The forward is the per-expert computation of "Marlin MoE kernel occupancy ..."
(sglang PR #31552), test_fused_marlin_moe_large_non_ep_schedule (per-expert loop,
bias added after each matmul, top-k weights applied in fp32 in the combine), with
the gated activations of "013-moe-middle-tiles.py" (silu_and_mul, first half gate)
and of "SM120 MXFP4 MoE ... Marlin" (sglang PR #28231,
swiglu_gpt_oss_sigmoid_alpha_contiguous), and the post-expert norm of
"013-moe-middle-tiles.py" (_expert_norm_factors / _expert_norm_sum).

Pins, each able to catch a different class of mistake in the oracle:
  * dense brute force: every expert evaluated on every token with numpy matmuls
    and torch's own float8 decoders, then selected by routing -- no alignment, no
    sort, no per-pair loop (catches index, transpose, nibble, scale-group,
    interleave, bias, gs and combine mistakes);
  * closed form with unit scales and constant codes;
  * token-permutation invariance;
  * expert-parallel decomposition: partial outputs of disjoint expert ranges sum
    to the single-range result;
  * interleaved storage equals pre-deinterleaved storage;
  * post-norm output has unit RMS when one pair with weight 1 is routed.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from weight_only_bit_moe_gb300 import workloads as wk

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6], dtype=np.float64)


def rne_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even) by integer rounding of the fp64
    bit pattern at the 8th significant bit; valid for |x| >= 2^-126 and 0."""
    x = np.asarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    drop = np.uint64(45)  # 52 - 7 mantissa bits
    lsb = (u >> drop) & np.uint64(1)
    r = (u + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    out = r.view(np.float64)
    assert np.all((np.abs(x) >= 2.0 ** -126) | (x == 0))
    return out


def bf16v(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_matrix(fmt, codes, scales, group):
    """[E, R, C/2] codes + [E, R, C/g] scales -> fp64 [E, R, C] via torch decoders."""
    q = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.int64)
    q[..., 0::2] = codes & 15
    q[..., 1::2] = codes >> 4
    if fmt == "int4":
        val = (q - 8).astype(np.float64)
        sv = bf16v(scales)
    else:
        val = E2M1[q]
        if fmt == "mxfp4":
            sv = np.ldexp(1.0, scales.astype(np.int64) - 127)
        else:
            sv = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return val * np.repeat(sv, group, axis=-1)


def dense_reference(wl, W, X, rsf=1.0):
    """Every expert on every token, then select; fp64 throughout, the caller
    rounds the output to bf16."""
    E, K, N = W.E, W.K, W.N
    R = 2 * N if W.gated else N
    W13 = decode_matrix(W.fmt, W.w13, W.w13_s, W.group)  # [E, R, K]
    b13 = bf16v(W.b13) if W.b13 is not None else np.zeros((E, R))
    if W.interleaved:  # stored rows g0,u0,g1,u1,... -> gate block then up block
        W13 = np.concatenate([W13[:, 0::2], W13[:, 1::2]], axis=1)
        b13 = np.concatenate([b13[:, 0::2], b13[:, 1::2]], axis=1)
    W2 = decode_matrix(W.fmt, W.w2, W.w2_s, W.group)     # [E, K, N]
    b2 = bf16v(W.b2) if W.b2 is not None else np.zeros((E, K))
    gs13 = W.w13_gs.astype(np.float64) if W.w13_gs is not None else np.ones(E)
    gs2 = W.w2_gs.astype(np.float64) if W.w2_gs is not None else np.ones(E)
    x = bf16v(X.x)                                        # [M, K]
    M = x.shape[0]
    Y = np.empty((E, M, K))
    for e in range(E):
        h = gs13[e] * (x @ W13[e].T) + b13[e]
        g, u = h[:, :N], h[:, N:]
        if not W.gated:
            a = np.square(np.maximum(h, 0.0))
        elif wl.act == "silu_mul":
            a = g / (1 + np.exp(-g)) * u
        else:
            gc = np.minimum(g, wl.limit)
            uc = np.clip(u, -wl.limit, wl.limit)
            a = gc / (1 + np.exp(-wl.alpha * gc)) * (uc + 1)
        Y[e] = gs2[e] * (a @ W2[e].T) + b2[e]
    out = np.zeros((M, K))
    if wl.post_norm:
        nw = rne_bf16(np.float32(1.0) + bf16v(X.post_norm_w).astype(np.float32))
    for t in range(M):
        for j in range(X.topk_ids.shape[1]):
            e = int(X.topk_ids[t, j]) - wl.expert_base
            if not 0 <= e < E:
                continue
            w = float(X.topk_weights[t, j])
            if wl.post_norm:
                z = Y[e, t] * nw
                inv = 1.0 / math.sqrt(np.sum(z * z) / K + wl.norm_eps)
                out[t] += w * inv * z
            else:
                out[t] += w * Y[e, t]
    return out * rsf


SMALL = {
    "int4-tiny": wk.WORKLOADS["tiny-int4"],
    "int4-bias-small": dataclasses.replace(wk.WORKLOADS["int4-bias"], K=256, N=128, Ms=(9,)),
    "mxfp4-alpha-small": dataclasses.replace(wk.WORKLOADS["mxfp4-alpha"], K=96, N=64, E=4, Ms=(7,)),
    "mxfp4-alpha-clamp": dataclasses.replace(wk.WORKLOADS["mxfp4-alpha"], K=96, N=64, E=4, Ms=(7,), limit=7.0),
    "nvfp4-ep-small": dataclasses.replace(wk.WORKLOADS["nvfp4-ep-norm"], K=64, N=48, E=4, E_global=16,
                                          expert_base=4, Ms=(12,)),
    "int4-zipf-small": dataclasses.replace(wk.WORKLOADS["int4-skew"], K=256, N=128, E=16, Ms=(10,)),
    "int4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], K=256, N=256, E=4, Ms=(11,)),
    "nvfp4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], fmt="nvfp4", K=64, N=48, E=4,
                                             Ms=(9,)),
    "mxfp4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], fmt="mxfp4", K=96, N=64, E=4,
                                             Ms=(7,)),
}


def make_small(name, seed=7):
    wl = SMALL[name]
    return wl, wk.make_weights(wl, seed), wk.make_batch(wl, wl.Ms[0], seed + 1)


@pytest.mark.parametrize("name", list(SMALL))
def test_dense_bruteforce(orc, name):
    wl, W, X = make_small(name)
    got_bits, got_acc = orc.forward_workload(wl, W, X, return_acc=True)
    ref = dense_reference(wl, W, X)
    # same arithmetic, different loop structure: the pre-rounding values agree to
    # fp64 noise, and the bf16 outputs bit for bit except where that noise
    # straddles a rounding boundary
    np.testing.assert_allclose(got_acc, ref, rtol=1e-11, atol=1e-11)
    same = bf16v(got_bits) == rne_bf16(ref)
    assert same.mean() > 0.9999, same.mean()
    assert np.abs(ref).max() > 0.0


@pytest.mark.parametrize("fmt", ["int4", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("act", ["silu_mul", "sigmoid_alpha", "relu2"])
def test_closed_form_unit_scales(orc, fmt, act):
    """Unit scales, zero bias, every w13 code c1, every w2 code c2 and x in
    {-1/8, 0, 1/8}: h = v1*S_t on every row, a = act(h, h) (relu(h)^2 for the
    non-gated experts), y = v2*N*a, out_t = bf16(rsf * sum_j w_tj * y_t)."""
    K, N, E, k, M = 128, 128, 3, 2, 6
    group = {"int4": 128, "mxfp4": 32, "nvfp4": 16}[fmt]
    gated = act != "relu2"
    R = 2 * N if gated else N
    c1, c2 = (11, 6) if fmt == "int4" else (3, 10)    # int4: 3 and -2; e2m1: 1.5 and -1.0
    v1 = c1 - 8.0 if fmt == "int4" else E2M1[c1]
    v2 = c2 - 8.0 if fmt == "int4" else E2M1[c2]
    unit = {"int4": np.uint16(0x3F80), "mxfp4": np.uint8(127), "nvfp4": np.uint8(0x38)}[fmt]
    W = wk.LayerWeights(fmt, E, K, N, group, False,
                        np.full((E, R, K // 2), c1 | (c1 << 4), np.uint8),
                        np.full((E, R, K // group), unit), np.ones(E, np.float32) if fmt == "nvfp4" else None,
                        None,
                        np.full((E, K, N // 2), c2 | (c2 << 4), np.uint8),
                        np.full((E, K, N // group), unit), np.ones(E, np.float32) if fmt == "nvfp4" else None,
                        None, gated=gated)
    rng = np.random.default_rng(3)
    xv = rng.integers(-1, 2, size=(M, K)) / 8.0
    x = torch.from_numpy(xv.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2], [2, 1], [1, 0]], dtype=np.int32)
    w = rng.uniform(0.1, 0.9, size=(M, k)).astype(np.float32)
    X = wk.BatchInputs(x, ids, w, None)
    rsf = 1.5
    got_bits, got_acc = orc.forward(W, X, act=act, rsf=rsf, return_acc=True)
    got = bf16v(got_bits)
    for t in range(M):
        S = xv[t].sum()
        h = v1 * S
        if act == "relu2":
            a = max(h, 0.0) ** 2
        elif act == "silu_mul":
            a = h / (1 + math.exp(-h)) * h
        else:
            a = h / (1 + math.exp(-1.702 * h)) * (h + 1)
        y = v2 * N * a
        expect = rsf * float(w[t].astype(np.float64).sum()) * y
        # fp64 evaluation order differs from the oracle's sums only in the last bits
        np.testing.assert_allclose(got_acc[t], expect, rtol=1e-12, atol=1e-300)
        assert np.all(got[t] == float(rne_bf16(np.array(expect)))), (t, got[t][:4], expect)


def test_relu2_rejects_gated_mismatch(orc):
    """The non-gated layout goes only with relu2, and relu2 only with it."""
    wl, W, X = make_small("int4-relu2-small")
    with pytest.raises(ValueError):
        orc.forward(W, X, act="silu_mul")
    wg, Wg, Xg = make_small("int4-bias-small")
    with pytest.raises(ValueError):
        orc.forward(Wg, Xg, act="relu2")


def test_relu2_negative_rows_give_zero(orc):
    """relu2 clips: with every w13 row negated the intermediates of rows whose
    h was positive become zero, so the two outputs are y(+W) and y(-W), whose
    activations a+ and a- have disjoint supports and satisfy a+ + a- = h^2."""
    wl, W, X = make_small("int4-relu2-small")
    # negate each int4 code: q -> 16 - q maps (q - 8) to -(q - 8); code 0 (-8) has no
    # negation, so it is first replaced by 8 (zero) in both layers
    q_lo, q_hi = W.w13 & 15, W.w13 >> 4
    ok = (q_lo != 0) & (q_hi != 0)
    lo = np.where(q_lo == 0, 8, q_lo)
    hi = np.where(q_hi == 0, 8, q_hi)
    Wp = dataclasses.replace(W, w13=(lo | (hi << 4)).astype(np.uint8), b13=None)
    Wn = dataclasses.replace(W, w13=(((16 - lo) & 15) | (((16 - hi) & 15) << 4)).astype(np.uint8), b13=None)
    assert ok.mean() > 0.8
    for e, t in [(0, 0), (1, 3), (3, 7)]:
        hp, ap, _ = orc.ffn_pair(Wp, X, e, t, act="relu2")
        hn, an, _ = orc.ffn_pair(Wn, X, e, t, act="relu2")
        np.testing.assert_allclose(hn, -hp, rtol=0, atol=1e-12)
        assert np.all((ap == 0) | (an == 0))
        np.testing.assert_allclose(ap + an, hp * hp, rtol=1e-12, atol=1e-300)
        assert (ap > 0).any() and (an > 0).any()


@pytest.mark.parametrize("name", ["int4-bias-small", "nvfp4-ep-small", "mxfp4-alpha-small"])
def test_token_permutation(orc, name):
    wl, W, X = make_small(name)
    perm = np.random.default_rng(5).permutation(X.x.shape[0])
    Xp = wk.BatchInputs(X.x[perm], X.topk_ids[perm], X.topk_weights[perm], X.post_norm_w)
    a = orc.forward_workload(wl, W, X)
    b = orc.forward_workload(wl, W, Xp)
    np.testing.assert_array_equal(a[perm], b)


def test_expert_parallel_decomposition(orc):
    """Four ranks owning experts [4r, 4r+4) of 16: their pre-rounding partial
    outputs sum to the output of one rank owning all 16."""
    full = dataclasses.replace(SMALL["nvfp4-ep-small"], E=16, expert_base=0)
    W = wk.make_weights(full, 11)
    X = wk.make_batch(full, 12, 13)
    _, ref = orc.forward_workload(full, W, X, return_acc=True)
    total = np.zeros_like(ref)
    for r in range(4):
        sl = slice(4 * r, 4 * r + 4)
        Wr = dataclasses.replace(W, E=4, w13=W.w13[sl], w13_s=W.w13_s[sl], w13_gs=W.w13_gs[sl],
                                 w2=W.w2[sl], w2_s=W.w2_s[sl], w2_gs=W.w2_gs[sl])
        wr = dataclasses.replace(full, E=4, expert_base=4 * r)
        _, part = orc.forward_workload(wr, Wr, X, return_acc=True)
        total += part
    np.testing.assert_allclose(total, ref, rtol=1e-12, atol=1e-12)


def test_interleaved_equals_deinterleaved(orc):
    wl, W, X = make_small("mxfp4-alpha-small")
    D = dataclasses.replace(W, interleaved=False,
                            w13=np.concatenate([W.w13[:, 0::2], W.w13[:, 1::2]], axis=1),
                            w13_s=np.concatenate([W.w13_s[:, 0::2], W.w13_s[:, 1::2]], axis=1),
                            b13=np.concatenate([W.b13[:, 0::2], W.b13[:, 1::2]], axis=1))
    np.testing.assert_array_equal(orc.forward_workload(wl, W, X), orc.forward_workload(wl, D, X))


def test_post_norm_unit_rms(orc):
    """One local pair per token with weight 1: out = z / rms(z), so rms(out) ~ 1."""
    wl = dataclasses.replace(SMALL["nvfp4-ep-small"], top_k=1)
    W = wk.make_weights(wl, 21)
    X = wk.make_batch(wl, 8, 22)
    X = wk.BatchInputs(X.x, np.full((8, 1), 5, np.int32), np.ones((8, 1), np.float32), X.post_norm_w)
    out = bf16v(orc.forward_workload(wl, W, X))
    rms = np.sqrt((out ** 2).mean(axis=1))
    np.testing.assert_allclose(rms, 1.0, atol=4e-3)


def test_non_local_pairs_contribute_nothing(orc):
    wl, W, X = make_small("nvfp4-ep-small")
    ids = X.topk_ids.copy()
    ids[:, :] = 0  # every id below expert_base=4: nothing is local
    out = orc.forward_workload(wl, W, wk.BatchInputs(X.x, ids, X.topk_weights, X.post_norm_w))
    assert np.all(bf16v(out) == 0)
