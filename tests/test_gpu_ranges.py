"""Operand-range edges of the 16-bit tensor-core path, and device-side checks
of the alignment inputs.

The kernels feed dequantised weights to fp16 tensor-core operands.  Each expert
matrix's scales are shifted at repack by a power of two into the window where
those operands are exact, and the expert's fp32 epilogue factor undoes the
shift; so every scale whose expert matrix spreads less than the window decodes
exactly.  These cases put whole banks at the ends of the formats' ranges
(E8M0 bytes 107..112 and 132..136, INT4 scales near 1e-6, 1e-4 and 4e3, E4M3
subnormals) and check every output against the oracle, on both GEMM paths
(block_m 8: register-fed, block_m 64: tcgen05).  The inputs are scaled so the
outputs are of order one (and x stays inside fp16's normal range, where its
conversion keeps every bf16 bit), and the bound is the one scaled to the output's RMS
as well as the pages' (|d| <= 0.06 + 0.04 |ref|, the assert_close of
test_fused_marlin_moe_large_non_ep_schedule, "Marlin MoE kernel occupancy ...",
sglang PR #31552).  Spreads wider than the window, inputs beyond the fp16 range
and inconsistent alignments must complete and be reported through
moe_get_status.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import bf16_to_f32, check_close_scaled, need_gpu, run_layer

pytestmark = pytest.mark.gpu

PATHS = (8, 64)  # register-fed kernel, tcgen05 kernel


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    oracle.build()


def _rng(seed):
    return np.random.default_rng(seed)


def mx_case(w13_bytes, x_scale, seed, w2_bytes=(119, 123), top_k=4):
    """MXFP4 bank (K=1024, N=256, 4 experts, interleaved, sigmoid-alpha) whose w13
    E8M0 bytes are uniform over w13_bytes (inclusive) and w2's over w2_bytes."""
    wl = dataclasses.replace(wk.WORKLOADS["mxfp4-alpha"], K=1024, N=256, E=4, top_k=top_k, Ms=(24,),
                             bias_std=0.0, x_scale=x_scale)
    W = wk.make_weights(wl, seed)
    r = _rng(seed)
    W.w13_s = r.integers(w13_bytes[0], w13_bytes[1] + 1, size=W.w13_s.shape).astype(np.uint8)
    W.w2_s = r.integers(w2_bytes[0], w2_bytes[1] + 1, size=W.w2_s.shape).astype(np.uint8)
    return wl, W, wk.make_batch(wl, 24, seed + 1)


def int4_case(lo, hi, x_scale, seed, w2_range=None):
    """INT4 bank (K=1024, N=256, 4 experts) whose w13 scales (and w2's, if given)
    are log-uniform in [lo, hi]."""
    wl = dataclasses.replace(wk.WORKLOADS["int4-skew"], K=1024, N=256, E=4, Ms=(24,), x_scale=x_scale,
                             routing="uniform")
    W = wk.make_weights(wl, seed)
    r = _rng(seed)
    W.w13_s = wk.to_bf16_bits(np.exp(r.uniform(np.log(lo), np.log(hi), size=W.w13_s.shape)).astype(np.float32))
    if w2_range:
        W.w2_s = wk.to_bf16_bits(np.exp(r.uniform(np.log(w2_range[0]), np.log(w2_range[1]),
                                                  size=W.w2_s.shape)).astype(np.float32))
    return wl, W, wk.make_batch(wl, 24, seed + 1)


def nv_subnormal_case(seed):
    """NVFP4 bank whose w13 E4M3 scales are all subnormal (bytes 1..7: m/8 * 2^-6)."""
    wl = dataclasses.replace(wk.WORKLOADS["nvfp4-ep-norm"], K=1024, N=256, E=4, E_global=4, Ms=(24,),
                             x_scale=4.0, post_norm=False)
    W = wk.make_weights(wl, seed)
    r = _rng(seed)
    W.w13_s = r.integers(1, 8, size=W.w13_s.shape).astype(np.uint8)
    W.w13_gs = r.uniform(0.5, 1.0, size=W.E).astype(np.float32)
    return wl, W, wk.make_batch(wl, 24, seed + 1)


CASES = {
    # E8M0 bytes at and below the old window's floor (2^-20 .. 2^-15): shifted up by 5
    "mxfp4-bytes-107-112": lambda: mx_case((107, 112), 4000.0, 11),
    # the top of the range stated for GPT-OSS-like scales (2^5 .. 2^9): no shift
    "mxfp4-bytes-132-136": lambda: mx_case((132, 136), 1e-4, 12),
    # one matrix spanning 36 binades (bytes 100..136): exactly the window's width
    "mxfp4-bytes-100-136": lambda: mx_case((100, 136), 2e-4, 13),
    # INT4 scales where s / 16 leaves the fp16 grid (e = -14, -20) and near the top (2^11)
    "int4-scales-1e-4": lambda: int4_case(1e-4, 2e-4, 80.0, 14),
    "int4-scales-1e-6": lambda: int4_case(1e-6, 2e-6, 8000.0, 15),
    # (x stays well inside fp16's normal range; w2's scales near 1e-4 bring the outputs to order one)
    "int4-scales-4e3": lambda: int4_case(1e3, 4e3, 2e-4, 16, w2_range=(5e-5, 1e-4)),
    "nvfp4-subnormal-e4m3": lambda: nv_subnormal_case(17),
}


def _ref(wl, W, X):
    return bf16_to_f32(oracle.forward_workload(wl, W, X))


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("block_m", PATHS)
def test_scale_range_edges(name, block_m):
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl, W, X = CASES[name]()
    ref = _ref(wl, W, X)
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    assert 0.05 < rms < 50.0, f"{name}: case not scaled to order-one outputs (rms {rms})"
    layer = MoELayer.from_numpy(W)
    out = run_layer(layer, wl, X, block_m=block_m)
    check_close_scaled(out.float().cpu().numpy(), ref, f"{name} block_m={block_m}")
    assert layer.status() == B.MOE_OK


@pytest.mark.parametrize("block_m", PATHS)
def test_mxfp4_spread_wider_than_window_is_reported(block_m):
    # bytes 100..140 span 41 values: the largest stay exact, the blob is marked
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl, W, X = mx_case((100, 140), 2e-5, 21)
    layer = MoELayer.from_numpy(W)
    assert layer.packed[:4].cpu().numpy().view(np.uint32)[0] != 0
    out = run_layer(layer, wl, X, block_m=block_m)
    assert layer.status() == B.MOE_ERR_UNSUPPORTED
    check_close_scaled(out.float().cpu().numpy(), _ref(wl, W, X), "wide MXFP4 spread")


def test_int4_spread_wider_than_window():
    # INT4 scales over 2^-20 .. 2^12: the tcgen05 path (fp16 scales) reports it, the
    # register-fed path applies scales in fp32 and is exact
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl, W, X = int4_case(2.0 ** -20, 2.0 ** 12, 1e-4, 22)
    layer = MoELayer.from_numpy(W)
    ref = _ref(wl, W, X)
    out = run_layer(layer, wl, X, block_m=8)
    assert layer.status() == B.MOE_OK
    check_close_scaled(out.float().cpu().numpy(), ref, "wide INT4 spread, register-fed")
    out = run_layer(layer, wl, X, block_m=64)
    assert layer.status() == B.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("block_m", PATHS)
def test_input_beyond_fp16_is_reported(block_m):
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl = dataclasses.replace(wk.WORKLOADS["int4-bias"], K=256, N=128, Ms=(9,))
    W = wk.make_weights(wl, 23)
    X = wk.make_batch(wl, 9, 24)
    layer = MoELayer.from_numpy(W)
    run_layer(layer, wl, X, block_m=block_m)
    assert layer.status() == B.MOE_OK
    X.x[3, 17] = wk.to_bf16_bits(np.array([1.0e5], dtype=np.float32))[0]  # above fp16's 65504
    run_layer(layer, wl, X, block_m=block_m)
    assert layer.status() == B.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("block_m", PATHS)
def test_nan_scale_propagates_and_is_reported(block_m):
    # E8M0 byte 255 is NaN: the tokens routed to that expert come out NaN on both sides
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl, W, X = mx_case((119, 123), 1.0, 25, top_k=2)
    W.w13_s[2, 5, 3] = 255
    ref = _ref(wl, W, X)
    layer = MoELayer.from_numpy(W)
    out = run_layer(layer, wl, X, block_m=block_m).float().cpu().numpy()
    assert layer.status() == B.MOE_ERR_UNSUPPORTED
    np.testing.assert_array_equal(np.isnan(out), np.isnan(ref))
    assert np.isnan(ref).any() and not np.isnan(ref).all()


# ------------------------------------------------------------------ alignment inputs

def _forward_with(layer, wl, X, sorted_ids, expert_ids, n_padded, block_m):
    from weight_only_bit_moe_gb300.layer import AlignOut, batch_to_device
    x, ids, w, _ = batch_to_device(X)
    a = AlignOut(block_m, sorted_ids, expert_ids, n_padded)
    out = layer.forward(x, ids, w, a, act=wl.act)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("block_m", PATHS)
def test_inconsistent_alignment_is_reported(block_m):
    """n_padded beyond the capacity, an expert id outside [0, E) and a sorted id
    that is neither a pair nor the sentinel: all buffers are sized for the
    call's capacity, so every access stays inside them; the forward completes
    and moe_get_status reports MOE_ERR_INVALID; a correct alignment afterwards
    runs clean."""
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer, batch_to_device
    wl = dataclasses.replace(wk.WORKLOADS["int4-bias"], K=256, N=128, Ms=(20,))
    W = wk.make_weights(wl, 26)
    X = wk.make_batch(wl, 20, 27)
    layer = MoELayer.from_numpy(W)
    _, ids, _, _ = batch_to_device(X)
    good = layer.align(ids, 0, block_m)
    cap = good.sorted_ids.numel()
    for bad in ("n_padded", "expert", "sorted"):
        s, e, n = good.sorted_ids.clone(), good.expert_ids.clone(), good.n_padded.clone()
        if bad == "n_padded":
            n.fill_(cap + block_m)
        elif bad == "expert":
            e[0] = 99
        else:
            s[0] = 20 * wl.top_k + 5
        _forward_with(layer, wl, X, s, e, n, block_m)
        assert layer.status() == B.MOE_ERR_INVALID, bad
    out = _forward_with(layer, wl, X, good.sorted_ids, good.expert_ids, good.n_padded, block_m)
    assert layer.status() == B.MOE_OK
    check_close_scaled(out.float().cpu().numpy(), _ref(wl, W, X), "after the bad calls")
