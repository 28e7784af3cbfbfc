"""Shared helpers for the GPU parity tests: build/load the library, run the
layer through the C ABI, and compare with the oracle under the pages' bound."""
import dataclasses

import numpy as np
import pytest
import torch

from weight_only_bit_moe_gb300 import workloads as wk

# |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise on bf16 outputs: the
# assert_close(rtol=0.04, atol=0.06) of test_fused_marlin_moe_large_non_ep_schedule
# in "Marlin MoE kernel occupancy ..." (sglang PR #31552).
ATOL, RTOL = 0.06, 0.04


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from weight_only_bit_moe_gb300 import build, binding
    build.build()
    binding.load()


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def tensor_bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def check_close(got: np.ndarray, ref: np.ndarray, what: str = "", atol: float = ATOL, rtol: float = RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    assert np.all(np.isfinite(ref)), f"{what}: non-finite oracle output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    ratio = float((err / bound).max()) if err.size else 0.0
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} of {err.size} outside |d| <= {atol:.3g} + {rtol}|ref|; "
                           f"max err/bound {ratio:.3f}; first {bad[:5].tolist()} "
                           f"got {got[tuple(bad[0])]:.5f} ref {ref[tuple(bad[0])]:.5f}")
    return ratio


# A bound scaled to the output's own size, for workloads whose outputs are far
# below 1 (the relu2 test writes x = randn/10, bias = randn/100, so |out| ~ 0.1
# and the absolute 0.06 above would pass almost anything): |d| <= 0.02 rms(ref)
# + 0.01 |ref|.  The arithmetic's own error is the bf16 output rounding (2^-9
# relative, inside the 0.01) plus the 16-bit operand roundings, a few 2^-11 of
# the typical output.
SCALED_ATOL, SCALED_RTOL = 0.02, 0.01


def check_close_scaled(got: np.ndarray, ref: np.ndarray, what: str = ""):
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    assert rms > 0.0, f"{what}: all-zero oracle output"
    check_close(got, ref, what)  # the pages' own bound as well
    return check_close(got, ref, what, atol=SCALED_ATOL * rms, rtol=SCALED_RTOL)


def run_layer(layer, wl, X, block_m=None, **kw):
    from weight_only_bit_moe_gb300.layer import batch_to_device
    x, ids, w, pnw = batch_to_device(X)
    out = layer(x, ids, w, expert_base=wl.expert_base, block_m=block_m, num_routed_ids=wl.n_ids,
                act=wl.act, alpha=wl.alpha, limit=wl.limit, post_norm_w=pnw if wl.post_norm else None,
                norm_eps=wl.norm_eps, **kw)
    torch.cuda.synchronize()
    return out


def sample_tokens(M: int, n: int, seed: int = 0) -> np.ndarray:
    if M <= n:
        return np.arange(M, dtype=np.int32)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid])).astype(np.int32)


# Small variants of the workloads with shapes the kernels accept (hidden % 64,
# int4 hidden % 128) that still span several tiles and a ragged tail: N below
# the 128-row tile, hidden below the 256-row GEMM2 tile.
GPU_SMALL = {
    "tiny-int4": wk.WORKLOADS["tiny-int4"],
    "int4-bias-small": dataclasses.replace(wk.WORKLOADS["int4-bias"], K=256, N=384, Ms=(37,)),
    "mxfp4-alpha-small": dataclasses.replace(wk.WORKLOADS["mxfp4-alpha"], K=192, N=160, E=4, Ms=(29,)),
    "mxfp4-alpha-clamp": dataclasses.replace(wk.WORKLOADS["mxfp4-alpha"], K=192, N=96, E=4, Ms=(13,), limit=7.0),
    "nvfp4-ep-small": dataclasses.replace(wk.WORKLOADS["nvfp4-ep-norm"], K=320, N=48, E=4, E_global=16,
                                          expert_base=4, Ms=(21,)),
    "int4-zipf-small": dataclasses.replace(wk.WORKLOADS["int4-skew"], K=384, N=256, E=16, Ms=(50,)),
    # non-gated relu2 experts: N=384 pads to two 256-row GEMM1 tiles, the second ragged
    "int4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], K=256, N=384, E=4, Ms=(37,)),
    "mxfp4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], fmt="mxfp4", K=192, N=160, E=4,
                                             Ms=(29,)),
    "nvfp4-relu2-small": dataclasses.replace(wk.WORKLOADS["int4-relu2"], fmt="nvfp4", K=320, N=48, E=4,
                                             Ms=(21,), bias_std=0.0),
}


def check_workload(got, ref, wl, what=""):
    """The pages' bound, and for workloads with small outputs the scaled one too."""
    if wl.x_scale < 1.0:
        return check_close_scaled(got, ref, what)
    return check_close(got, ref, what)
