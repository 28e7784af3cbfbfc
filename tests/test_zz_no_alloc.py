"""The allocation-free forward (moe_w4a16_forward_noalloc) against the
caller-workspace forward, through the C ABI.

The two entry points run the same kernels; the fixed-scratch one may choose
fewer split-K slices, so outputs agree within the layer's tolerance rather than
bit for bit.  Each case calls the allocation-free entry point twice in a row on
the same inputs (the second call reuses the scratch the first one left behind)
and compares both results.  This file sorts last so that it also runs after
every other GPU test in one process.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import GPU_SMALL, bf16_to_f32, check_close, check_workload, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _run_both(wl, W, X, block_m=None):
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import ACT, MoELayer, batch_to_device
    layer = MoELayer.from_numpy(W)
    x, ids, w, pnw = batch_to_device(X)
    pnw = pnw if wl.post_norm else None
    M, k = ids.shape
    a = layer.align(ids, wl.expert_base, block_m, wl.n_ids)
    ref = layer.forward(x, ids, w, a, expert_base=wl.expert_base, act=wl.act, alpha=wl.alpha, limit=wl.limit,
                        post_norm_w=pnw, norm_eps=wl.norm_eps)
    outs = []
    for _ in range(2):
        out = torch.full((M, wl.K), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.moe_w4a16_forward_noalloc(layer.desc, layer.packed, x, M, k, ids, w, wl.expert_base, a.sorted_ids,
                                    a.expert_ids, a.n_padded, a.block_m, ACT[wl.act], wl.alpha, wl.limit, 1.0,
                                    pnw, wl.norm_eps, out)
        outs.append(out)
    torch.cuda.synchronize()
    # (the status read here is the workspace forward's: the allocation-free calls
    # record theirs in the fixed array, which this entry point does not report)
    assert layer.status() == 0
    return ref.float().cpu().numpy(), [o.float().cpu().numpy() for o in outs]


CASES = [("int4-bias", 2304), ("mxfp4-alpha", 1), ("mxfp4-alpha", 32), ("nvfp4-ep-norm", 8),
         ("int4-skew", 16), ("int4-relu2", 2304)]


@pytest.mark.parametrize("name,M", CASES)
def test_noalloc_matches_workspace_forward(name, M):
    wl = wk.WORKLOADS[name]
    W = wk.make_weights(wl, wk.weight_seed(name))
    X = wk.make_batch(wl, M, wk.batch_seed(name, M))
    ref, outs = _run_both(wl, W, X)
    for i, o in enumerate(outs):
        check_workload(o, ref, wl, f"{name} M={M} noalloc call {i}")
    torch.cuda.empty_cache()


def test_noalloc_small_against_oracle():
    oracle.build()
    wl = GPU_SMALL["nvfp4-ep-small"]
    W = wk.make_weights(wl, 91)
    X = wk.make_batch(wl, 21, 92)
    ref, outs = _run_both(wl, W, X, block_m=16)
    want = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_close(ref, want, "workspace forward")
    for i, o in enumerate(outs):
        check_close(o, want, f"noalloc call {i}")


def test_noalloc_rejects_oversize_shape():
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import ACT, MoELayer, batch_to_device
    # 32768 tokens x top-2 x hidden 512: the fp16 expert outputs alone take 64 MiB, the gathered
    # rows and the activations 190 MiB more
    wl = dataclasses.replace(wk.WORKLOADS["int4-bias"], Ms=(32768,))
    W = wk.make_weights(wl, 7)
    X = wk.make_batch(wl, 32768, 8)
    layer = MoELayer.from_numpy(W)
    x, ids, w, _ = batch_to_device(X)
    a = layer.align(ids, 0, None, wl.n_ids)
    out = torch.zeros((32768, wl.K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoeError) as exc:
        B.moe_w4a16_forward_noalloc(layer.desc, layer.packed, x, 32768, wl.top_k, ids, w, 0, a.sorted_ids,
                                    a.expert_ids, a.n_padded, a.block_m, ACT[wl.act], wl.alpha, wl.limit, 1.0,
                                    None, wl.norm_eps, out)
    assert exc.value.status == B.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing was launched
