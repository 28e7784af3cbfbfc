"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Alignment is compared bit for bit; layer outputs elementwise under
|gpu - oracle| <= 0.06 + 0.04 |oracle| (the bound of the PR #31552 test).  Small
shapes span several tiles and ragged tails; the full workload shapes are
checked on every token, in the launch configuration the benchmark uses.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import GPU_SMALL, bf16_to_f32, check_close, check_workload, need_gpu, run_layer, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    oracle.build()


def _layer(W):
    from weight_only_bit_moe_gb300.layer import MoELayer
    return MoELayer.from_numpy(W)


# ------------------------------------------------------------------ align

ALIGN_CASES = [
    # (M, top_k, E, block_m, expert_base, routed ids, routing)
    (1, 2, 8, 16, 0, 8, "uniform"),
    (16, 2, 8, 8, 0, 8, "uniform"),
    (123, 2, 8, 16, 0, 8, "uniform"),
    (2304, 2, 8, 128, 0, 8, "uniform"),
    (1, 8, 32, 16, 0, 256, "uniform"),
    (64, 8, 32, 32, 96, 256, "uniform"),
    (512, 8, 32, 64, 0, 256, "uniform"),
    (1000, 8, 128, 16, 0, 128, "zipf"),
    (4096, 8, 128, 128, 0, 128, "zipf"),
    (4096, 8, 128, 64, 0, 128, "uniform"),
    (3, 4, 1024, 8, 0, 1024, "uniform"),
    # up to 32 pairs: the one-warp path (decode batches), with experts shared by tokens
    (2, 8, 8, 16, 0, 8, "uniform"),
    (4, 8, 8, 8, 0, 8, "uniform"),
    (4, 8, 128, 128, 0, 128, "zipf"),
    (1, 8, 32, 8, 96, 256, "uniform"),
    (5, 6, 16, 32, 3, 24, "uniform"),
    (1, 16, 16, 64, 0, 16, "uniform"),
]


@pytest.mark.parametrize("M,k,E,B,base,nid,routing", ALIGN_CASES)
def test_align_bit_exact(M, k, E, B, base, nid, routing):
    from weight_only_bit_moe_gb300 import binding
    # (the name only selects the seed of the Zipf rank permutation)
    wl = wk.Workload("int4-skew", "int4", K=128, N=128, E=E, top_k=k, Ms=(M,), E_global=nid,
                     expert_base=base, routing=routing)
    X = wk.make_batch(wl, M, 1234 + M)
    ids = torch.from_numpy(X.topk_ids).cuda()
    cap = binding.moe_align_capacity(M, k, E, B)
    s = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    e = torch.full((max(cap // B, 1),), -7, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    binding.moe_align(ids, M, k, base, E, B, s, e, n)
    torch.cuda.synchronize()
    rs, re, rn = oracle.align(X.topk_ids, E, B, base)
    assert cap == len(rs)
    assert int(n.item()) == rn
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(e.cpu().numpy()[:cap // B], re)


def test_align_empty_batch():
    from weight_only_bit_moe_gb300 import binding
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    s = torch.empty(1, dtype=torch.int32, device="cuda")
    binding.moe_align(torch.empty((0, 2), dtype=torch.int32, device="cuda"), 0, 2, 0, 8, 16, s, s, n)
    torch.cuda.synchronize()
    assert int(n.item()) == 0


# ------------------------------------------------------------------ forward, small shapes

@pytest.mark.parametrize("name", list(GPU_SMALL))
def test_forward_small(name):
    wl = GPU_SMALL[name]
    W = wk.make_weights(wl, 31)
    X = wk.make_batch(wl, wl.Ms[0], 32)
    layer = _layer(W)
    out = run_layer(layer, wl, X)
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_workload(out.float().cpu().numpy(), ref, wl, name)
    assert layer.status() == 0


@pytest.mark.parametrize("name", ["int4-zipf-small", "int4-relu2-small", "nvfp4-ep-small", "mxfp4-alpha-small",
                                  "mxfp4-relu2-small"])
@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
def test_forward_every_block_m(name, B):
    wl = GPU_SMALL[name]
    W = wk.make_weights(wl, 41)
    X = wk.make_batch(wl, 50, 42)
    layer = _layer(W)
    out = run_layer(layer, wl, X, block_m=B)
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_workload(out.float().cpu().numpy(), ref, wl, f"{name} block_m={B}")


@pytest.mark.parametrize("name", ["int4-zipf-small", "nvfp4-ep-small", "mxfp4-alpha-small", "int4-relu2-small"])
@pytest.mark.parametrize("B", [8, 64])
@pytest.mark.parametrize("M", [1, 3, 50])
def test_forward_own_alignment_equals_moe_align(name, B, M):
    # the forward aligning the routing in its own first kernel gives bitwise the
    # same output as the forward on moe_align's result (one-warp path up to 32
    # pairs, the counting sort beyond)
    wl = GPU_SMALL[name]
    W = wk.make_weights(wl, 141)
    X = wk.make_batch(wl, M, 142 + M)
    layer = _layer(W)
    a = run_layer(layer, wl, X, block_m=B).clone()
    b = run_layer(layer, wl, X, block_m=B, separate_align=True).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    check_workload(a.float().cpu().numpy(), bf16_to_f32(oracle.forward_workload(wl, W, X)), wl, f"{name} M={M}")


def test_forward_bitwise_reproducible():
    wl = GPU_SMALL["mxfp4-alpha-small"]
    W = wk.make_weights(wl, 51)
    X = wk.make_batch(wl, 29, 52)
    layer = _layer(W)
    a = run_layer(layer, wl, X).clone()
    b = run_layer(layer, wl, X).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_token_permutation():
    wl = GPU_SMALL["nvfp4-ep-small"]
    W = wk.make_weights(wl, 61)
    X = wk.make_batch(wl, 21, 62)
    perm = np.random.default_rng(0).permutation(21)
    Xp = wk.BatchInputs(X.x[perm], X.topk_ids[perm], X.topk_weights[perm], X.post_norm_w)
    layer = _layer(W)
    a = run_layer(layer, wl, X).float().cpu().numpy()
    b = run_layer(layer, wl, Xp).float().cpu().numpy()
    check_close(b, a[perm], "permuted")


def test_forward_nothing_local():
    wl = GPU_SMALL["nvfp4-ep-small"]
    W = wk.make_weights(wl, 71)
    X = wk.make_batch(wl, 5, 72)
    X = wk.BatchInputs(X.x, np.zeros_like(X.topk_ids), X.topk_weights, X.post_norm_w)  # ids below the local range
    out = run_layer(_layer(W), wl, X)
    assert torch.count_nonzero(out.float()).item() == 0


def test_forward_single_token():
    wl = dataclasses.replace(GPU_SMALL["int4-bias-small"], Ms=(1,))
    W = wk.make_weights(wl, 81)
    X = wk.make_batch(wl, 1, 82)
    out = run_layer(_layer(W), wl, X)
    check_close(out.float().cpu().numpy(), bf16_to_f32(oracle.forward_workload(wl, W, X)), "M=1")


# ------------------------------------------------------------------ forward, full workload shapes

FULL = [("tiny-int4", 16), ("int4-bias", 123), ("int4-bias", 2304), ("mxfp4-alpha", 1), ("mxfp4-alpha", 32),
        ("mxfp4-alpha", 1024), ("nvfp4-ep-norm", 1), ("nvfp4-ep-norm", 8), ("nvfp4-ep-norm", 64),
        ("nvfp4-ep-norm", 512), ("int4-skew", 1), ("int4-skew", 16), ("int4-skew", 256), ("int4-skew", 4096),
        ("int4-uniform", 1), ("int4-uniform", 16), ("int4-uniform", 256), ("int4-uniform", 4096),
        ("int4-relu2", 123), ("int4-relu2", 2304)]

_weights_cache = {}


def _full_layer(name):
    if name not in _weights_cache:
        _weights_cache.clear()
        torch.cuda.empty_cache()
        wl, W = wk.WORKLOADS[name], wk.make_weights(wk.WORKLOADS[name], wk.weight_seed(name))
        _weights_cache[name] = (wl, W, _layer(W))
    return _weights_cache[name]


@pytest.mark.parametrize("name,M", FULL)
def test_forward_full_every_token(name, M):
    # every output of every token against the oracle, at the workload's own size
    # and with the block size the benchmark chooses (the largest shapes take the
    # oracle a minute or two on the host cores)
    wl, W, layer = _full_layer(name)
    X = wk.make_batch(wl, M, wk.batch_seed(name, M))
    out = run_layer(layer, wl, X).clone()
    assert layer.status() == 0
    # bitwise reproducible: split-K and stream-K partials are summed in a fixed order
    again = run_layer(layer, wl, X)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16)), f"{name} M={M} not reproducible"
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_workload(out.float().cpu().numpy(), ref, wl, f"{name} M={M}")


# ------------------------------------------------------------------ edge cases

def test_forward_routed_scaling_factor():
    wl = GPU_SMALL["int4-bias-small"]
    W = wk.make_weights(wl, 91)
    X = wk.make_batch(wl, 19, 92)
    out = run_layer(_layer(W), wl, X, routed_scaling_factor=2.5)
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X, rsf=2.5))
    check_close(out.float().cpu().numpy(), ref, "rsf=2.5")


def test_forward_top_k_16():
    # the combine's largest slot count; 16 distinct experts per token
    wl = dataclasses.replace(GPU_SMALL["int4-zipf-small"], E=32, top_k=16, routing="uniform")
    W = wk.make_weights(wl, 101)
    X = wk.make_batch(wl, 23, 102)
    out = run_layer(_layer(W), wl, X)
    check_close(out.float().cpu().numpy(), bf16_to_f32(oracle.forward_workload(wl, W, X)), "top_k=16")


@pytest.mark.parametrize("B", [8, 64, 128])
def test_forward_all_tokens_on_two_experts(B):
    # one extreme of routing skew: every token picks experts 3 and 5, so two
    # experts own many blocks and the rest none
    wl = GPU_SMALL["int4-zipf-small"]
    W = wk.make_weights(wl, 111)
    X = wk.make_batch(wl, 300, 112)
    ids = np.tile(np.array([[3, 5]], dtype=np.int32), (300, 1))[:, : wl.top_k]
    if wl.top_k > 2:
        ids = np.concatenate([ids, np.tile(np.arange(6, 6 + wl.top_k - 2, dtype=np.int32), (300, 1))], axis=1)
    X = wk.BatchInputs(X.x, ids, X.topk_weights, X.post_norm_w)
    out = run_layer(_layer(W), wl, X, block_m=B)
    toks = sample_tokens(300, 24, seed=B)
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X, tokens=toks))
    check_close(out.float().cpu().numpy()[toks], ref, f"two hot experts, block_m={B}")


@pytest.mark.parametrize("fmt,K,N", [("nvfp4", 64, 16), ("mxfp4", 64, 32), ("int4", 128, 128)])
def test_forward_smallest_shapes(fmt, K, N):
    # one K-stage, the smallest intermediate each format accepts, a ragged tile
    wl = wk.Workload(f"{fmt}-min", fmt, K=K, N=N, E=3, top_k=2, Ms=(7,))
    W = wk.make_weights(wl, 121)
    X = wk.make_batch(wl, 7, 122)
    for B in (8, 64):
        out = run_layer(_layer(W), wl, X, block_m=B)
        check_close(out.float().cpu().numpy(), bf16_to_f32(oracle.forward_workload(wl, W, X)), f"{fmt} K={K} N={N} B={B}")


def test_non_gated_workspace_is_smaller():
    # relu2 banks keep N partial columns for the tcgen05 GEMM1's split-K instead
    # of 2N; the register-fed kernels' partial tiles ([256 rows][block_m] per
    # CTA) do not depend on the gating, only its counters do (the plan reads the SM
    # count, hence a GPU test)
    from weight_only_bit_moe_gb300 import binding as B
    D = B.moe_layer_desc
    for M in (1, 123, 2304):
        g = B.moe_workspace_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 0), M, 2, 64)
        ng = B.moe_workspace_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 1), M, 2, 64)
        assert 0 < ng < g, (M, g, ng)
        g16 = B.moe_workspace_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 0), M, 2, 16)
        ng16 = B.moe_workspace_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 1), M, 2, 16)
        assert 0 < ng16 <= g16, (M, g16, ng16)


def test_device_wait_timeout_is_reported():
    # The failure path without a fault: with the test hook on, CTA 0 of each
    # register-fed GEMM ends with a bounded wait that nothing completes.  The
    # wait runs out (2 s), the status word reports MOE_ERR_TIMEOUT, the outputs
    # are still right, and the next forward runs clean on the same context.
    from weight_only_bit_moe_gb300 import binding as B
    wl = GPU_SMALL["int4-zipf-small"]
    W = wk.make_weights(wl, 131)
    X = wk.make_batch(wl, 20, 132)
    layer = _layer(W)
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    B.moe_set_test_starve_wait(True)
    try:
        out = run_layer(layer, wl, X, block_m=8)
    finally:
        B.moe_set_test_starve_wait(False)
    assert layer.status() == B.MOE_ERR_TIMEOUT
    check_close(out.float().cpu().numpy(), ref, "starved run")
    out = run_layer(layer, wl, X, block_m=8)
    assert layer.status() == B.MOE_OK
    check_close(out.float().cpu().numpy(), ref, "clean run after the timeout")
