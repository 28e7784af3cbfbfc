"""GPU parity of the INT4 variants -- zero points (integer and float), act-order
and group sizes 32 / 64 / 128 / one per row -- against the oracle, through the
C ABI (moe_repack_weights_ex and the forward), on both GEMM paths.  These are
the w*_zeros, is_zp_float, g_idx / sort_indices and group_blocks of
fused_marlin_moe in "Marlin MoE kernel occupancy ..." (sglang PR #31552).

Shapes span several 128-row GEMM1 tiles and 256-row GEMM2 tiles with a ragged
last tile (N not a multiple of 128, K not a multiple of 256).  Integer zero
points make (q - z) * s a 12-bit product, rounded once to fp16; float zero
points form q * s - z * s in fp16: both within the pages' bound, which every
output is checked against (and the output-scaled bound for the small outputs
of the relu2 case)."""
import dataclasses

import numpy as np
import pytest

import oracle
from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import bf16_to_f32, check_workload, need_gpu, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    oracle.build()


BASE = dataclasses.replace(wk.WORKLOADS["int4-skew"], K=384, N=320, E=6, top_k=2, routing="uniform", Ms=(40,))
VARIANTS = {
    "zp-int-g128": dataclasses.replace(BASE, N=384, zero_kind="int"),
    "zp-int-g64": dataclasses.replace(BASE, zero_kind="int", group_size=64),
    "zp-float-g32": dataclasses.replace(BASE, zero_kind="float", group_size=32),
    "sym-g32": dataclasses.replace(BASE, group_size=32),
    "sym-g64-bias": dataclasses.replace(BASE, group_size=64, bias_std=0.1),
    "channelwise": dataclasses.replace(BASE, N=384, group_size=-1),
    "actorder-g128": dataclasses.replace(BASE, N=384, act_order=True),
    "actorder-zp-g64": dataclasses.replace(BASE, act_order=True, zero_kind="int", group_size=64, bias_std=0.1),
    "actorder-zpf-g32": dataclasses.replace(BASE, act_order=True, zero_kind="float", group_size=32),
    "actorder-zp-g64-relu2": dataclasses.replace(wk.WORKLOADS["int4-relu2"], K=384, N=320, E=6, Ms=(40,),
                                                 act_order=True, zero_kind="int", group_size=64),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
@pytest.mark.parametrize("block_m", [8, 16, 32, 64, 128])
def test_int4_variant_parity(name, block_m):
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl = VARIANTS[name]
    W = wk.make_weights(wl, 201)
    X = wk.make_batch(wl, wl.Ms[0], 202)
    layer = MoELayer.from_numpy(W)
    out = run_layer(layer, wl, X, block_m=block_m)
    assert layer.status() == B.MOE_OK
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_workload(out.float().cpu().numpy(), ref, wl, f"{name} block_m={block_m}")


@pytest.mark.parametrize("name", ["actorder-zp-g64", "zp-float-g32"])
def test_int4_variant_separate_alignment(name):
    # the forward on moe_align's result (the prologue then places x's rows from the
    # given alignment, in each expert's column order for act-order) equals the
    # forward aligning itself, bit for bit
    import torch
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl = VARIANTS[name]
    W = wk.make_weights(wl, 211)
    X = wk.make_batch(wl, 33, 212)
    layer = MoELayer.from_numpy(W)
    for B in (8, 64):
        a = run_layer(layer, wl, X, block_m=B).clone()
        b = run_layer(layer, wl, X, block_m=B, separate_align=True).clone()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_act_order_groups_must_be_whole():
    # g_idx whose groups are not group_size indices each cannot be stored with
    # contiguous groups: the blob is marked and the forward reports it
    from weight_only_bit_moe_gb300 import binding as B
    from weight_only_bit_moe_gb300.layer import MoELayer
    wl = VARIANTS["actorder-g128"]
    W = wk.make_weights(wl, 221)
    W.w13_gidx[1, :3] = (W.w13_gidx[1, :3] + 1) % (wl.K // 128)
    layer = MoELayer.from_numpy(W)
    X = wk.make_batch(wl, 9, 222)
    run_layer(layer, wl, X, block_m=8)
    assert layer.status() == B.MOE_ERR_UNSUPPORTED


_full_variant = {}


def _full_variant_layer():
    if not _full_variant:
        from weight_only_bit_moe_gb300.layer import MoELayer
        wl = dataclasses.replace(wk.WORKLOADS["int4-uniform"], act_order=True, zero_kind="int", group_size=64)
        W = wk.make_weights(wl, 231)
        _full_variant["v"] = (wl, W, MoELayer.from_numpy(W))
    return _full_variant["v"]


@pytest.mark.parametrize("M", [1, 2, 256])
def test_int4_variant_full_shape(M):
    # zero points and act-order at the K=4096, N=1536, E=128, top_k=8 shape, every
    # token against the oracle: M=1 and 2 run the register-fed kernels with their
    # K cut across CTAs (stream-K), M=256 the tcgen05 kernels
    from weight_only_bit_moe_gb300 import binding as B
    wl, W, layer = _full_variant_layer()
    X = wk.make_batch(wl, M, 232 + M)
    out = run_layer(layer, wl, X)
    assert layer.status() == B.MOE_OK
    ref = bf16_to_f32(oracle.forward_workload(wl, W, X))
    check_workload(out.float().cpu().numpy(), ref, wl, f"int4 zp act-order M={M}")
