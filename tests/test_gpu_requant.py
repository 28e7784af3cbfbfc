"""The FP8 requantisation kernel (moe_requant_fp8) against the oracle, byte for
byte: every valid element of every expert, rows at or past masked_m untouched,
both scale layouts, several launch geometries giving the same bytes ("W4AFP8
requant ...", sglang PR #35760: the kernel's outputs are bitwise identical
across launch geometries), empty experts, clamped masked_m and in-place use."""
import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_moe_gb300 import workloads as wk
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    oracle.build()


def run(X, group, layout="group-major", expected_rows=-1, out=None, in_place=False):
    from weight_only_bit_moe_gb300 import binding as B
    E, max_m, K = X.x.shape
    G = K // group
    if layout == "group-major":
        scale = X.scale
        strides = (G * max_m, max_m, 1)
    else:
        scale = np.ascontiguousarray(np.transpose(X.scale, (0, 2, 1)))
        strides = (max_m * G, 1, G)
    dx = torch.from_numpy(X.x).cuda()
    ds = torch.from_numpy(np.ascontiguousarray(scale)).cuda()
    dm = torch.from_numpy(X.masked_m).cuda()
    dS = torch.tensor([X.tensor_scale], dtype=torch.float32, device="cuda")
    dout = dx if in_place else (torch.from_numpy(out).cuda() if out is not None else torch.zeros_like(dx))
    B.moe_requant_fp8(dx, ds, strides, dm, E, max_m, K, group, dS, dout, expected_rows)
    torch.cuda.synchronize()
    return dout.cpu().numpy()


CASES = [
    # (E, max_m, K, rows, mean_rows, group, seed)
    (1, 1, 128, "one", 1, 128, 1),
    (8, 17, 896, "random", 1, 128, 2),
    (40, 32, 7168, "random", 1, 128, 3),
    (256, 4, 7168, "one", 1, 128, 4),
    (3, 64, 384, "uniform", 40, 64, 5),
    (32, 256, 7168, "skew", 8, 128, 6),
    (1024, 2, 256, "random", 1, 128, 7),
]


@pytest.mark.parametrize("E,max_m,K,rows,mean,group,seed", CASES)
@pytest.mark.parametrize("layout", ["group-major", "row-major"])
def test_requant_bit_exact(E, max_m, K, rows, mean, group, seed, layout):
    wl = wk.RequantWorkload("t", E=E, max_m=max_m, K=K, rows=rows, mean_rows=mean, group=group)
    X = wk.make_requant(wl, seed)
    canvas = np.full_like(X.x, 0xA5)
    want = oracle.requant(X.x, X.scale, X.masked_m, X.tensor_scale, group=group, out=canvas)
    got = run(X, group, layout, out=canvas)
    np.testing.assert_array_equal(got, want)


def test_requant_geometry_does_not_change_bytes():
    wl = wk.RequantWorkload("t", E=56, max_m=48, K=3584, rows="random")
    X = wk.make_requant(wl, 11)
    want = oracle.requant(X.x, X.scale, X.masked_m, X.tensor_scale)
    for rows in (-1, 1, 8, 9, 48, 1024):
        np.testing.assert_array_equal(run(X, 128, expected_rows=rows), want, err_msg=f"expected_rows={rows}")


def test_requant_empty_experts_and_clamps():
    wl = wk.RequantWorkload("t", E=9, max_m=5, K=256, rows="random")
    X = wk.make_requant(wl, 12)
    X.masked_m[:] = [0, 5, -3, 7, 0, 1, 0, 0, 2]  # negative -> 0, beyond max_m -> max_m
    canvas = np.full_like(X.x, 0x3C)
    want = oracle.requant(X.x, X.scale, X.masked_m, X.tensor_scale, out=canvas)
    np.testing.assert_array_equal(run(X, 128, out=canvas), want)
    X.masked_m[:] = 0
    np.testing.assert_array_equal(run(X, 128, out=canvas), canvas)  # nothing valid: nothing written


def test_requant_in_place():
    wl = wk.RequantWorkload("t", E=4, max_m=9, K=1024, rows="random")
    X = wk.make_requant(wl, 13)
    want = oracle.requant(X.x, X.scale, X.masked_m, X.tensor_scale, out=X.x)
    np.testing.assert_array_equal(run(X, 128, in_place=True), want)


def test_requant_page_decode_shape():
    # 256 local experts with one row each at DeepSeek-V3 width, every row checked
    X = wk.make_requant(wk.REQUANT_WORKLOADS["requant-ll-1row"], 14)
    want = oracle.requant(X.x, X.scale, X.masked_m, X.tensor_scale)
    np.testing.assert_array_equal(run(X, 128, expected_rows=1), want)
