"""Host-side checks of the C-ABI library that need no GPU: it builds for
sm_103a, loads, exports every function include/moe_w4a16.h declares, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from weight_only_bit_moe_gb300 import build, binding
    build.build()
    return binding


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    L = lib.load()
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(lib.EXPORTED)


def test_capacity_matches_oracle(lib, orc):
    for M, k, E, B in [(0, 2, 8, 16), (1, 8, 32, 16), (123, 2, 8, 16), (4096, 8, 128, 128), (7, 3, 1024, 8)]:
        assert lib.moe_align_capacity(M, k, E, B) == orc.align_capacity(M, k, E, B)


def test_repack_size_rules(lib):
    D = lib.moe_layer_desc
    assert lib.moe_repack_size(D(0, 8, 512, 1024, 128, 0, 1, 1)) > 0
    assert lib.moe_repack_size(D(1, 32, 2880, 2880, 32, 1, 1, 1)) > 0     # tile padding allowed
    assert lib.moe_repack_size(D(2, 32, 4096, 4096, 16, 0, 0, 0)) > 0
    for g in (32, 64, 128, -1):                       # INT4 group sizes
        assert lib.moe_repack_size(D(0, 8, 512, 1024, g, 0, 1, 1)) > 0
    assert lib.moe_repack_size(D(0, 8, 512, 1024, 64, 0, 1, 1, 0, 1, 1)) > 0  # zero points + act-order
    assert lib.moe_repack_size(D(0, 8, 512, 1024, 32, 0, 1, 1, 0, 2, 0)) > 0  # float zero points
    for bad in [D(0, 8, 512, 1024, 96, 0, 0, 0),      # not a group size for int4
                D(0, 8, 512, 1024, 16, 0, 0, 0),
                D(0, 8, 512, 1024, -1, 0, 0, 0, 0, 0, 1),  # act-order needs group sizes
                D(0, 8, 512, 1024, 128, 0, 0, 0, 0, 3, 0),  # unknown zero kind
                D(1, 8, 512, 512, 32, 0, 0, 0, 0, 1, 0),    # zero points are INT4-only
                D(2, 8, 512, 512, 16, 0, 0, 0, 0, 0, 1),    # act-order is INT4-only
                D(0, 8, 576, 1024, 128, 0, 0, 0),     # int4 hidden % 128
                D(1, 8, 2880, 2890, 32, 0, 0, 0),     # inter % group
                D(1, 8, 2900, 2880, 32, 0, 0, 0),     # hidden % 64
                D(3, 8, 512, 512, 16, 0, 0, 0),       # unknown format
                D(2, 0, 512, 512, 16, 0, 0, 0)]:      # no experts
        with pytest.raises(lib.MoeError):
            lib.moe_repack_size(bad)


def test_non_gated_layout_rules(lib):
    """Non-gated w13 tiles hold 256 rows of h instead of 128 gate + 128 up rows:
    at K=512, N=1024 (INT4, 8 experts) the bank loses half its w13 tiles -- 4
    tiles x 4 scale periods x (512 scale bytes + 2 x 8192 code bytes) per expert --
    and half its GEMM1 bias (1024 bf16 per expert)."""
    D = lib.moe_layer_desc
    gated = lib.moe_repack_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 0))
    plain = lib.moe_repack_size(D(0, 8, 512, 1024, 128, 0, 1, 1, 1))
    assert gated - plain == 8 * 4 * 4 * (512 + 2 * 8192) + 8 * 1024 * 2
    assert lib.moe_repack_size(D(1, 4, 192, 160, 32, 0, 0, 0, 1)) > 0   # N pads to 256
    for bad in [D(1, 8, 512, 512, 32, 1, 0, 0, 1),    # non-gated rows cannot be interleaved
                D(0, 8, 512, 1024, 128, 0, 0, 0, 2)]:  # flag is 0 or 1
        with pytest.raises(lib.MoeError):
            lib.moe_repack_size(bad)


def test_binding_struct_matches_header(lib):
    """The ctypes moe_layer_desc has the header struct's fields, in order, all int32."""
    text = open(os.path.join(ROOT, "include", "moe_w4a16.h")).read()
    body = re.search(r"typedef struct moe_layer_desc \{(.*?)\} moe_layer_desc;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"int32_t\s+(\w+)\s*;", body)
    assert fields == [f for f, _ in lib.moe_layer_desc._fields_]
    assert all(t is ctypes.c_int32 for _, t in lib.moe_layer_desc._fields_)
    assert ctypes.sizeof(lib.moe_layer_desc) == 4 * len(fields)


def test_rejects_bad_arguments_without_device(lib):
    L = lib.load()
    # align: bad block_m, too many experts, null outputs -> MOE_ERR_INVALID before any CUDA call
    assert L.moe_align(None, 4, 2, 0, 8, 24, 1, 1, 1, None) == lib.MOE_ERR_INVALID
    assert L.moe_align(None, 4, 2, 0, 2000, 16, 1, 1, 1, None) == lib.MOE_ERR_INVALID
    assert L.moe_align(1, 4, 2, 0, 8, 16, None, 1, 1, None) == lib.MOE_ERR_INVALID
    d = lib.moe_layer_desc(0, 8, 512, 1024, 128, 0, 0, 0)
    fwd = L.moe_w4a16_forward
    args = [ctypes.byref(d), 256, 256, 4, 2, 8, 8, 0, 8, 8, 8, 16, 0, 1.0, 1.0, 1.0, None, 1e-8, 8, 256, 1 << 30,
            None]
    bad_act = list(args)
    bad_act[12] = 7
    assert fwd(*bad_act) == lib.MOE_ERR_INVALID
    bad_bm = list(args)
    bad_bm[11] = 24
    assert fwd(*bad_bm) == lib.MOE_ERR_INVALID
    bad_topk = list(args)
    bad_topk[4] = 17
    assert fwd(*bad_topk) == lib.MOE_ERR_INVALID
    misaligned = list(args)
    misaligned[1] = 257  # packed not 256-byte aligned
    assert fwd(*misaligned) == lib.MOE_ERR_INVALID
    zero = list(args)
    zero[3] = 0          # M == 0 is a no-op
    assert fwd(*zero) == lib.MOE_OK
    # the activation must match the experts' gating, even for an empty batch
    relu2_on_gated = list(zero)
    relu2_on_gated[12] = lib.MOE_ACT_RELU2
    assert fwd(*relu2_on_gated) == lib.MOE_ERR_INVALID
    ng = lib.moe_layer_desc(0, 8, 512, 1024, 128, 0, 0, 0, 1)
    silu_on_plain = list(zero)
    silu_on_plain[0] = ctypes.byref(ng)
    assert fwd(*silu_on_plain) == lib.MOE_ERR_INVALID
    silu_on_plain[12] = lib.MOE_ACT_RELU2
    assert fwd(*silu_on_plain) == lib.MOE_OK
    assert lib.status_string(lib.MOE_ERR_TIMEOUT) == "device wait timed out"


def test_block_m_chooser(lib):
    """The choice minimises expected blocks (Poisson rows per expert) times a
    block's measured cost; every pair below was measured faster on GB300 than
    the alternatives named beside it."""
    d = lib.moe_layer_desc(0, 128, 4096, 1536, 128, 0, 0, 0)
    nv = lib.moe_layer_desc(2, 32, 4096, 4096, 16, 0, 0, 0)
    mx = lib.moe_layer_desc(1, 32, 2880, 2880, 32, 1, 1, 1)
    small_k = lib.moe_layer_desc(0, 8, 512, 1024, 128, 0, 1, 1)  # 8 K-stages: 64-token tiles
    assert lib.moe_choose_block_m(d, 1, 8, 128) == 8
    assert lib.moe_choose_block_m(d, 16, 8, 128) == 8
    assert lib.moe_choose_block_m(d, 128, 8, 128) == 16      # int4, 8 rows: vs 8 and 64
    assert lib.moe_choose_block_m(d, 256, 8, 128) == 64      # int4, 16 rows: vs 16
    assert lib.moe_choose_block_m(d, 512, 8, 128) == 64      # int4, 32 rows: vs 32
    assert lib.moe_choose_block_m(d, 768, 8, 128) == 64      # int4, 48 rows: vs 128
    assert lib.moe_choose_block_m(d, 1024, 8, 128) == 128    # int4, 64 rows: vs 64
    assert lib.moe_choose_block_m(d, 4096, 8, 128) == 128    # vs 64
    assert lib.moe_choose_block_m(nv, 128, 8, 256) == 8      # nvfp4, 4 rows: vs 64
    assert lib.moe_choose_block_m(nv, 256, 8, 256) == 64     # nvfp4, 8 rows: vs 8 and 16
    assert lib.moe_choose_block_m(nv, 512, 8, 256) == 64     # nvfp4, 16 rows: vs 16 and 32
    assert lib.moe_choose_block_m(mx, 32, 4, 32) == 8        # mxfp4, 4 rows: vs 16
    assert lib.moe_choose_block_m(mx, 64, 4, 32) == 64       # mxfp4, 8 rows: vs 8 and 16
    assert lib.moe_choose_block_m(mx, 128, 4, 32) == 64      # mxfp4, 16 rows: vs 16 and 32
    assert lib.moe_choose_block_m(mx, 384, 4, 32) == 64      # mxfp4, 48 rows: vs 32 and 128
    assert lib.moe_choose_block_m(mx, 1024, 4, 32) == 128    # vs 64
    assert lib.moe_choose_block_m(small_k, 2304, 2, 8) == 64  # short K: vs 128
    # monotone in the token count, every format
    for desc, k, nid in [(d, 8, 128), (nv, 8, 256), (mx, 4, 32)]:
        prev = 0
        for M in [1, 2, 8, 32, 64, 96, 128, 192, 256, 384, 512, 1024, 4096, 65536]:
            b = lib.moe_choose_block_m(desc, M, k, nid)
            assert b >= prev and b in (8, 16, 32, 64, 128), (M, b, prev)
            prev = b
