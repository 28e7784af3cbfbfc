"""Seeded synthetic inputs for the W4A16 fused-MoE layer.

This module only draws random numbers and stores them in the input formats the
layer consumes (bf16 bits, packed 4-bit codes, E8M0 / E4M3 scale bytes). It holds
none of the layer's arithmetic: no dequantisation, no GEMM, no activation, no
routing alignment and no combine. Both the CPU oracle (through the tests and the
benchmark) and the CUDA path are fed from the arrays returned here.

The workloads follow the problem statements on the source pages:

* ``tiny-int4``       the small int4 case (K=256, N=128, E=8, top_k=2).
* ``int4-bias``       the int4 shape of the large-M schedule test in
                      "Marlin MoE kernel occupancy ..." (sglang PR #31552),
                      section 关键源码片段 (test_fused_marlin_moe_large_non_ep_schedule):
                      n=1024, k=512, e=8, topk=2, group 128, per-expert bias.
* ``mxfp4-alpha``     GPT-OSS-like MXFP4 experts with interleaved gate/up rows and
                      the sigmoid-alpha gate, "SM120 MXFP4 MoE ... Marlin"
                      (sglang PR #28231), sections 实现拆解 and 关键源码片段.
* ``nvfp4-ep-norm``   one EP8 rank of the Muse Spark NVFP4 expert path with the
                      post-expert norm, "013-moe-middle-tiles.py" (``Weights``,
                      ``Config``, ``Inputs``).
* ``int4-skew`` / ``int4-uniform``  int4 K=4096, N=1536, E=128, top_k=8 with
                      Zipf(1.2) or uniform routing.
* ``int4-relu2``      the PR #31552 test shape as that test writes it: non-gated
                      experts (w1 [E, N, K]) with relu(h)^2, x = randn/10, bias
                      = randn/100.

Distributions not fixed by the pages (stated here once): x ~ N(0,1) in bf16
(times the workload's x_scale);
routing ids distinct per token (Gumbel-top-k over the routing distribution);
top-k weights = softmax over the k slots of N(0,1) logits, in fp32; NVFP4 global
scales ~ U[0.008, 0.012].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

FMT_INT4 = "int4"    # uint4b8: code q in 0..15 stands for q - 8, bf16 scale per group
FMT_MXFP4 = "mxfp4"  # E2M1 codes, E8M0 scale byte per 32 along the reduction dim
FMT_NVFP4 = "nvfp4"  # E2M1 codes, E4M3 scale per 16, fp32 global scale per expert

ACT_SILU_MUL = "silu_mul"
ACT_SIGMOID_ALPHA = "sigmoid_alpha"
ACT_RELU2 = "relu2"  # non-gated experts: relu(h)^2

GROUP = {FMT_INT4: 128, FMT_MXFP4: 32, FMT_NVFP4: 16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    fmt: str
    K: int            # hidden size (GEMM1 reduction, GEMM2 output)
    N: int            # intermediate size (GEMM1 output is 2N, GEMM2 reduction)
    E: int            # local experts held by this GPU
    top_k: int
    Ms: tuple         # token counts exercised
    E_global: int = 0  # routed id range; 0 means equal to E (no expert parallelism)
    expert_base: int = 0
    bias_std: float = 0.0          # 0 = no bias
    interleaved: bool = False      # w13 rows stored gate0, up0, gate1, up1, ...
    act: str = ACT_SILU_MUL
    alpha: float = 1.702
    limit: float = math.inf
    post_norm: bool = False
    norm_eps: float = 1e-8
    routing: str = "uniform"       # "uniform" | "zipf"
    zipf_s: float = 1.2
    gated: bool = True             # False: w1 has N rows and act is relu2
    x_scale: float = 1.0           # x ~ N(0, x_scale^2)
    group_size: int = 0            # INT4: 0 = the format's 128; 32 / 64 / 128; -1 = one group per row
    zero_kind: str = ""            # INT4 zero points: "" (uint4b8), "int" (bytes 0..15), "float" (bf16)
    act_order: bool = False        # INT4: groups given per reduction index (g_idx) in a random order

    @property
    def group(self) -> int:
        return self.group_size or GROUP[self.fmt]

    @property
    def n_ids(self) -> int:
        return self.E_global or self.E


WORKLOADS = {
    "tiny-int4": Workload("tiny-int4", FMT_INT4, K=256, N=128, E=8, top_k=2, Ms=(16,)),
    "int4-bias": Workload("int4-bias", FMT_INT4, K=512, N=1024, E=8, top_k=2,
                          Ms=(123, 2304), bias_std=0.1),
    "mxfp4-alpha": Workload("mxfp4-alpha", FMT_MXFP4, K=2880, N=2880, E=32, top_k=4,
                            Ms=(1, 32, 1024), bias_std=0.05, interleaved=True,
                            act=ACT_SIGMOID_ALPHA),
    "nvfp4-ep-norm": Workload("nvfp4-ep-norm", FMT_NVFP4, K=4096, N=4096, E=32, top_k=8,
                              Ms=(1, 8, 64, 512), E_global=256, expert_base=0,
                              post_norm=True),
    "int4-skew": Workload("int4-skew", FMT_INT4, K=4096, N=1536, E=128, top_k=8,
                          Ms=(1, 16, 256, 4096), routing="zipf"),
    "int4-uniform": Workload("int4-uniform", FMT_INT4, K=4096, N=1536, E=128, top_k=8,
                             Ms=(1, 16, 256, 4096), routing="uniform"),
    # the large-M schedule test of "Marlin MoE kernel occupancy ..." (PR #31552)
    # as it is written: non-gated relu2 experts, x = randn/10, bias = randn/100
    "int4-relu2": Workload("int4-relu2", FMT_INT4, K=512, N=1024, E=8, top_k=2,
                           Ms=(123, 2304), bias_std=0.01, gated=False, act=ACT_RELU2, x_scale=0.1),
}

WORKLOAD_INDEX = {"tiny-int4": 0, "int4-bias": 1, "mxfp4-alpha": 2, "nvfp4-ep-norm": 3,
                  "int4-skew": 4, "int4-uniform": 5, "int4-relu2": 6}


def weight_seed(name: str) -> int:
    """Weights depend on the workload only: seed = 1000 * workload index."""
    return 1000 * WORKLOAD_INDEX[name]


def batch_seed(name: str, M: int, rep: int = 0) -> int:
    """seed = 1000 * workload index + 1 + (M mod 997) + 100000 * repetition."""
    return 1000 * WORKLOAD_INDEX[name] + 1 + (M % 997) + 100000 * rep


# ---------------------------------------------------------------- encodings of draws

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 draws to bf16 (round-to-nearest-even, torch's cast) -> uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 draws to FP8 E4M3 (torch's float8_e4m3fn cast) -> uint8 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


# ---------------------------------------------------------------- layer weights

@dataclasses.dataclass
class LayerWeights:
    """Raw expert weights, in the layout the pages' checkpoints use.

    w13    uint8 [E, R, K/2]   two 4-bit codes per byte, low nibble = even index;
                               R = 2N (gate and up) or N for non-gated experts
    w13_s  [E, R, K/g]         uint16 bf16 bits (int4) | uint8 E8M0 (mxfp4) | uint8 E4M3 (nvfp4)
    w13_gs float32 [E]         nvfp4 only (one global scale per expert, gate and up)
    b13    uint16 bf16 bits [E, R] or None
    w2     uint8 [E, K, N/2];  w2_s [E, K, N/g];  w2_gs float32 [E];  b2 uint16 [E, K] or None
    When ``interleaved`` the 2N rows of w13 (and its scale and bias rows) are
    gate0, up0, gate1, up1, ...; otherwise gate rows [0, N) then up rows [N, 2N).
    """
    fmt: str
    E: int
    K: int
    N: int
    group: int
    interleaved: bool
    w13: np.ndarray
    w13_s: np.ndarray
    w13_gs: Optional[np.ndarray]
    b13: Optional[np.ndarray]
    w2: np.ndarray
    w2_s: np.ndarray
    w2_gs: Optional[np.ndarray]
    b2: Optional[np.ndarray]
    gated: bool = True
    zero_kind: str = ""                 # INT4 zero points: "", "int" or "float"
    w13_z: Optional[np.ndarray] = None  # [E, R, K/g] uint8 (int) or uint16 bf16 bits (float)
    w2_z: Optional[np.ndarray] = None   # [E, K, N/g]
    w13_gidx: Optional[np.ndarray] = None  # int32 [E, K]: group of each reduction index (act-order)
    w2_gidx: Optional[np.ndarray] = None   # int32 [E, N]
    w13_perm: Optional[np.ndarray] = None  # int32 [E, K]: reduction indices ordered by group (sort_indices)
    w2_perm: Optional[np.ndarray] = None   # int32 [E, N]


def _scales(rng: np.random.Generator, fmt: str, shape) -> np.ndarray:
    if fmt == FMT_INT4:
        return to_bf16_bits(rng.uniform(0.005, 0.02, size=shape).astype(np.float32))
    if fmt == FMT_MXFP4:
        # E8M0 byte = 127 + exponent, exponent uniform in [-8, -4]
        return (127 + rng.integers(-8, -3, size=shape)).astype(np.uint8)
    if fmt == FMT_NVFP4:
        return to_e4m3_bits(rng.uniform(0.5, 2.0, size=shape).astype(np.float32))
    raise ValueError(fmt)


def _groups(g: int, cols: int) -> int:
    return 1 if g < 0 else cols // g


def _act_order(rng: np.random.Generator, E: int, cols: int, g: int):
    """Per expert a random order of the reduction indices; index k belongs to
    group (its place in that order) // g, as GPTQ's act-order assigns them.  Returns
    g_idx [E, cols] and sort_indices [E, cols] (indices by ascending group, ties in
    index order)."""
    size = cols if g < 0 else g
    gidx = np.empty((E, cols), dtype=np.int32)
    for e in range(E):
        order = rng.permutation(cols)
        gidx[e, order] = np.arange(cols) // size
    perm = np.argsort(gidx, axis=1, kind="stable").astype(np.int32)
    return gidx, perm


def make_weights(wl: Workload, seed: int) -> LayerWeights:
    rng = np.random.Generator(np.random.PCG64(seed))
    E, K, N, g = wl.E, wl.K, wl.N, wl.group
    R = 2 * N if wl.gated else N  # rows of w13
    # every code value equally likely: uniform bytes give uniform nibbles
    w13 = rng.integers(0, 256, size=(E, R, K // 2), dtype=np.uint8)
    w13_s = _scales(rng, wl.fmt, (E, R, _groups(g, K)))
    w2 = rng.integers(0, 256, size=(E, K, N // 2), dtype=np.uint8)
    w2_s = _scales(rng, wl.fmt, (E, K, _groups(g, N)))
    w13_gs = w2_gs = None
    if wl.fmt == FMT_NVFP4:
        w13_gs = rng.uniform(0.008, 0.012, size=E).astype(np.float32)
        w2_gs = rng.uniform(0.008, 0.012, size=E).astype(np.float32)
    b13 = b2 = None
    if wl.bias_std > 0:
        b13 = to_bf16_bits(rng.normal(0.0, wl.bias_std, size=(E, R)).astype(np.float32))
        b2 = to_bf16_bits(rng.normal(0.0, wl.bias_std, size=(E, K)).astype(np.float32))
    extra = {}
    if wl.zero_kind == "int":  # a zero point per (row, group), uniform over the 16 codes
        extra["w13_z"] = rng.integers(0, 16, size=w13_s.shape, dtype=np.uint8)
        extra["w2_z"] = rng.integers(0, 16, size=w2_s.shape, dtype=np.uint8)
    elif wl.zero_kind == "float":  # HQQ-style float zero points in the code range
        extra["w13_z"] = to_bf16_bits(rng.uniform(0.0, 15.0, size=w13_s.shape).astype(np.float32))
        extra["w2_z"] = to_bf16_bits(rng.uniform(0.0, 15.0, size=w2_s.shape).astype(np.float32))
    if wl.act_order:
        extra["w13_gidx"], extra["w13_perm"] = _act_order(rng, E, K, g)
        extra["w2_gidx"], extra["w2_perm"] = _act_order(rng, E, N, g)
    return LayerWeights(wl.fmt, E, K, N, g, wl.interleaved, w13, w13_s, w13_gs, b13,
                        w2, w2_s, w2_gs, b2, gated=wl.gated, zero_kind=wl.zero_kind, **extra)


# ---------------------------------------------------------------- per-batch inputs

@dataclasses.dataclass
class BatchInputs:
    x: np.ndarray             # uint16 bf16 bits [M, K]
    topk_ids: np.ndarray      # int32 [M, top_k], ids in [0, n_ids)
    topk_weights: np.ndarray  # float32 [M, top_k]
    post_norm_w: Optional[np.ndarray]  # uint16 bf16 bits [K] (applied as 1 + w) or None


def routing_log_probs(wl: Workload) -> np.ndarray:
    """Log routing probabilities over the routed ids (fixed per workload)."""
    n = wl.n_ids
    if wl.routing == "uniform":
        return np.zeros(n)
    if wl.routing == "zipf":
        rng = np.random.Generator(np.random.PCG64(weight_seed(wl.name) + 17))
        ranks = rng.permutation(n) + 1          # seeded rank -> expert id assignment
        return -wl.zipf_s * np.log(ranks.astype(np.float64))
    raise ValueError(wl.routing)


def make_batch(wl: Workload, M: int, seed: int) -> BatchInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = to_bf16_bits(rng.standard_normal((M, wl.K), dtype=np.float32) * np.float32(wl.x_scale))
    logp = routing_log_probs(wl)
    # Gumbel-top-k: k distinct ids per token, drawn without replacement from p
    gumbel = -np.log(-np.log(rng.uniform(1e-12, 1.0, size=(M, wl.n_ids))))
    keys = logp[None, :] + gumbel
    ids = np.argsort(-keys, axis=1, kind="stable")[:, : wl.top_k].astype(np.int32)
    logits = rng.standard_normal((M, wl.top_k)).astype(np.float32)
    ex = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    pnw = None
    if wl.post_norm:
        pnw = to_bf16_bits(rng.normal(0.0, 0.02, size=wl.K).astype(np.float32))
    return BatchInputs(x, ids, w, pnw)


def make_case(name: str, M: int, rep: int = 0):
    wl = WORKLOADS[name]
    return wl, make_weights(wl, weight_seed(name)), make_batch(wl, M, batch_seed(name, M, rep))


# ---------------------------------------------------------------- W4AFP8 activation requantisation

@dataclasses.dataclass(frozen=True)
class RequantWorkload:
    """An expert-major FP8 activation payload as a low-latency dispatcher hands it
    to the W4AFP8 expert GEMM ("W4AFP8 requant ..." (sglang PR #35760)): E experts
    of max_m row slots of K columns, masked_m valid rows each, one fp32 scale per
    (row, 128-column group)."""
    name: str
    E: int
    max_m: int
    K: int
    rows: str            # "one" (1 row per expert), "uniform", "skew" (one hot expert), "random"
    mean_rows: int = 1
    skew: int = 16       # "skew": the hot expert takes skew * mean_rows (capped at max_m)
    group: int = 128


REQUANT_WORKLOADS = {
    # the page's decode case: 256 local experts, one row each, DeepSeek-V3 width
    "requant-ll-1row": RequantWorkload("requant-ll-1row", E=256, max_m=128, K=7168, rows="one"),
    # a loaded low-latency batch, evenly and unevenly routed
    "requant-ll-uniform": RequantWorkload("requant-ll-uniform", E=32, max_m=512, K=7168, rows="uniform",
                                          mean_rows=256),
    "requant-ll-skew": RequantWorkload("requant-ll-skew", E=32, max_m=1024, K=7168, rows="skew", mean_rows=64),
}


@dataclasses.dataclass
class RequantInputs:
    x: np.ndarray         # uint8 E4M3 [E, max_m, K]
    scale: np.ndarray     # fp32 [E, K/group, max_m] (group-major per expert, the dispatcher's layout)
    masked_m: np.ndarray  # int32 [E]
    tensor_scale: float   # S


def make_requant(wl: RequantWorkload, seed: int) -> RequantInputs:
    """Codes uniform over the finite E4M3 values, scales U[0.002, 0.02], S = 0.01 (so
    that products span the format and some saturate), valid rows by wl.rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = rng.integers(0, 254, size=(wl.E, wl.max_m, wl.K), dtype=np.int64)
    codes = codes + (codes >= 0x7F)  # skip 0x7F (NaN); 0xFF is past the range
    x = codes.astype(np.uint8)
    scale = rng.uniform(0.002, 0.02, size=(wl.E, wl.K // wl.group, wl.max_m)).astype(np.float32)
    if wl.rows == "one":
        mm = np.ones(wl.E, dtype=np.int32)
    elif wl.rows == "uniform":
        mm = np.full(wl.E, wl.mean_rows, dtype=np.int32)
    elif wl.rows == "skew":
        mm = np.full(wl.E, wl.mean_rows, dtype=np.int32)
        mm[int(rng.integers(0, wl.E))] = wl.skew * wl.mean_rows
    else:
        mm = rng.integers(0, wl.max_m + 1, size=wl.E).astype(np.int32)
    mm = np.minimum(mm, wl.max_m).astype(np.int32)
    return RequantInputs(x, scale, mm, 0.01)
