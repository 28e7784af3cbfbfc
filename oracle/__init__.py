"""CPU oracle for the weight-only 4-bit fused MoE layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never imports, links or calls it, and it shares no code with
the CUDA path: the arithmetic lives in ``moe_oracle.c`` (plain loops, fp64
accumulation, formats decoded from their bit-level definitions) and this module
only compiles it with gcc and marshals numpy arrays through ctypes.

Functions and the passages they follow are listed in ``moe_oracle.c``.  Every
function here is pinned by ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"libmoe_oracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

FMT_CODES = {"int4": 0, "mxfp4": 1, "nvfp4": 2}
ACT_CODES = {"silu_mul": 0, "sigmoid_alpha": 1, "relu2": 2}


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("num_experts", ctypes.c_int), ("hidden", ctypes.c_int),
                ("inter", ctypes.c_int), ("group", ctypes.c_int), ("interleaved", ctypes.c_int),
                ("w13", ctypes.c_void_p), ("w13_s", ctypes.c_void_p), ("w13_gs", ctypes.c_void_p),
                ("b13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w2_s", ctypes.c_void_p),
                ("w2_gs", ctypes.c_void_p), ("b2", ctypes.c_void_p), ("gated", ctypes.c_int),
                ("zero_kind", ctypes.c_int), ("w13_z", ctypes.c_void_p), ("w2_z", ctypes.c_void_p),
                ("w13_gidx", ctypes.c_void_p), ("w2_gidx", ctypes.c_void_p)]

ZERO_KINDS = {"": 0, "int": 1, "float": 2}


class _Batch(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("top_k", ctypes.c_int), ("expert_base", ctypes.c_int),
                ("act", ctypes.c_int), ("alpha", ctypes.c_double), ("limit", ctypes.c_double),
                ("rsf", ctypes.c_double), ("norm_eps", ctypes.c_double),
                ("x", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p),
                ("topk_weights", ctypes.c_void_p), ("post_norm_w", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            d, u16, i32, i64 = ctypes.c_double, ctypes.c_uint16, ctypes.c_int, ctypes.c_long
            p = ctypes.c_void_p
            L.orc_bf16_value.restype = d
            L.orc_bf16_value.argtypes = [u16]
            L.orc_bf16_round.restype = u16
            L.orc_bf16_round.argtypes = [d]
            for n in ("orc_e2m1_value", "orc_e8m0_value", "orc_e4m3_value", "orc_int4_value"):
                getattr(L, n).restype = d
                getattr(L, n).argtypes = [ctypes.c_uint]
            L.orc_dequant.restype = None
            L.orc_dequant.argtypes = [i32, p, p, i32, i32, i32, p, p]
            L.orc_dequant_ex.restype = None
            L.orc_dequant_ex.argtypes = [i32, p, p, p, i32, p, i32, i32, i32, p, p]
            L.orc_align_capacity.restype = i64
            L.orc_align_capacity.argtypes = [i32, i32, i32, i32]
            L.orc_align.restype = i32
            L.orc_align.argtypes = [p, i32, i32, i32, i32, i32, p, i64, p, p]
            L.orc_forward.restype = i32
            L.orc_forward.argtypes = [ctypes.POINTER(_Layer), ctypes.POINTER(_Batch), p, i32, p, p]
            L.orc_ffn_pair.restype = i32
            L.orc_ffn_pair.argtypes = [ctypes.POINTER(_Layer), ctypes.POINTER(_Batch), i32, i32, p, p, p]
            L.orc_num_threads.restype = i32
            L.orc_num_threads.argtypes = []
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_requant.restype = i32
            L.orc_requant.argtypes = [p, p, i64, i64, i64, p, i32, i32, i32, i32, ctypes.c_float, p]
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ formats

def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def bf16_round(v: float) -> int:
    return int(lib().orc_bf16_round(float(v)))


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e8m0_value(b: int) -> float:
    return lib().orc_e8m0_value(int(b))


def e4m3_value(b: int) -> float:
    return lib().orc_e4m3_value(int(b))


def int4_value(q: int) -> float:
    return lib().orc_int4_value(int(q))


def dequant(fmt: str, codes: np.ndarray, scales: np.ndarray, group: int,
            row_map: Optional[np.ndarray] = None, zeros: Optional[np.ndarray] = None, zero_kind: str = "",
            gidx: Optional[np.ndarray] = None) -> np.ndarray:
    """One expert's matrix: codes uint8 [R, C/2], scales [R, C/g] (and INT4 zero
    points [R, C/g], uint8 or bf16 bits, and act-order groups gidx int32 [C])
    -> float32 [rows, C].  group <= 0: one group per row."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    rows = codes.shape[0] if row_map is None else len(row_map)
    cols = codes.shape[1] * 2
    out = np.empty((rows, cols), dtype=np.float32)
    rm = None if row_map is None else np.ascontiguousarray(row_map, dtype=np.int32)
    z = None if zeros is None else np.ascontiguousarray(zeros)
    gi = None if gidx is None else np.ascontiguousarray(gidx, dtype=np.int32)
    lib().orc_dequant_ex(FMT_CODES[fmt], _ptr(codes), _ptr(scales), _ptr(z), ZERO_KINDS[zero_kind], _ptr(gi),
                         rows, cols, group, _ptr(rm), _ptr(out))
    return out


# ------------------------------------------------------------------ align

def align_capacity(M: int, top_k: int, num_experts: int, block_m: int) -> int:
    return int(lib().orc_align_capacity(M, top_k, num_experts, block_m))


def align(topk_ids: np.ndarray, num_experts: int, block_m: int, expert_base: int = 0):
    """-> (sorted_ids int32[cap], expert_ids int32[cap/block_m], n_padded int)."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    M, k = ids.shape
    cap = align_capacity(M, k, num_experts, block_m)
    sorted_ids = np.empty(cap, dtype=np.int32)
    expert_ids = np.empty(cap // block_m, dtype=np.int32)
    n_padded = np.zeros(1, dtype=np.int32)
    rc = lib().orc_align(_ptr(ids), M, k, expert_base, num_experts, block_m, _ptr(sorted_ids), cap,
                         _ptr(expert_ids), _ptr(n_padded))
    if rc != 0:
        raise ValueError("oracle align rejected its arguments")
    return sorted_ids, expert_ids, int(n_padded[0])


# ------------------------------------------------------------------ forward

def _structs(W, X, expert_base, act, alpha, limit, rsf, norm_eps, post_norm, keep):
    M, k = X.topk_ids.shape

    def c(a, dt=None):
        if a is None:
            return None
        a = np.ascontiguousarray(a if dt is None else a.astype(dt, copy=False))
        keep.append(a)
        return _ptr(a)

    zk = getattr(W, "zero_kind", "")
    layer = _Layer(FMT_CODES[W.fmt], W.E, W.K, W.N, W.group, int(W.interleaved),
                   c(W.w13, np.uint8), c(W.w13_s), c(W.w13_gs, np.float32), c(W.b13, np.uint16),
                   c(W.w2, np.uint8), c(W.w2_s), c(W.w2_gs, np.float32), c(W.b2, np.uint16),
                   int(getattr(W, "gated", True)), ZERO_KINDS[zk], c(getattr(W, "w13_z", None)),
                   c(getattr(W, "w2_z", None)), c(getattr(W, "w13_gidx", None), np.int32),
                   c(getattr(W, "w2_gidx", None), np.int32))
    pnw = X.post_norm_w if post_norm else None
    b = _Batch(M, k, expert_base, ACT_CODES[act], alpha, limit, rsf, norm_eps,
               c(X.x, np.uint16), c(X.topk_ids, np.int32), c(X.topk_weights, np.float32),
               c(pnw, np.uint16))
    return layer, b


def forward(weights, batch, *, expert_base: int = 0, act: str = "silu_mul", alpha: float = 1.702,
            limit: float = float("inf"), rsf: float = 1.0, norm_eps: float = 1e-8,
            post_norm: bool = False, tokens: Optional[Sequence[int]] = None,
            return_acc: bool = False):
    """Layer output for the listed tokens (all tokens when ``tokens`` is None).

    ``weights`` is a workloads.LayerWeights, ``batch`` a workloads.BatchInputs.
    Returns uint16 bf16 bits [len(tokens), K] (and the fp64 values before the
    final rounding when ``return_acc``).
    """
    W, X = weights, batch
    M, k = X.topk_ids.shape
    toks = np.arange(M, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    keep = []  # keep the contiguous copies alive during the call
    layer, b = _structs(W, X, expert_base, act, alpha, limit, rsf, norm_eps, post_norm, keep)
    out = np.empty((len(toks), W.K), dtype=np.uint16)
    acc = np.empty((len(toks), W.K), dtype=np.float64) if return_acc else None
    rc = lib().orc_forward(ctypes.byref(layer), ctypes.byref(b), _ptr(toks), len(toks), _ptr(out), _ptr(acc))
    if rc != 0:
        raise ValueError("oracle forward rejected its arguments")
    return (out, acc) if return_acc else out


def ffn_pair(weights, batch, e: int, t: int, *, expert_base: int = 0, act: str = "silu_mul",
             alpha: float = 1.702, limit: float = float("inf")):
    """(h[R], a[N], y[K]) of token t on local expert e, in fp64; R = 2N for
    gated experts, N for non-gated ones."""
    keep = []
    layer, b = _structs(weights, batch, expert_base, act, alpha, limit, 1.0, 1e-8, False, keep)
    N, K = weights.N, weights.K
    R = 2 * N if getattr(weights, "gated", True) else N
    h, a, y = np.empty(R), np.empty(N), np.empty(K)
    if lib().orc_ffn_pair(ctypes.byref(layer), ctypes.byref(b), e, t, _ptr(h), _ptr(a), _ptr(y)) != 0:
        raise ValueError("oracle ffn_pair rejected its arguments")
    return h, a, y


def forward_workload(wl, weights, batch, **kw):
    """forward() with the workload's own activation, norm and expert range."""
    return forward(weights, batch, expert_base=wl.expert_base, act=wl.act, alpha=wl.alpha,
                   limit=wl.limit, norm_eps=wl.norm_eps, post_norm=wl.post_norm, **kw)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits -> float32 values (shifts into the high half)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ requant (W4AFP8 activations)

def e4m3_encode(v: float) -> int:
    """fp32 value -> E4M3 byte: nearest, ties to even, saturating at +-448."""
    return int(lib().orc_e4m3_encode(float(v)))


def requant(x: np.ndarray, scale: np.ndarray, masked_m: np.ndarray, tensor_scale: float, group: int = 128,
            scale_strides: Optional[Sequence[int]] = None, out: Optional[np.ndarray] = None) -> np.ndarray:
    """Per-token -> per-tensor FP8 requantisation (see moe_oracle.c, orc_requant).

    x uint8 E4M3 [E, max_m, K]; scale: a contiguous fp32 buffer in which entry
    (e, g, m) sits at e*se + g*sg + m*sm, (se, sg, sm) = ``scale_strides``
    (default: [E, K/group, max_m], group-major per expert); masked_m int32 [E].
    Rows at or past masked_m keep ``out``'s bytes (zeros when ``out`` is None)."""
    x = np.ascontiguousarray(x, dtype=np.uint8)
    E, max_m, K = x.shape
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    if scale_strides is None:
        scale_strides = ((K // group) * max_m, max_m, 1)
    se, sg, sm = (int(v) for v in scale_strides)
    mm = np.ascontiguousarray(masked_m, dtype=np.int32)
    res = np.zeros_like(x) if out is None else np.array(out, dtype=np.uint8, copy=True)
    if lib().orc_requant(_ptr(x), _ptr(scale), se, sg, sm, _ptr(mm), E, max_m, K, group, float(tensor_scale),
                         _ptr(res)) != 0:
        raise ValueError("oracle requant rejected its arguments")
    return res
