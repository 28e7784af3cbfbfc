"""ctypes binding of the C ABI declared in include/moe_w4a16.h.

Argument marshalling only: torch tensors are passed as their data pointers,
streams as their CUDA handles; every step of the layer runs in the library's
CUDA kernels.  The functions carry the C names.  Loading fails loudly when the
library has not been built (``python -m weight_only_bit_moe_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import platform
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", f"libmoe_w4a16_{platform.machine()}.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
MOE_W_INT4_U4B8, MOE_W_MXFP4, MOE_W_NVFP4 = 0, 1, 2
MOE_ACT_SILU_MUL, MOE_ACT_SIGMOID_ALPHA, MOE_ACT_RELU2 = 0, 1, 2

EXPORTED = ("moe_repack_size", "moe_repack_weights", "moe_repack_weights_ex", "moe_align_capacity", "moe_align", "moe_choose_block_m",
            "moe_workspace_size", "moe_w4a16_forward", "moe_w4a16_forward_noalloc", "moe_get_status",
            "moe_set_trace_events", "moe_set_test_starve_wait", "moe_status_string", "moe_requant_fp8",
            "moe_requant_launch_geometry")
MOE_NOALLOC_SCRATCH_BYTES = 64 << 20  # fixed workspace of moe_w4a16_forward_noalloc


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({status_string(status)})")
        self.status = status


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("group_size", ctypes.c_int32), ("w13_interleaved", ctypes.c_int32),
                ("has_bias13", ctypes.c_int32), ("has_bias2", ctypes.c_int32), ("non_gated", ctypes.c_int32),
                ("zero_kind", ctypes.c_int32), ("act_order", ctypes.c_int32)]


class moe_repack_tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w13", "w13_s", "w13_gs", "b13", "w13_zeros", "w13_g_idx", "w13_sort_indices",
        "w2", "w2_s", "w2_gs", "b2", "w2_zeros", "w2_g_idx", "w2_sort_indices")]


_lib = None
_lock = threading.Lock()


def load(path: str = ""):
    """Load the CUDA library (once).  Raises if it is missing: there is no fallback.
    MOE_W4A16_LIB overrides the library path (e.g. an alternative build)."""
    global _lib
    path = path or os.environ.get("MOE_W4A16_LIB", LIB_PATH)
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} is missing "
                                   "(run python -m weight_only_bit_moe_gb300.build)")
            L = ctypes.CDLL(path)
            p, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            D = ctypes.POINTER(moe_layer_desc)
            sig = {
                "moe_repack_size": (i64, [D]),
                "moe_repack_weights": (i32, [D, p, p, p, p, p, p, p, p, p, p]),
                "moe_repack_weights_ex": (i32, [D, ctypes.POINTER(moe_repack_tensors), p, p]),
                "moe_align_capacity": (i64, [i32, i32, i32, i32]),
                "moe_align": (i32, [p, i32, i32, i32, i32, i32, p, p, p, p]),
                "moe_choose_block_m": (i32, [D, i32, i32, i32]),
                "moe_workspace_size": (i64, [D, i32, i32, i32]),
                "moe_w4a16_forward": (i32, [D, p, p, i32, i32, p, p, i32, p, p, p, i32, i32, f32, f32, f32, p,
                                            f32, p, p, i64, p]),
                "moe_w4a16_forward_noalloc": (i32, [D, p, p, i32, i32, p, p, i32, p, p, p, i32, i32, f32, f32, f32,
                                                    p, f32, p, p]),
                "moe_get_status": (i32, [p, p]),
                "moe_set_trace_events": (i32, [ctypes.POINTER(ctypes.c_void_p), i32]),
                "moe_set_test_starve_wait": (i32, [i32]),
                "moe_status_string": (ctypes.c_char_p, [i32]),
                "moe_requant_fp8": (i32, [p, p, i64, i64, i64, p, i32, i32, i32, i32, p, p, i32, p]),
                "moe_requant_launch_geometry": (i32, [i32, i32, i32, i32, ctypes.POINTER(i32),
                                                      ctypes.POINTER(i32)]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _lib = L
    return _lib


def _p(t):
    """Device/host pointer of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc != MOE_OK:
        raise MoeError(fn, rc)
    return rc


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_repack_size(desc: moe_layer_desc) -> int:
    n = load().moe_repack_size(ctypes.byref(desc))
    if n < 0:
        raise MoeError("moe_repack_size", MOE_ERR_INVALID)
    return n


def moe_repack_weights(desc, w13, w13_s, w13_gs, b13, w2, w2_s, w2_gs, b2, packed, stream=None):
    return _check("moe_repack_weights", load().moe_repack_weights(
        ctypes.byref(desc), _p(w13), _p(w13_s), _p(w13_gs), _p(b13), _p(w2), _p(w2_s), _p(w2_gs), _p(b2),
        _p(packed), _stream(stream)))


def moe_repack_weights_ex(desc, tensors: dict, packed, stream=None):
    """tensors: the moe_repack_tensors fields by name (tensors or None)."""
    t = moe_repack_tensors(**{k: _p(v) for k, v in tensors.items()})
    return _check("moe_repack_weights_ex", load().moe_repack_weights_ex(
        ctypes.byref(desc), ctypes.byref(t), _p(packed), _stream(stream)))


def moe_align_capacity(M: int, top_k: int, num_experts: int, block_m: int) -> int:
    n = load().moe_align_capacity(M, top_k, num_experts, block_m)
    if n < 0:
        raise MoeError("moe_align_capacity", MOE_ERR_INVALID)
    return n


def moe_align(topk_ids, M, top_k, expert_base, num_experts, block_m, sorted_ids, expert_ids, n_padded,
              stream=None):
    return _check("moe_align", load().moe_align(
        _p(topk_ids), M, top_k, expert_base, num_experts, block_m, _p(sorted_ids), _p(expert_ids),
        _p(n_padded), _stream(stream)))


def moe_choose_block_m(desc, M: int, top_k: int, num_routed_ids: int) -> int:
    b = load().moe_choose_block_m(ctypes.byref(desc), M, top_k, num_routed_ids)
    if b <= 0:
        raise MoeError("moe_choose_block_m", b)
    return b


def moe_workspace_size(desc, M: int, top_k: int, block_m: int) -> int:
    n = load().moe_workspace_size(ctypes.byref(desc), M, top_k, block_m)
    if n < 0:
        raise MoeError("moe_workspace_size", MOE_ERR_INVALID)
    return n


def moe_w4a16_forward(desc, packed, x, M, top_k, topk_ids, topk_weights, expert_base, sorted_ids, expert_ids,
                      n_padded, block_m, act, alpha, limit, routed_scaling_factor, post_norm_w, norm_eps, out,
                      workspace, workspace_bytes, stream=None):
    return _check("moe_w4a16_forward", load().moe_w4a16_forward(
        ctypes.byref(desc), _p(packed), _p(x), M, top_k, _p(topk_ids), _p(topk_weights), expert_base,
        _p(sorted_ids), _p(expert_ids), _p(n_padded), block_m, act, alpha, limit, routed_scaling_factor,
        _p(post_norm_w), norm_eps, _p(out), _p(workspace), workspace_bytes, _stream(stream)))


def moe_w4a16_forward_noalloc(desc, packed, x, M, top_k, topk_ids, topk_weights, expert_base, sorted_ids,
                              expert_ids, n_padded, block_m, act, alpha, limit, routed_scaling_factor, post_norm_w,
                              norm_eps, out, stream=None):
    """moe_w4a16_forward on the library's fixed device scratch (no workspace argument)."""
    rc = load().moe_w4a16_forward_noalloc(
        ctypes.byref(desc), _p(packed), _p(x), M, top_k, _p(topk_ids), _p(topk_weights), expert_base,
        _p(sorted_ids), _p(expert_ids), _p(n_padded), block_m, act, alpha, limit, routed_scaling_factor,
        _p(post_norm_w), norm_eps, _p(out), _stream(stream))
    if rc == MOE_ERR_WORKSPACE:
        raise MoeError("moe_w4a16_forward_noalloc (shape needs more than the "
                       f"{MOE_NOALLOC_SCRATCH_BYTES >> 20} MiB fixed scratch)", rc)
    return _check("moe_w4a16_forward_noalloc", rc)


def moe_get_status(workspace, stream=None) -> int:
    return load().moe_get_status(_p(workspace), _stream(stream))


def moe_set_trace_events(events) -> None:
    """events: four torch.cuda.Event (created with enable_timing) or None to stop."""
    if events is None:
        _check("moe_set_trace_events", load().moe_set_trace_events(None, 0))
        return
    handles = []
    for ev in events:
        if ev.cuda_event == 0:
            ev.record()  # torch creates the CUDA event on its first record
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles)
    _check("moe_set_trace_events", load().moe_set_trace_events(arr, len(handles)))


def moe_set_test_starve_wait(on: bool) -> None:
    """Test hook of the device failure path (see include/moe_w4a16.h)."""
    _check("moe_set_test_starve_wait", load().moe_set_test_starve_wait(1 if on else 0))


def moe_requant_fp8(x, scale, scale_strides, masked_m, num_experts, max_m, K, group, tensor_scale, out,
                    expected_rows=-1, stream=None):
    """Per-token -> per-tensor FP8 requantisation (include/moe_requant.h).  scale_strides
    = (e, g, m) element strides of the fp32 scale buffer."""
    se, sg, sm = (int(v) for v in scale_strides)
    return _check("moe_requant_fp8", load().moe_requant_fp8(
        _p(x), _p(scale), se, sg, sm, _p(masked_m), num_experts, max_m, K, group, _p(tensor_scale), _p(out),
        int(expected_rows), _stream(stream)))


def moe_requant_launch_geometry(num_experts: int, K: int, expected_rows: int, sm_count: int):
    """(ctas, threads) moe_requant_fp8 launches with (host only)."""
    c, t = ctypes.c_int(0), ctypes.c_int(0)
    _check("moe_requant_launch_geometry", load().moe_requant_launch_geometry(
        num_experts, K, expected_rows, sm_count, ctypes.byref(c), ctypes.byref(t)))
    return c.value, t.value
