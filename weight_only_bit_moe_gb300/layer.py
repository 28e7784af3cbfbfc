"""A thin PyTorch-facing wrapper of the C ABI: owns the device buffers (packed
weights, alignment outputs, workspace) as torch tensors and calls the library
in order.  It performs no arithmetic of the layer itself.

Typical use::

    layer = MoELayer.from_numpy(weights, device="cuda")        # repack once
    out = layer(x, topk_ids, topk_weights)                      # aligns inside the forward
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

from . import binding as B

FMT = {"int4": B.MOE_W_INT4_U4B8, "mxfp4": B.MOE_W_MXFP4, "nvfp4": B.MOE_W_NVFP4}
ACT = {"silu_mul": B.MOE_ACT_SILU_MUL, "sigmoid_alpha": B.MOE_ACT_SIGMOID_ALPHA, "relu2": B.MOE_ACT_RELU2}
GROUP = {"int4": 128, "mxfp4": 32, "nvfp4": 16}
ZERO_KIND = {"": 0, "int": 1, "float": 2}


def _dev(a: Optional[np.ndarray], device, dtype=None) -> Optional[torch.Tensor]:
    """Host array -> device tensor with the same bytes (uint16 travels as int16)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


@dataclasses.dataclass
class AlignOut:
    block_m: int
    sorted_ids: torch.Tensor
    expert_ids: torch.Tensor
    n_padded: torch.Tensor


class MoELayer:
    """One layer's expert bank on one GPU, repacked for the kernels."""

    def __init__(self, fmt: str, num_experts: int, hidden: int, inter: int, w13, w13_s, w13_gs, b13, w2, w2_s,
                 w2_gs, b2, interleaved: bool = False, gated: bool = True, group_size: int = 0,
                 zero_kind: str = "", w13_zeros=None, w2_zeros=None, w13_g_idx=None, w2_g_idx=None,
                 w13_sort_indices=None, w2_sort_indices=None, stream=None):
        """group_size 0: the format's own; INT4 variants: zero_kind "int" / "float" with
        w*_zeros, act-order with w*_g_idx and w*_sort_indices, group_size 32/64/128/-1."""
        self.fmt = fmt
        self.E, self.K, self.N = num_experts, hidden, inter
        self.gated = gated  # False: w13 holds N rows and the activation is relu2
        act_order = w13_g_idx is not None
        self.desc = B.moe_layer_desc(FMT[fmt], num_experts, hidden, inter, group_size or GROUP[fmt],
                                     int(interleaved), int(b13 is not None), int(b2 is not None), int(not gated),
                                     ZERO_KIND[zero_kind], int(act_order))
        dev = w13.device
        self.device = dev
        self.packed = torch.empty(B.moe_repack_size(self.desc), dtype=torch.uint8, device=dev)
        B.moe_repack_weights_ex(self.desc, dict(
            w13=w13, w13_s=w13_s, w13_gs=w13_gs, b13=b13, w13_zeros=w13_zeros, w13_g_idx=w13_g_idx,
            w13_sort_indices=w13_sort_indices, w2=w2, w2_s=w2_s, w2_gs=w2_gs, b2=b2, w2_zeros=w2_zeros,
            w2_g_idx=w2_g_idx, w2_sort_indices=w2_sort_indices), self.packed, stream)
        self._ws = {}

    @classmethod
    def from_numpy(cls, W, device="cuda", stream=None) -> "MoELayer":
        """W: a workloads.LayerWeights (host arrays in checkpoint layout)."""
        t = dict(w13=_dev(W.w13, device), w13_s=_dev(W.w13_s, device), w13_gs=_dev(W.w13_gs, device),
                 b13=_dev(W.b13, device), w2=_dev(W.w2, device), w2_s=_dev(W.w2_s, device),
                 w2_gs=_dev(W.w2_gs, device), b2=_dev(W.b2, device),
                 w13_zeros=_dev(getattr(W, "w13_z", None), device), w2_zeros=_dev(getattr(W, "w2_z", None), device),
                 w13_g_idx=_dev(getattr(W, "w13_gidx", None), device),
                 w2_g_idx=_dev(getattr(W, "w2_gidx", None), device),
                 w13_sort_indices=_dev(getattr(W, "w13_perm", None), device),
                 w2_sort_indices=_dev(getattr(W, "w2_perm", None), device))
        layer = cls(W.fmt, W.E, W.K, W.N, interleaved=W.interleaved, gated=W.gated, group_size=W.group,
                    zero_kind=getattr(W, "zero_kind", ""), stream=stream, **t)
        torch.cuda.current_stream(device).synchronize()  # source tensors may be freed after this
        return layer

    # ------------------------------------------------------------ align
    def alloc_align(self, M: int, top_k: int, block_m: int) -> AlignOut:
        cap = B.moe_align_capacity(M, top_k, self.E, block_m)
        d = self.device
        return AlignOut(block_m, torch.empty(cap, dtype=torch.int32, device=d),
                        torch.empty(max(cap // block_m, 1), dtype=torch.int32, device=d),
                        torch.empty(1, dtype=torch.int32, device=d))

    def align(self, topk_ids: torch.Tensor, expert_base: int = 0, block_m: Optional[int] = None,
              num_routed_ids: Optional[int] = None, out: Optional[AlignOut] = None, stream=None) -> AlignOut:
        M, k = topk_ids.shape
        if block_m is None:
            block_m = self.choose_block_m(M, k, num_routed_ids or self.E)
        a = out if out is not None else self.alloc_align(M, k, block_m)
        B.moe_align(topk_ids, M, k, expert_base, self.E, block_m, a.sorted_ids, a.expert_ids, a.n_padded, stream)
        return a

    def choose_block_m(self, M: int, top_k: int, num_routed_ids: int) -> int:
        return B.moe_choose_block_m(self.desc, M, top_k, num_routed_ids)

    # ------------------------------------------------------------ forward
    def workspace(self, M: int, top_k: int, block_m: int) -> torch.Tensor:
        key = (M, top_k, block_m)
        ws = self._ws.get(key)
        if ws is None:
            n = B.moe_workspace_size(self.desc, M, top_k, block_m)
            ws = torch.empty(n, dtype=torch.uint8, device=self.device)
            self._ws = {key: ws}  # keep one workspace alive
        return ws

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                a: Optional[AlignOut] = None, expert_base: int = 0, act: Optional[str] = None,
                alpha: float = 1.702, limit: float = math.inf, routed_scaling_factor: float = 1.0,
                post_norm_w: Optional[torch.Tensor] = None, norm_eps: float = 1e-8,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                block_m: Optional[int] = None, num_routed_ids: Optional[int] = None, stream=None) -> torch.Tensor:
        """The layer on an alignment from align() (a), or with a = None on the
        alignment the forward computes itself in its first kernel (block_m chosen
        by the library unless given)."""
        M, k = topk_ids.shape
        if act is None:  # the layer's own kind: silu_and_mul when gated, relu2 otherwise
            act = "silu_mul" if self.gated else "relu2"
        if out is None:
            out = torch.empty((M, self.K), dtype=torch.bfloat16, device=self.device)
        if a is not None:
            bm, s_ids, e_ids, n_pad = a.block_m, a.sorted_ids, a.expert_ids, a.n_padded
        else:
            bm = block_m or self.choose_block_m(M, k, num_routed_ids or self.E)
            s_ids = e_ids = n_pad = None
        ws = workspace if workspace is not None else self.workspace(M, k, bm)
        B.moe_w4a16_forward(self.desc, self.packed, x, M, k, topk_ids, topk_weights, expert_base, s_ids, e_ids,
                            n_pad, bm, ACT[act], alpha, limit, routed_scaling_factor, post_norm_w, norm_eps, out, ws,
                            ws.numel(), stream)
        return out

    def __call__(self, x, topk_ids, topk_weights, expert_base: int = 0, block_m: Optional[int] = None,
                 num_routed_ids: Optional[int] = None, separate_align: bool = False, **kw) -> torch.Tensor:
        """align + forward.  By default the forward aligns the routing itself (one
        launch fewer); separate_align = True runs moe_align first, as the pages do."""
        if not separate_align:
            return self.forward(x, topk_ids, topk_weights, None, expert_base=expert_base, block_m=block_m,
                                num_routed_ids=num_routed_ids, **kw)
        a = self.align(topk_ids, expert_base, block_m, num_routed_ids)
        return self.forward(x, topk_ids, topk_weights, a, expert_base=expert_base, **kw)

    def status(self, workspace: Optional[torch.Tensor] = None, stream=None) -> int:
        ws = workspace if workspace is not None else next(iter(self._ws.values()))
        return B.moe_get_status(ws, stream)


def batch_to_device(X, device="cuda"):
    """workloads.BatchInputs -> (x bf16, topk_ids int32, topk_weights fp32, post_norm_w bf16 or None)."""
    x = _dev(X.x, device, torch.bfloat16)
    ids = _dev(X.topk_ids.astype(np.int32, copy=False), device)
    w = _dev(X.topk_weights.astype(np.float32, copy=False), device)
    pnw = _dev(X.post_norm_w, device, torch.bfloat16)
    return x, ids, w, pnw
