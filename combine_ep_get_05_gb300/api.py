"""Convenience layer over the C ABI: allocate the caller-owned buffers with torch
and chain the entry points. It adds no computation: every step still runs in
the library's kernels (see _lib.py)."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib as L


@dataclass
class Layout:
    tokens_per_expert: torch.Tensor  # int32 [E]
    tokens_per_rank: torch.Tensor    # int32 [R]
    tokens_per_node: Optional[torch.Tensor]  # int32 [N] or None
    is_token_in_rank: torch.Tensor   # uint8 [T][R]
    is_token_in_node: Optional[torch.Tensor]  # uint8 [T][N] or None
    slot: torch.Tensor               # int32 [T][R]
    workspace: torch.Tensor          # uint8, zero-filled once, reusable
    status: torch.Tensor             # int32 [1]
    num_experts: int
    num_ranks: int
    ranks_per_node: int


@dataclass
class Dispatched:
    recv_x: torch.Tensor              # bf16 or uint8 (e4m3) [R][max_tokens][H]
    recv_scales: Optional[torch.Tensor]   # fp32 [R][max_tokens][H/128] (e4m3 only)
    recv_src_idx: Optional[torch.Tensor]  # int32 [R][max_tokens]
    recv_topk_idx: Optional[torch.Tensor]  # int32 [R][max_tokens][k]
    recv_topk_w: Optional[torch.Tensor]    # fp32 [R][max_tokens][k]
    status: torch.Tensor
    max_tokens: int


def alloc_layout(T: int, num_experts: int, num_ranks: int, ranks_per_node: int = 0, device="cuda") -> Layout:
    dev = torch.device(device)
    N = num_ranks // ranks_per_node if ranks_per_node > 0 else 0
    ws_bytes = L.ep_layout_workspace_size(T, num_experts, num_ranks, ranks_per_node)
    i32 = dict(dtype=torch.int32, device=dev)
    return Layout(
        tokens_per_expert=torch.empty(num_experts, **i32),
        tokens_per_rank=torch.empty(num_ranks, **i32),
        tokens_per_node=torch.empty(N, **i32) if N else None,
        is_token_in_rank=torch.empty((T, num_ranks), dtype=torch.uint8, device=dev),
        is_token_in_node=torch.empty((T, N), dtype=torch.uint8, device=dev) if N else None,
        slot=torch.empty((T, num_ranks), **i32),
        workspace=torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev),
        status=torch.zeros(1, **i32),
        num_experts=num_experts, num_ranks=num_ranks, ranks_per_node=ranks_per_node,
    )


def alloc_dispatch(num_ranks: int, max_tokens: int, H: int, k: int, fp8: bool = False, metadata: bool = True,
                   device="cuda") -> Dispatched:
    dev = torch.device(device)
    shape = (num_ranks, max_tokens, H)
    return Dispatched(
        recv_x=torch.empty(shape, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
        recv_scales=torch.empty((num_ranks, max_tokens, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
        recv_src_idx=torch.empty((num_ranks, max_tokens), dtype=torch.int32, device=dev) if metadata else None,
        recv_topk_idx=torch.empty((num_ranks, max_tokens, k), dtype=torch.int32, device=dev) if metadata else None,
        recv_topk_w=torch.empty((num_ranks, max_tokens, k), dtype=torch.float32, device=dev) if metadata else None,
        status=torch.zeros(1, dtype=torch.int32, device=dev),
        max_tokens=max_tokens,
    )


def get_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, ranks_per_node: int = 0,
               out: Optional[Layout] = None, stream=None) -> Layout:
    T = topk_idx.shape[0]
    lay = out if out is not None else alloc_layout(T, num_experts, num_ranks, ranks_per_node, topk_idx.device)
    L.ep_get_layout(topk_idx, num_experts, num_ranks, ranks_per_node, lay.tokens_per_expert, lay.tokens_per_rank,
                    lay.tokens_per_node, lay.is_token_in_rank, lay.is_token_in_node, lay.slot, lay.workspace,
                    lay.status, stream)
    return lay


def dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, layout: Layout, max_tokens: int,
             fp8: bool = False, out: Optional[Dispatched] = None, stream=None) -> Dispatched:
    T, H = x.shape
    k = topk_idx.shape[1]
    d = out if out is not None else alloc_dispatch(layout.num_ranks, max_tokens, H, k, fp8, device=x.device)
    L.ep_dispatch(x, L.DTYPE_E4M3 if fp8 else L.DTYPE_BF16, topk_idx, topk_w, layout.slot, layout.num_experts,
                  layout.num_ranks, max_tokens, d.recv_x, d.recv_scales, d.recv_src_idx, d.recv_topk_idx,
                  d.recv_topk_w, d.status, stream)
    return d


def combine(y: torch.Tensor, layout: Layout, max_tokens: int, out: Optional[torch.Tensor] = None,
            status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T = layout.slot.shape[0]
    H = y.shape[2]
    o = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    L.ep_combine(y, layout.slot, max_tokens, o, status, stream)
    return o


def read_flags(status: torch.Tensor) -> int:
    """Synchronise and return the asynchronous EP_FLAG_* bits of a status word."""
    return int(status.item())


def combine_fp8(y, y_scales, layout: Layout, max_tokens: int, out=None, status=None) -> torch.Tensor:
    """Combine of FP8 expert outputs (E4M3 codes [R][max_tokens][H] + scales) into bf16 [T][H]."""
    R, _, H = y.shape
    T = layout.slot.shape[0]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    L.ep_combine_fp8(y, y_scales, layout.slot, max_tokens, out, status)
    return out


def combine_weights(recv_topk_w, layout: Layout, max_tokens: int, out=None, status=None) -> torch.Tensor:
    """The combined top-k weights [T][k]: the received weight rows summed back to token order."""
    T = layout.slot.shape[0]
    if out is None:
        out = torch.empty((T, recv_topk_w.shape[2]), dtype=torch.float32, device=recv_topk_w.device)
    L.ep_combine_weights(recv_topk_w, layout.slot, max_tokens, out, status)
    return out

