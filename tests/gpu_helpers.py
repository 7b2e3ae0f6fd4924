"""Shared helpers of the GPU parity tests: numpy <-> torch marshalling, the two
sides of the pipeline (CUDA library / oracle) on the same seeded inputs, and
guarded output buffers that catch out-of-bounds writes."""
from __future__ import annotations

import numpy as np
import torch

import combine_ep_get_05_gb300 as ep
import oracle

GUARD = 4096  # guard elements before and after every guarded buffer
SENT_BF16 = 0x7FBF  # a NaN pattern no kernel produces
SENT_I32 = -123456
SENT_F32 = -7.5


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 / uint8 / int / float tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def guarded(shape, dtype, fill) -> tuple[torch.Tensor, torch.Tensor]:
    """A buffer of `shape` inside a larger allocation whose head and tail hold `fill`.

    Returns (view, backing); check_guards(backing, ...) verifies the guards."""
    n = int(np.prod(shape)) if len(shape) else 1
    backing = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        backing.view(torch.int16).fill_(int(np.array(fill, np.uint16).view(np.int16)))
    else:
        backing.fill_(fill)
    return backing[GUARD:GUARD + n].view(shape), backing


def check_guards(backing: torch.Tensor, n: int, fill) -> None:
    head = host_bits(backing[:GUARD])
    tail = host_bits(backing[GUARD + n:])
    assert np.all(head == fill) and np.all(tail == fill), "a kernel wrote outside its output buffer"


def gpu_expert(recv_x: torch.Tensor, recv_topk_w: torch.Tensor, recv_scales=None) -> torch.Tensor:
    """The harness expert on the GPU (torch elementwise ops, not a step of the path):
    y = bf16(v * w), w = ((0 + w_0) + w_1) + ... in fp32, v = x or float(q) * scale."""
    w = torch.zeros(recv_topk_w.shape[:2], dtype=torch.float32, device=recv_topk_w.device)
    for j in range(recv_topk_w.shape[2]):
        w = w + recv_topk_w[:, :, j]
    if recv_scales is None:
        v = recv_x.float()
    else:
        q = recv_x.view(torch.float8_e4m3fn).float()
        v = q * recv_scales.repeat_interleave(128, dim=2)
    return (v * w[:, :, None]).to(torch.bfloat16)


def oracle_expert(w, D, L):
    if w.expert == "identity":
        return D["recv_x"]
    return oracle.expert_scale(D["recv_x"], D["recv_topk_w"], L["tokens_per_rank"], D["recv_scales"])


def gpu_layout(w):
    topk = torch.from_numpy(w.topk_idx).cuda()
    lay = ep.alloc_layout(w.T, w.E, w.R, w.ranks_per_node)
    ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
    return topk, lay


def layout_to_host(lay) -> dict:
    out = {
        "tokens_per_expert": host_bits(lay.tokens_per_expert),
        "tokens_per_rank": host_bits(lay.tokens_per_rank),
        "is_token_in_rank": host_bits(lay.is_token_in_rank),
        "slot": host_bits(lay.slot),
    }
    if lay.tokens_per_node is not None:
        out["tokens_per_node"] = host_bits(lay.tokens_per_node)
        out["is_token_in_node"] = host_bits(lay.is_token_in_node)
    return out
