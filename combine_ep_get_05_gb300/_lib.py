"""ctypes binding of libep_gb300.so (include/ep.h): argument marshalling only.

Every function takes torch tensors, checks their device, dtype, shape and
contiguity, passes raw device pointers and the current (or given) CUDA stream
to the C entry point of the same name, and raises ``EpError`` on a non-OK
synchronous status. All work happens in the library's CUDA kernels; there is
no CPU path. If the library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

EP_OK = 0
EP_ERR_INVALID = 1
EP_ERR_CUDA = 2
EP_ERR_SCRATCH = 3
LAYOUT_NOALLOC_SCRATCH_BYTES = 1 << 20

FLAG_CAPACITY = 1
FLAG_BAD_EXPERT = 2
FLAG_TIMEOUT = 4
FLAG_WORKSPACE = 8

DTYPE_BF16 = 0
DTYPE_E4M3 = 1

NODES_DENSE = 0
NODES_SPARSE = 1

ABI_VERSION = 1

EXPORTS = (
    "ep_abi_version", "ep_status_str", "ep_last_cuda_error", "ep_layout_workspace_size",
    "ep_get_layout", "ep_get_layout_noalloc", "ep_dispatch", "ep_restripe_prob", "ep_dispatch_nodes", "ep_combine",
    "ep_combine_fp8", "ep_combine_weights",
    "ep_expert_layout_workspace_size", "ep_get_expert_layout", "ep_dispatch_permuted", "ep_permute_received",
    "ep_combine_permuted", "ep_dispatch_permuted_ll", "ep_combine_send", "ep_combine_permuted_ll",
)


class EpError(RuntimeError):
    """A library call returned a non-OK synchronous status."""

    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        msg = f"{fn}: {lib().ep_status_str(status).decode()}"
        if status == EP_ERR_CUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)
        self.status = status
        self.cuda_error = cuda_error


_lock = threading.Lock()
_lib = None


def lib():
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build the CUDA library first "
                        "(python -m combine_ep_get_05_gb300.build or __graft_entry__.build())")
                L = ctypes.CDLL(LIB_PATH)
                P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
                sigs = {
                    "ep_abi_version": (i32, []),
                    "ep_status_str": (ctypes.c_char_p, [i32]),
                    "ep_last_cuda_error": (i32, []),
                    "ep_layout_workspace_size": (sz, [i32, i32, i32, i32]),
                    "ep_get_layout": (i32, [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P, P]),
                    "ep_get_layout_noalloc": (i32, [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P]),
                    "ep_dispatch": (i32, [P, i32, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]),
                    "ep_restripe_prob": (i32, [P, i32, i32, i32, i32, P, P]),
                    "ep_dispatch_nodes": (i32, [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P, P]),
                    "ep_combine": (i32, [P, P, i32, i32, i32, i32, P, P, P]),
                    "ep_combine_fp8": (i32, [P, P, P, i32, i32, i32, i32, P, P, P]),
                    "ep_dispatch_permuted_ll": (i32, [P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]),
                    "ep_combine_weights": (i32, [P, P, i32, i32, i32, i32, P, P, P]),
                    "ep_expert_layout_workspace_size": (sz, [i32, i32]),
                    "ep_get_expert_layout": (i32, [P, i32, i32, i32, P, P, P, sz, P, P]),
                    "ep_dispatch_permuted": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P]),
                    "ep_permute_received": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                                  P, P]),
                    "ep_combine_permuted": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]),
                    "ep_combine_permuted_ll": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]),
                    "ep_combine_send": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P]),
                }
                for name, (res, args) in sigs.items():
                    f = getattr(L, name)
                    f.restype, f.argtypes = res, args
                if L.ep_abi_version() != ABI_VERSION:
                    raise RuntimeError(f"{LIB_PATH}: ABI version {L.ep_abi_version()} != {ABI_VERSION}")
                _lib = L
    return _lib


# --------------------------------------------------------------------------- helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(name, t, dtype, shape=None, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _done(fn, rc):
    if rc != EP_OK:
        raise EpError(fn, rc, lib().ep_last_cuda_error() if rc == EP_ERR_CUDA else 0)


# --------------------------------------------------------------------------- entry points

def ep_layout_workspace_size(T: int, E: int, R: int, ranks_per_node: int = 0) -> int:
    return int(lib().ep_layout_workspace_size(T, E, R, ranks_per_node))


def ep_get_layout(topk_idx, num_experts, num_ranks, ranks_per_node, tokens_per_expert, tokens_per_rank,
                  tokens_per_node, is_token_in_rank, is_token_in_node, slot, workspace, status=None,
                  stream=None):
    T, k = topk_idx.shape
    E, R = num_experts, num_ranks
    N = R // ranks_per_node if ranks_per_node > 0 else 0
    _check("topk_idx", topk_idx, torch.int64)
    _check("tokens_per_expert", tokens_per_expert, torch.int32, (E,))
    _check("tokens_per_rank", tokens_per_rank, torch.int32, (R,))
    _check("tokens_per_node", tokens_per_node, torch.int32, (N,), optional=N == 0)
    _check("is_token_in_rank", is_token_in_rank, torch.uint8, (T, R))
    _check("is_token_in_node", is_token_in_node, torch.uint8, (T, N), optional=N == 0)
    _check("slot", slot, torch.int32, (T, R))
    _check("workspace", workspace, torch.uint8)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_get_layout(
        _ptr(topk_idx), T, k, E, R, ranks_per_node, _ptr(tokens_per_expert), _ptr(tokens_per_rank),
        _ptr(tokens_per_node) if N else None, _ptr(is_token_in_rank), _ptr(is_token_in_node) if N else None,
        _ptr(slot), _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _done("ep_get_layout", rc)


def ep_get_layout_noalloc(topk_idx, num_experts, num_ranks, ranks_per_node, tokens_per_expert, tokens_per_rank,
                          tokens_per_node, is_token_in_rank, is_token_in_node, slot, status=None, stream=None):
    """ep_get_layout without a workspace (for callers that cannot allocate one); see include/ep.h."""
    T, k = topk_idx.shape
    E, R = num_experts, num_ranks
    N = R // ranks_per_node if ranks_per_node > 0 else 0
    _check("topk_idx", topk_idx, torch.int64)
    _check("tokens_per_expert", tokens_per_expert, torch.int32, (E,))
    _check("tokens_per_rank", tokens_per_rank, torch.int32, (R,))
    _check("tokens_per_node", tokens_per_node, torch.int32, (N,), optional=N == 0)
    _check("is_token_in_rank", is_token_in_rank, torch.uint8, (T, R))
    _check("is_token_in_node", is_token_in_node, torch.uint8, (T, N), optional=N == 0)
    _check("slot", slot, torch.int32, (T, R))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_get_layout_noalloc(
        _ptr(topk_idx), T, k, E, R, ranks_per_node, _ptr(tokens_per_expert), _ptr(tokens_per_rank),
        _ptr(tokens_per_node) if N else None, _ptr(is_token_in_rank), _ptr(is_token_in_node) if N else None,
        _ptr(slot), _ptr(status), _stream(stream))
    _done("ep_get_layout_noalloc", rc)


def ep_dispatch(x, out_dtype, topk_idx, topk_w, slot, num_experts, num_ranks, max_tokens, recv_x,
                recv_scales=None, recv_src_idx=None, recv_topk_idx=None, recv_topk_w=None, status=None,
                stream=None):
    T, H = x.shape
    k = topk_idx.shape[1]
    R = num_ranks
    fp8 = out_dtype == DTYPE_E4M3
    _check("x", x, torch.bfloat16)
    _check("topk_idx", topk_idx, torch.int64, (T, k))
    _check("topk_w", topk_w, torch.float32, (T, k), optional=True)
    _check("slot", slot, torch.int32, (T, R))
    _check("recv_x", recv_x, torch.uint8 if fp8 else torch.bfloat16, (R, max_tokens, H))
    _check("recv_scales", recv_scales, torch.float32, (R, max_tokens, H // 128), optional=not fp8)
    _check("recv_src_idx", recv_src_idx, torch.int32, (R, max_tokens), optional=True)
    _check("recv_topk_idx", recv_topk_idx, torch.int32, (R, max_tokens, k), optional=True)
    _check("recv_topk_w", recv_topk_w, torch.float32, (R, max_tokens, k), optional=True)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_dispatch(
        _ptr(x), out_dtype, _ptr(topk_idx), _ptr(topk_w), _ptr(slot), T, H, k, num_experts, R, max_tokens,
        _ptr(recv_x), _ptr(recv_scales), _ptr(recv_src_idx), _ptr(recv_topk_idx), _ptr(recv_topk_w),
        _ptr(status), _stream(stream))
    _done("ep_dispatch", rc)


def ep_restripe_prob(prob, max_tokens, out, stream=None):
    T, N, P = prob.shape
    _check("prob", prob, torch.float32)
    _check("out", out, torch.float32, (N, max_tokens, P))
    rc = lib().ep_restripe_prob(_ptr(prob), T, N, P, max_tokens, _ptr(out), _stream(stream))
    _done("ep_restripe_prob", rc)


def ep_dispatch_nodes(x, prob_staging, is_token_in_node, num_nodes, max_tokens, chunk_tokens, mode, recv_x_node,
                      recv_prob_node=None, num_runs=None, stream=None):
    T, H = x.shape
    N = num_nodes
    P = prob_staging.shape[2] if prob_staging is not None else 0
    _check("x", x, torch.bfloat16)
    _check("prob_staging", prob_staging, torch.float32, (N, max_tokens, P), optional=True)
    _check("is_token_in_node", is_token_in_node, torch.uint8, (T, N), optional=mode == NODES_DENSE)
    _check("recv_x_node", recv_x_node, torch.bfloat16, (N, max_tokens, H))
    _check("recv_prob_node", recv_prob_node, torch.float32, (N, max_tokens, P), optional=prob_staging is None)
    nchunks = (T + chunk_tokens - 1) // chunk_tokens if chunk_tokens > 0 else 0
    _check("num_runs", num_runs, torch.int32, (N, nchunks), optional=True)
    rc = lib().ep_dispatch_nodes(
        _ptr(x), _ptr(prob_staging), _ptr(is_token_in_node), T, H, N, P, max_tokens, chunk_tokens, mode,
        _ptr(recv_x_node), _ptr(recv_prob_node), _ptr(num_runs), _stream(stream))
    _done("ep_dispatch_nodes", rc)


def ep_combine(y, slot, max_tokens, out, status=None, stream=None):
    R, M, H = y.shape
    T = slot.shape[0]
    _check("y", y, torch.bfloat16, (R, max_tokens, H))
    _check("slot", slot, torch.int32, (T, R))
    _check("out", out, torch.bfloat16, (T, H))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine(_ptr(y), _ptr(slot), T, H, R, max_tokens, _ptr(out), _ptr(status), _stream(stream))
    _done("ep_combine", rc)


def ep_combine_fp8(y, y_scales, slot, max_tokens, out, status=None, stream=None):
    R, M, H = y.shape
    T = slot.shape[0]
    _check("y", y, torch.uint8, (R, max_tokens, H))
    _check("y_scales", y_scales, torch.float32, (R, max_tokens, H // 128))
    _check("slot", slot, torch.int32, (T, R))
    _check("out", out, torch.bfloat16, (T, H))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine_fp8(_ptr(y), _ptr(y_scales), _ptr(slot), T, H, R, max_tokens, _ptr(out), _ptr(status),
                              _stream(stream))
    _done("ep_combine_fp8", rc)


def ep_combine_weights(recv_topk_w, slot, max_tokens, combined_w, status=None, stream=None):
    R, M, k = recv_topk_w.shape
    T = slot.shape[0]
    _check("recv_topk_w", recv_topk_w, torch.float32, (R, max_tokens, k))
    _check("slot", slot, torch.int32, (T, R))
    _check("combined_w", combined_w, torch.float32, (T, k))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine_weights(_ptr(recv_topk_w), _ptr(slot), T, k, R, max_tokens, _ptr(combined_w),
                                  _ptr(status), _stream(stream))
    _done("ep_combine_weights", rc)


# --------------------------------------------------------------------------- expert-major path

def ep_expert_layout_workspace_size(T: int, E: int) -> int:
    return int(lib().ep_expert_layout_workspace_size(T, E))


def ep_get_expert_layout(topk_idx, num_experts, expert_offsets, expert_slot, workspace, status=None, stream=None):
    T, k = topk_idx.shape
    E = num_experts
    _check("topk_idx", topk_idx, torch.int64)
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("workspace", workspace, torch.uint8)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_get_expert_layout(_ptr(topk_idx), T, k, E, _ptr(expert_offsets), _ptr(expert_slot),
                                    _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _done("ep_get_expert_layout", rc)


def ep_dispatch_permuted(x, topk_idx, topk_w, expert_offsets, expert_slot, num_experts, num_ranks, max_rows, perm_x,
                         perm_src=None, perm_w=None, status=None, stream=None):
    T, H = x.shape
    k = topk_idx.shape[1]
    E, R = num_experts, num_ranks
    _check("x", x, torch.bfloat16)
    _check("topk_idx", topk_idx, torch.int64, (T, k))
    _check("topk_w", topk_w, torch.float32, (T, k), optional=True)
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("perm_x", perm_x, torch.bfloat16, (R, max_rows, H))
    _check("perm_src", perm_src, torch.int32, (R, max_rows), optional=True)
    _check("perm_w", perm_w, torch.float32, (R, max_rows), optional=True)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_dispatch_permuted(_ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offsets), _ptr(expert_slot),
                                    T, H, k, E, R, max_rows, _ptr(perm_x), _ptr(perm_src), _ptr(perm_w),
                                    _ptr(status), _stream(stream))
    _done("ep_dispatch_permuted", rc)


def ep_permute_received(recv_x, recv_src_idx, recv_topk_idx, recv_topk_w, tokens_per_rank, expert_offsets,
                        expert_slot, num_experts, max_rows, perm_x, perm_src=None, perm_w=None, status=None,
                        stream=None):
    R, M, H = recv_x.shape
    k = recv_topk_idx.shape[2]
    T = expert_slot.shape[0]
    E = num_experts
    _check("recv_x", recv_x, torch.bfloat16)
    _check("recv_src_idx", recv_src_idx, torch.int32, (R, M))
    _check("recv_topk_idx", recv_topk_idx, torch.int32, (R, M, k))
    _check("recv_topk_w", recv_topk_w, torch.float32, (R, M, k), optional=True)
    _check("tokens_per_rank", tokens_per_rank, torch.int32, (R,))
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("perm_x", perm_x, torch.bfloat16, (R, max_rows, H))
    _check("perm_src", perm_src, torch.int32, (R, max_rows), optional=True)
    _check("perm_w", perm_w, torch.float32, (R, max_rows), optional=True)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_permute_received(_ptr(recv_x), _ptr(recv_src_idx), _ptr(recv_topk_idx), _ptr(recv_topk_w),
                                   _ptr(tokens_per_rank), _ptr(expert_offsets), _ptr(expert_slot), T, H, k, E, R, M,
                                   max_rows, _ptr(perm_x), _ptr(perm_src), _ptr(perm_w), _ptr(status),
                                   _stream(stream))
    _done("ep_permute_received", rc)


def ep_combine_permuted(y, topk_idx, topk_w, expert_offsets, expert_slot, num_experts, out, status=None, stream=None):
    R, max_rows, H = y.shape
    T, k = topk_idx.shape
    E = num_experts
    _check("y", y, torch.bfloat16)
    _check("topk_idx", topk_idx, torch.int64, (T, k))
    _check("topk_w", topk_w, torch.float32, (T, k), optional=True)
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("out", out, torch.bfloat16, (T, H))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine_permuted(_ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offsets), _ptr(expert_slot),
                                   T, H, k, E, R, max_rows, _ptr(out), _ptr(status), _stream(stream))
    _done("ep_combine_permuted", rc)


def ep_dispatch_permuted_ll(x, topk_idx, topk_w, num_experts, num_ranks, max_rows, expert_offsets, expert_slot, perm_x,
                            perm_src=None, perm_w=None, status=None, stream=None):
    T, H = x.shape
    k = topk_idx.shape[1]
    E, R = num_experts, num_ranks
    _check("x", x, torch.bfloat16, (T, H))
    _check("topk_idx", topk_idx, torch.int64, (T, k))
    _check("topk_w", topk_w, torch.float32, (T, k), optional=True)
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("perm_x", perm_x, torch.bfloat16, (R, max_rows, H))
    _check("perm_src", perm_src, torch.int32, (R, max_rows), optional=True)
    _check("perm_w", perm_w, torch.float32, (R, max_rows), optional=True)
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_dispatch_permuted_ll(_ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, E, R, max_rows,
                                       _ptr(expert_offsets), _ptr(expert_slot), _ptr(perm_x), _ptr(perm_src),
                                       _ptr(perm_w), _ptr(status), _stream(stream))
    _done("ep_dispatch_permuted_ll", rc)



def ep_combine_permuted_ll(y, topk_idx, topk_w, expert_offsets, expert_slot, num_experts, out, status=None,
                           stream=None):
    """ep_combine_permuted for a decode-sized batch (T <= 1024), shaped for latency; same results."""
    R, max_rows, H = y.shape
    T, k = topk_idx.shape
    E = num_experts
    _check("y", y, torch.bfloat16)
    _check("topk_idx", topk_idx, torch.int64, (T, k))
    _check("topk_w", topk_w, torch.float32, (T, k), optional=True)
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("out", out, torch.bfloat16, (T, H))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine_permuted_ll(_ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_offsets), _ptr(expert_slot),
                                      T, H, k, E, R, max_rows, _ptr(out), _ptr(status), _stream(stream))
    _done("ep_combine_permuted_ll", rc)


def ep_combine_send(y_perm, recv_src_idx, recv_topk_idx, recv_topk_w, tokens_per_rank, expert_offsets, expert_slot,
                    num_experts, y_rank, status=None, stream=None):
    """Send phase of a split combine: expert-major rows reduced back into the rank-level slabs
    y_rank [R][max_tokens][H], which ep_combine (the receive phase) reads. recv_topk_w None:
    unweighted."""
    R, max_rows, H = y_perm.shape
    M = recv_src_idx.shape[1]
    k = recv_topk_idx.shape[2]
    T = expert_slot.shape[0]
    E = num_experts
    _check("y_perm", y_perm, torch.bfloat16)
    _check("recv_src_idx", recv_src_idx, torch.int32, (R, M))
    _check("recv_topk_idx", recv_topk_idx, torch.int32, (R, M, k))
    _check("recv_topk_w", recv_topk_w, torch.float32, (R, M, k), optional=True)
    _check("tokens_per_rank", tokens_per_rank, torch.int32, (R,))
    _check("expert_offsets", expert_offsets, torch.int32, (E + 1,))
    _check("expert_slot", expert_slot, torch.int32, (T, k))
    _check("y_rank", y_rank, torch.bfloat16, (R, M, H))
    _check("status", status, torch.int32, (1,), optional=True)
    rc = lib().ep_combine_send(_ptr(y_perm), _ptr(recv_src_idx), _ptr(recv_topk_idx), _ptr(recv_topk_w),
                               _ptr(tokens_per_rank), _ptr(expert_offsets), _ptr(expert_slot), T, H, k, E, R, M,
                               max_rows, _ptr(y_rank), _ptr(status), _stream(stream))
    _done("ep_combine_send", rc)
