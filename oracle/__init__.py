"""The oracle: a plain single-threaded C statement of the EP dispatch/combine path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The CUDA
library (``combine_ep_get_05_gb300``) never imports it, and it never imports
the CUDA library.

Each wrapper below marshals numpy arrays into the C routine of the same name in
``ep_oracle.c``; all arithmetic happens there. bf16 arrays are ``np.uint16``
bit patterns, e4m3 arrays are ``np.uint8`` codes.

Parity is pinned (tests/test_oracle_*.py) by brute force on tiny inputs,
closed forms (identity-expert combine, restripe inverse), invariants (count
sums, stable slot order, exactly-once delivery) and library routines
(torch's CPU float8_e4m3fn / bfloat16 conversions, a nearest-value search
over all 256 e4m3 codes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_HDR = os.path.join(_HERE, "ep_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libep_oracle.so")

FLAG_CAPACITY = 1
FLAG_BAD_EXPERT = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into a shared library (plain gcc, -ffp-contract=off)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, _HDR)
    )
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            sig = {
                "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_f32_to_e4m3": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_e4m3_to_f32": (ctypes.c_float, [ctypes.c_uint8]),
                "oracle_quantize_row_e4m3": (None, [P, i32, P, P]),
                "oracle_layout": (i32, [P, i32, i32, i32, i32, i32, P, P, P, P, P, P]),
                "oracle_dispatch": (i32, [P, i32, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P]),
                "oracle_restripe_prob": (None, [P, i32, i32, i32, i32, P]),
                "oracle_dispatch_nodes": (i32, [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P]),
                "oracle_combine": (i32, [P, P, i32, i32, i32, i32, P]),
                "oracle_combine_fp8": (i32, [P, P, P, i32, i32, i32, i32, P]),
                "oracle_combine_weights": (i32, [P, P, i32, i32, i32, i32, P]),
                "oracle_expert_scale": (None, [P, i32, P, P, P, i32, i32, i32, i32, P]),
                "oracle_expert_layout": (i32, [P, i32, i32, i32, P, P]),
                "oracle_dispatch_permuted": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]),
                "oracle_permute_received": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P]),
                "oracle_combine_permuted": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]),
                "oracle_combine_send": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- #
# number formats
# --------------------------------------------------------------------------- #

def f32_to_bf16(v: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(v)))


def bf16_to_f32(b: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(b)))


def f32_to_e4m3(v: float) -> int:
    return int(_load().oracle_f32_to_e4m3(float(v)))


def e4m3_to_f32(q: int) -> float:
    return float(_load().oracle_e4m3_to_f32(int(q)))


def quantize_row_e4m3(x_bits: np.ndarray):
    """x_bits: uint16 [H] (H % 128 == 0) -> (uint8 [H] codes, float32 [H/128] scales)."""
    x = _c(x_bits, np.uint16)
    H = x.shape[-1]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.float32)
    _load().oracle_quantize_row_e4m3(_ptr(x), H, _ptr(q), _ptr(s))
    return q, s


# --------------------------------------------------------------------------- #
# the path
# --------------------------------------------------------------------------- #

def layout(topk_idx: np.ndarray, E: int, R: int, ranks_per_node: int = 0) -> dict:
    ti = _c(topk_idx, np.int64)
    T, k = ti.shape
    N = R // ranks_per_node if ranks_per_node > 0 else 0
    out = {
        "tokens_per_expert": np.zeros(E, np.int32),
        "tokens_per_rank": np.zeros(R, np.int32),
        "tokens_per_node": np.zeros(N, np.int32),
        "is_token_in_rank": np.zeros((T, R), np.uint8),
        "is_token_in_node": np.zeros((T, N), np.uint8),
        "slot": np.zeros((T, R), np.int32),
    }
    out["flags"] = int(_load().oracle_layout(
        _ptr(ti), T, k, E, R, ranks_per_node, _ptr(out["tokens_per_expert"]),
        _ptr(out["tokens_per_rank"]), _ptr(out["tokens_per_node"]) if N else None,
        _ptr(out["is_token_in_rank"]), _ptr(out["is_token_in_node"]) if N else None,
        _ptr(out["slot"])))
    return out


def dispatch(x_bits, topk_idx, topk_w, slot, E: int, R: int, max_tokens: int, fp8: bool = False,
             rows: bool = True, fill_x: int = 0, fill_idx: int = 0, fill_w: float = 0.0) -> dict:
    """Rank-level dispatch. Unreceived rows keep the fill values. rows=False skips the payload."""
    x = _c(x_bits, np.uint16)
    ti = _c(topk_idx, np.int64)
    tw = _c(topk_w, np.float32)
    sl = _c(slot, np.int32)
    T, H = x.shape
    k = ti.shape[1]
    out = {
        "recv_src_idx": np.full((R, max_tokens), fill_idx, np.int32),
        "recv_topk_idx": np.full((R, max_tokens, k), fill_idx, np.int32),
        "recv_topk_w": np.full((R, max_tokens, k), fill_w, np.float32),
        "recv_x": None,
        "recv_scales": None,
    }
    if rows:
        if fp8:
            out["recv_x"] = np.full((R, max_tokens, H), fill_x & 0xFF, np.uint8)
            out["recv_scales"] = np.full((R, max_tokens, H // 128), fill_w, np.float32)
        else:
            out["recv_x"] = np.full((R, max_tokens, H), fill_x, np.uint16)
    out["flags"] = int(_load().oracle_dispatch(
        _ptr(x), 1 if fp8 else 0, _ptr(ti), _ptr(tw), _ptr(sl), T, H, k, E, R, max_tokens,
        _ptr(out["recv_x"]), _ptr(out["recv_scales"]), _ptr(out["recv_src_idx"]),
        _ptr(out["recv_topk_idx"]), _ptr(out["recv_topk_w"])))
    return out


def restripe_prob(prob: np.ndarray, max_tokens: int, fill: float = 0.0) -> np.ndarray:
    p = _c(prob, np.float32)
    T, N, P = p.shape
    out = np.full((N, max_tokens, P), fill, np.float32)
    _load().oracle_restripe_prob(_ptr(p), T, N, P, max_tokens, _ptr(out))
    return out


def dispatch_nodes(x_bits, prob_staging, is_token_in_node, max_tokens: int, chunk_tokens: int = 256,
                   dense: bool = False, fill_x: int = 0, fill_prob: float = 0.0) -> dict:
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    inn = _c(is_token_in_node, np.uint8)
    N = inn.shape[1]
    ps = None if prob_staging is None else _c(prob_staging, np.float32)
    P = 0 if ps is None else ps.shape[2]
    nchunks = (T + chunk_tokens - 1) // chunk_tokens
    out = {
        "recv_x_node": np.full((N, max_tokens, H), fill_x, np.uint16),
        "recv_prob_node": None if ps is None else np.full((N, max_tokens, P), fill_prob, np.float32),
        "num_runs": np.zeros((N, nchunks), np.int32),
    }
    rc = int(_load().oracle_dispatch_nodes(
        _ptr(x), _ptr(ps), _ptr(inn), T, H, N, P, max_tokens, chunk_tokens, 0 if dense else 1,
        _ptr(out["recv_x_node"]), _ptr(out["recv_prob_node"]), _ptr(out["num_runs"])))
    if rc != 0:
        raise ValueError("oracle_dispatch_nodes: T > max_tokens or chunk_tokens <= 0")
    return out


def combine(y_bits, slot, max_tokens: int) -> tuple:
    y = _c(y_bits, np.uint16)
    sl = _c(slot, np.int32)
    R, _, H = y.shape
    T = sl.shape[0]
    out = np.zeros((T, H), np.uint16)
    flags = int(_load().oracle_combine(_ptr(y), _ptr(sl), T, H, R, max_tokens, _ptr(out)))
    return out, flags


def combine_fp8(y_codes, y_scales, slot, max_tokens: int) -> tuple:
    """Combine of FP8 rows: each row dequantised to fp32(e4m3(q) * scale), then as combine()."""
    y = _c(y_codes, np.uint8)
    sc = _c(y_scales, np.float32)
    sl = _c(slot, np.int32)
    R, _, H = y.shape
    T = sl.shape[0]
    out = np.zeros((T, H), np.uint16)
    flags = int(_load().oracle_combine_fp8(_ptr(y), _ptr(sc), _ptr(sl), T, H, R, max_tokens, _ptr(out)))
    return out, flags


def combine_weights(recv_topk_w, slot, max_tokens: int) -> tuple:
    """Combined top-k weights [T][k]: fp32 sum over ranks ascending of the received weight rows."""
    w = _c(recv_topk_w, np.float32)
    sl = _c(slot, np.int32)
    R, _, k = w.shape
    T = sl.shape[0]
    out = np.zeros((T, k), np.float32)
    flags = int(_load().oracle_combine_weights(_ptr(w), _ptr(sl), T, k, R, max_tokens, _ptr(out)))
    return out, flags


def expert_scale(recv_x, recv_topk_w, tokens_per_rank, recv_scales=None, fill: int = 0) -> np.ndarray:
    """The harness expert: y = bf16(row * sum_j w_j) on every received row (others = fill)."""
    fp8 = recv_x.dtype == np.uint8
    rx = _c(recv_x, np.uint8 if fp8 else np.uint16)
    R, max_tokens, H = rx.shape
    tw = _c(recv_topk_w, np.float32)
    k = tw.shape[2]
    tpr = _c(tokens_per_rank, np.int32)
    sc = None if recv_scales is None else _c(recv_scales, np.float32)
    y = np.full((R, max_tokens, H), fill, np.uint16)
    _load().oracle_expert_scale(_ptr(rx), 1 if fp8 else 0, _ptr(sc), _ptr(tw), _ptr(tpr), R,
                                max_tokens, H, k, _ptr(y))
    return y


# --------------------------------------------------------------------------- expert-major

def expert_layout(topk_idx, E: int) -> dict:
    ti = _c(topk_idx, np.int64)
    T, k = ti.shape
    out = {"expert_offsets": np.zeros(E + 1, np.int32), "expert_slot": np.zeros((T, k), np.int32)}
    out["flags"] = int(_load().oracle_expert_layout(_ptr(ti), T, k, E, _ptr(out["expert_offsets"]),
                                                   _ptr(out["expert_slot"])))
    return out


def rows_per_rank(expert_offsets, E: int, R: int) -> np.ndarray:
    """Entries each rank's expert-major slab holds (plain indexing of the offsets)."""
    epr = E // R
    off = np.asarray(expert_offsets)
    return (off[np.arange(1, R + 1) * epr] - off[np.arange(R) * epr]).astype(np.int32)


def dispatch_permuted(x_bits, topk_idx, topk_w, EL: dict, E: int, R: int, max_rows: int, fill_x: int = 0,
                      fill_idx: int = 0, fill_w: float = 0.0) -> dict:
    x = _c(x_bits, np.uint16)
    ti = _c(topk_idx, np.int64)
    tw = _c(topk_w, np.float32)
    T, H = x.shape
    k = ti.shape[1]
    out = {"perm_x": np.full((R, max_rows, H), fill_x, np.uint16),
           "perm_src": np.full((R, max_rows), fill_idx, np.int32),
           "perm_w": np.full((R, max_rows), fill_w, np.float32)}
    out["flags"] = int(_load().oracle_dispatch_permuted(
        _ptr(x), _ptr(ti), _ptr(tw), _ptr(_c(EL["expert_offsets"], np.int32)), _ptr(_c(EL["expert_slot"], np.int32)),
        T, H, k, E, R, max_rows, _ptr(out["perm_x"]), _ptr(out["perm_src"]), _ptr(out["perm_w"])))
    return out


def permute_received(D: dict, tokens_per_rank, EL: dict, T: int, E: int, R: int, max_rows: int, fill_x: int = 0,
                     fill_idx: int = 0, fill_w: float = 0.0) -> dict:
    rx = _c(D["recv_x"], np.uint16)
    R_, M, H = rx.shape
    k = D["recv_topk_idx"].shape[2]
    out = {"perm_x": np.full((R, max_rows, H), fill_x, np.uint16),
           "perm_src": np.full((R, max_rows), fill_idx, np.int32),
           "perm_w": np.full((R, max_rows), fill_w, np.float32)}
    out["flags"] = int(_load().oracle_permute_received(
        _ptr(rx), _ptr(_c(D["recv_src_idx"], np.int32)), _ptr(_c(D["recv_topk_idx"], np.int32)),
        _ptr(_c(D["recv_topk_w"], np.float32)), _ptr(_c(tokens_per_rank, np.int32)),
        _ptr(_c(EL["expert_offsets"], np.int32)), _ptr(_c(EL["expert_slot"], np.int32)), T, H, k, E, R, M,
        max_rows, _ptr(out["perm_x"]), _ptr(out["perm_src"]), _ptr(out["perm_w"])))
    return out


def combine_permuted(y_bits, topk_idx, topk_w, EL: dict, E: int, R: int) -> tuple:
    y = _c(y_bits, np.uint16)
    ti = _c(topk_idx, np.int64)
    tw = None if topk_w is None else _c(topk_w, np.float32)
    _, max_rows, H = y.shape
    T, k = ti.shape
    out = np.zeros((T, H), np.uint16)
    flags = int(_load().oracle_combine_permuted(
        _ptr(y), _ptr(ti), _ptr(tw), _ptr(_c(EL["expert_offsets"], np.int32)), _ptr(_c(EL["expert_slot"], np.int32)),
        T, H, k, E, R, max_rows, _ptr(out)))
    return out, flags


def combine_send(y_perm, D: dict, tokens_per_rank, EL: dict, T: int, E: int, R: int, weighted: bool = True,
                 fill: int = 0) -> tuple:
    """Send phase of a split combine: per rank and received row, the local experts' expert-major
    rows reduced (weighted by the received top-k weights, or not) into one bf16 rank-level row.
    Returns (y_rank [R][max_tokens][H] with unwritten rows at `fill`, flags)."""
    yp = _c(y_perm, np.uint16)
    _, max_rows, H = yp.shape
    src = _c(D["recv_src_idx"], np.int32)
    R_, M = src.shape
    k = D["recv_topk_idx"].shape[2]
    tw = _c(D["recv_topk_w"], np.float32) if weighted else None
    out = np.full((R, M, H), fill, np.uint16)
    flags = int(_load().oracle_combine_send(
        _ptr(yp), _ptr(src), _ptr(_c(D["recv_topk_idx"], np.int32)), _ptr(tw), _ptr(_c(tokens_per_rank, np.int32)),
        _ptr(_c(EL["expert_offsets"], np.int32)), _ptr(_c(EL["expert_slot"], np.int32)), T, H, k, E, R, M, max_rows,
        _ptr(out)))
    return out, flags
