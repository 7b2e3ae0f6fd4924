"""ep_get_layout_noalloc: the layout for callers that cannot allocate a workspace.

Some callers of this library cannot allocate device memory where they need the
routing layout (a fixed, pre-planned memory budget without an allocator of its
own, or a host runtime that can only pass pointers to arrays it already owns).
ep_get_layout_noalloc serves them from a fixed array inside the library. The
array keeps whatever the previous call left in it; every call zero-fills the
part it uses before its kernel runs.

These tests call it through the C ABI several times in a row, with different
sizes (a large batch, then smaller ones whose regions of the array overlap the
first), and check every output bit for bit against ep_get_layout with its own
workspace, and for one case directly against the oracle; one case has no node
split (ranks_per_node = 0). They also check that sizes beyond the fixed array
are refused before anything is launched.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test. It passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_ep_get_05_gb300 as ep
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _buffers(T, E, R, rpn):
    N = R // rpn if rpn else 0
    i32 = dict(dtype=torch.int32, device="cuda")
    return {
        "tpe": torch.full((E,), -1, **i32),
        "tpr": torch.full((R,), -1, **i32),
        "tpn": torch.full((N,), -1, **i32) if N else None,
        "in_rank": torch.full((T, R), 7, dtype=torch.uint8, device="cuda"),
        "in_node": torch.full((T, N), 7, dtype=torch.uint8, device="cuda") if N else None,
        "slot": torch.full((T, R), -9, **i32),
        "status": torch.zeros(1, **i32),
    }


def _call_noalloc(L, topk, E, R, rpn, b, stream):
    T, k = topk.shape
    return L.ep_get_layout_noalloc(_p(topk), T, k, E, R, rpn, _p(b["tpe"]), _p(b["tpr"]), _p(b["tpn"]),
                                   _p(b["in_rank"]), _p(b["in_node"]), _p(b["slot"]), _p(b["status"]), stream)


def _call_workspace(L, topk, E, R, rpn, b, stream):
    T, k = topk.shape
    ws_bytes = L.ep_layout_workspace_size(T, E, R, rpn)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    rc = L.ep_get_layout(_p(topk), T, k, E, R, rpn, _p(b["tpe"]), _p(b["tpr"]), _p(b["tpn"]), _p(b["in_rank"]),
                         _p(b["in_node"]), _p(b["slot"]), _p(ws), ws_bytes, _p(b["status"]), stream)
    return rc, ws


def test_noalloc_layout_matches_the_workspace_layout_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.build_library()
    L = ep.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    no_nodes = workloads.make("tiny", T=1500, H=8, E=64, k=6, R=16, ranks_per_node=0)
    cases = [workloads.make("dsv3", T=4096, H=8), workloads.make("skewed", T=3001, H=8), no_nodes]
    for w in cases:  # calls in a row, different T, E, R and node counts
        topk = torch.from_numpy(w.topk_idx).cuda()
        got = _buffers(w.T, w.E, w.R, w.ranks_per_node)
        ref = _buffers(w.T, w.E, w.R, w.ranks_per_node)
        assert _call_noalloc(L, topk, w.E, w.R, w.ranks_per_node, got, stream) == ep.EP_OK
        rc, ws = _call_workspace(L, topk, w.E, w.R, w.ranks_per_node, ref, stream)
        assert rc == ep.EP_OK
        torch.cuda.synchronize()
        for key in got:
            if got[key] is None:
                continue
            assert torch.equal(got[key], ref[key]), (w.name, key)
        assert int(got["status"].item()) == 0
        assert int(got["tpr"].sum().item()) == int(got["in_rank"].sum().item())
    # the last case (no node split) straight against the oracle as well
    O = oracle.layout(no_nodes.topk_idx, no_nodes.E, no_nodes.R, 0)
    for key, name in (("tpe", "tokens_per_expert"), ("tpr", "tokens_per_rank"), ("in_rank", "is_token_in_rank"),
                      ("slot", "slot")):
        assert np.array_equal(got[key].cpu().numpy(), O[name]), name


def test_noalloc_refuses_sizes_beyond_its_scratch():
    ep.build_library()
    L = ep.lib()
    T, E, R = 200_000, 256, 256  # 782 tiles x 256 ranks x 8 bytes of tile words > 1 MiB
    assert L.ep_layout_workspace_size(T, E, R, 0) > ep.LAYOUT_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    rc = L.ep_get_layout_noalloc(fake, T, 8, E, R, 0, fake, fake, None, fake, None, fake, None, None)
    assert rc == ep.EP_ERR_SCRATCH
    assert b"EP_ERR_SCRATCH" in L.ep_status_str(rc)

