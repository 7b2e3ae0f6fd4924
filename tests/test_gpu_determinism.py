"""Determinism: every output of the path is the same, byte for byte, when a call is
repeated on the same inputs -- with the same buffers and workspaces reused and with fresh
ones. (Stable slots and a fixed reduction order are what make this hold; the parity tests
check the values, this checks that nothing depends on scheduling.)"""
import numpy as np
import pytest
import torch

import combine_ep_get_05_gb300 as ep
import workloads
from gpu_helpers import dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.build_library()
    ep.lib()


def _rank_path(w, fp8, lay=None, d=None):
    topk = torch.from_numpy(w.topk_idx).cuda()
    x = dev_bf16(w.x)
    tw = torch.from_numpy(w.topk_w).cuda()
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
    M = int(lay.tokens_per_rank.max().item())
    d = ep.dispatch(x, topk, tw, lay, M, fp8=fp8, out=d if d is not None and d.max_tokens == M else None)
    counts = host_bits(lay.tokens_per_rank)
    got = {k: host_bits(getattr(lay, k)) for k in ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "slot")}
    for k in ("recv_x", "recv_src_idx", "recv_topk_idx", "recv_topk_w") + (("recv_scales",) if fp8 else ()):
        v = host_bits(getattr(d, k))
        got[k] = np.concatenate([v[r, :counts[r]].reshape(-1).view(np.uint8) for r in range(w.R)])
    if fp8:
        got["out"] = host_bits(ep.combine_fp8(d.recv_x, d.recv_scales, lay, M))
    else:
        got["out"] = host_bits(ep.combine(d.recv_x, lay, M))
    got["combined_w"] = host_bits(ep.combine_weights(d.recv_topk_w, lay, M))
    return got, lay, d


@pytest.mark.parametrize("name,fp8", [("dsv3", False), ("dsv3_fp8", True), ("skewed", False)])
def test_rank_path_repeats_byte_for_byte(name, fp8):
    w = workloads.make(name, T=3000, H=1024)
    first, lay, d = _rank_path(w, fp8)
    again, _, _ = _rank_path(w, fp8, lay, d)    # the same buffers and workspace
    fresh, _, _ = _rank_path(w, fp8)            # new buffers and workspace
    for k in first:
        assert np.array_equal(first[k], again[k]), k
        assert np.array_equal(first[k], fresh[k]), k


def test_expert_major_path_repeats_byte_for_byte():
    w = workloads.make("dsv3", T=700, H=512)
    topk = torch.from_numpy(w.topk_idx).cuda()
    x = dev_bf16(w.x)
    tw = torch.from_numpy(w.topk_w).cuda()
    E, R, T, k = w.E, w.R, w.T, w.k
    ws = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device="cuda")
    results = []
    for ll in (False, False, True, True):
        off = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
        slot = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        M = T * k
        px = torch.zeros((R, M // R + T, w.H), dtype=torch.bfloat16, device="cuda")
        ps = torch.zeros(px.shape[:2], dtype=torch.int32, device="cuda")
        pw = torch.zeros(px.shape[:2], dtype=torch.float32, device="cuda")
        if ll:
            ep.ep_dispatch_permuted_ll(x, topk, tw, E, R, px.shape[1], off, slot, px, ps, pw)
        else:
            ep.ep_get_expert_layout(topk, E, off, slot, ws)
            ep.ep_dispatch_permuted(x, topk, tw, off, slot, E, R, px.shape[1], px, ps, pw)
        out = torch.empty((T, w.H), dtype=torch.bfloat16, device="cuda")
        ep.ep_combine_permuted(px, topk, tw, off, slot, E, out)
        results.append([host_bits(t) for t in (off, slot, px, ps, pw, out)])
    for r in results[1:]:
        for a, b in zip(results[0], r):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
