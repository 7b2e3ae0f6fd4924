"""GPU parity: the CUDA library against the oracle, element by element, on the
same seeded inputs (workloads.py). Layout, dispatch (bf16 and E4M3), restripe
and node dispatch must be bit-exact; combine sums in ascending rank order, so
it must be bit-exact too. Every output buffer sits between guard regions that
must be unchanged afterwards, and rows a rank does not receive must keep their
sentinel.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_05_gb300 as ep
import oracle
import workloads
from gpu_helpers import (SENT_BF16, SENT_F32, SENT_I32, check_guards, dev_bf16, gpu_expert, gpu_layout, guarded,
                         host_bits, layout_to_host, oracle_expert)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.build_library()
    ep.lib()


def _max_tokens(w, L):
    return w.max_tokens if w.max_tokens is not None else max(1, int(L["tokens_per_rank"].max()))


def _assert_layout(w, lay, L):
    got = layout_to_host(lay)
    for key, v in got.items():
        assert np.array_equal(v, L[key]), key
    assert ep.read_flags(lay.status) == L["flags"]


def run_rank_path(w, max_tokens=None, full_compare=True):
    """Layout -> dispatch -> harness expert -> combine on both sides; compare everything."""
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    M = max_tokens if max_tokens is not None else _max_tokens(w, L)
    topk, lay = gpu_layout(w)
    _assert_layout(w, lay, L)

    x = dev_bf16(w.x)
    tw = torch.from_numpy(w.topk_w).cuda()
    H, R, k, fp8 = w.H, w.R, w.k, w.fp8
    fill_x = 0xAB if fp8 else SENT_BF16
    recv_x, bx = guarded((R, M, H), torch.uint8 if fp8 else torch.bfloat16, fill_x)
    recv_scales, bs = guarded((R, M, H // 128), torch.float32, SENT_F32) if fp8 else (None, None)
    src, bsrc = guarded((R, M), torch.int32, SENT_I32)
    tidx, btidx = guarded((R, M, k), torch.int32, SENT_I32)
    tww, btw = guarded((R, M, k), torch.float32, SENT_F32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(x, ep.DTYPE_E4M3 if fp8 else ep.DTYPE_BF16, topk, tw, lay.slot, w.E, R, M, recv_x, recv_scales,
                   src, tidx, tww, status)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, R, M, fp8=fp8, rows=full_compare,
                        fill_x=fill_x, fill_idx=SENT_I32, fill_w=SENT_F32)
    assert ep.read_flags(status) == D["flags"]
    assert np.array_equal(host_bits(src), D["recv_src_idx"])
    assert np.array_equal(host_bits(tidx), D["recv_topk_idx"])
    assert np.array_equal(host_bits(tww).view(np.uint32), D["recv_topk_w"].view(np.uint32))
    guards = [(bx, recv_x, fill_x), (bsrc, src, SENT_I32), (btidx, tidx, SENT_I32), (btw, tww, SENT_F32)]
    if fp8:
        guards.append((bs, recv_scales, SENT_F32))
    for backing, view, fill in guards:
        check_guards(backing, view.numel(), fill)
    if full_compare:
        assert np.array_equal(host_bits(recv_x), D["recv_x"])
        if fp8:
            assert np.array_equal(host_bits(recv_scales).view(np.uint32), D["recv_scales"].view(np.uint32))

    # harness expert on each side, then combine
    y = recv_x if (w.expert == "identity" and not fp8) else gpu_expert(recv_x, tww, recv_scales)
    out, bout = guarded((w.T, H), torch.bfloat16, SENT_BF16)
    cstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine(y, lay.slot, M, out, cstatus)
    torch.cuda.synchronize()
    check_guards(bout, out.numel(), SENT_BF16)
    if full_compare:
        Y = oracle_expert(w, D, L)
        received = np.arange(M)[None, :] < np.minimum(L["tokens_per_rank"], M)[:, None]  # [R][M]
        assert np.array_equal(host_bits(y)[received], Y[received])
        ref, cflags = oracle.combine(Y, L["slot"], M)
        assert ep.read_flags(cstatus) == cflags
        assert np.array_equal(host_bits(out), ref)
    return L, host_bits(out)


# ----------------------------------------------------------------------------- whole path

@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("tiny", {"T": 1}),
    ("tiny", {"T": 257, "H": 8}),
    ("dsv3", {"T": 1000, "H": 1024}),
    ("dsv3", {"T": 777, "H": 7168}),
    ("dsv3_fp8", {"T": 1000, "H": 1024}),
    ("dsv3_fp8", {"T": 333, "H": 384}),
    ("dsv3_fp8", {"T": 300, "H": 24576}),  # wide FP8 rows
    ("dsv3_fp8", {"T": 40, "H": 26624}),
    ("dsv3_fp8", {"T": 30, "H": 33024}),   # more than 256 blocks: scales stored per iteration
    # the shared-memory FP8 kernel (H % 512 == 0) with fewer tokens than CTAs: one CTA with
    # one token, a few CTAs with one token each, CTAs with one or two tokens
    ("dsv3_fp8", {"T": 1, "H": 512}),
    ("dsv3_fp8", {"T": 5, "H": 7168}),
    ("dsv3_fp8", {"T": 700, "H": 2048}),
    ("dsv3", {"T": 40, "H": 36864}),       # bf16 rows too large for the bulk-copy scatter
    ("skewed", {"T": 2000, "H": 256}),
    ("restripe", {"T": 700, "H": 512}),
])
def test_rank_path_matches_oracle(name, over):
    run_rank_path(workloads.make(name, **over))


@pytest.mark.parametrize("name", ["tiny", "dsv3", "dsv3_fp8"])
def test_rank_path_full_size(name):
    """The full workloads, as the benchmark launches them, compared in full."""
    run_rank_path(workloads.make(name))


def test_capacity_overflow_drops_and_flags():
    w = workloads.make("skewed", T=3000, H=128)
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    run_rank_path(w, max_tokens=int(L["tokens_per_rank"].max()) // 2)


def test_bad_expert_ids_are_skipped_and_flagged():
    w = workloads.make("tiny", T=200)
    w.topk_idx[5, 1] = w.E + 3
    w.topk_idx[77, 0] = 10 ** 9
    w.topk_idx[100, :] = -1  # routed nowhere: combine gives +0
    run_rank_path(w)


def test_duplicate_experts_on_one_rank_and_all_to_one_rank():
    w = workloads.make("tiny", T=300, H=64)
    w.topk_idx[:] = np.array([0, 1, 2, 3], np.int64)  # every token: four experts, all on rank 0
    run_rank_path(w)


@pytest.mark.parametrize("R,E,k", [(1, 8, 3), (256, 256, 8), (64, 8192, 32), (7, 21, 2)])
def test_rank_path_extreme_shapes(R, E, k):
    rng = np.random.Generator(np.random.PCG64(R * 1000 + k))
    T, H = 300, 64
    w = workloads.make("tiny", T=T, H=H, E=E, k=k, R=R, ranks_per_node=R)
    w.topk_idx = workloads.routing_uniform(rng, T, E, k)
    w.topk_w = rng.random((T, k), dtype=np.float32)
    w.expert = "scale"
    run_rank_path(w)


def test_full_size_skewed_in_full():
    """T=16384, H=4096, R=64, max_tokens sized to the hottest rank (15638): the element
    offsets of the receive slab pass 2^31. The metadata, every received row of every rank
    (rank by rank: the slab is 8 GB) and every combined token (in sub-batches of 512 tokens,
    each run through the oracle's own layout, dispatch, expert and combine) are compared."""
    w = workloads.make("skewed")
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    M = _max_tokens(w, L)
    assert w.R * M * w.H > 2 ** 31
    topk, lay = gpu_layout(w)
    _assert_layout(w, lay, L)
    x = dev_bf16(w.x)
    tw = torch.from_numpy(w.topk_w).cuda()
    d = ep.alloc_dispatch(w.R, M, w.H, w.k)
    ep.dispatch(x, topk, tw, lay, M, out=d)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, M, rows=False, fill_idx=SENT_I32,
                        fill_w=SENT_F32)
    cnt = np.minimum(L["tokens_per_rank"], M)
    valid = np.arange(M)[None, :] < cnt[:, None]
    assert np.array_equal(host_bits(d.recv_src_idx)[valid], D["recv_src_idx"][valid])
    assert np.array_equal(host_bits(d.recv_topk_idx)[valid], D["recv_topk_idx"][valid])
    assert np.array_equal(host_bits(d.recv_topk_w)[valid], D["recv_topk_w"][valid])
    for r in range(w.R):  # recv_x[r][s] = x[recv_src_idx[r][s]] for every received row
        n = int(cnt[r])
        assert np.array_equal(host_bits(d.recv_x[r, :n]), w.x[D["recv_src_idx"][r, :n]]), r
    # harness expert rank by rank (keeps the fp32 temporaries small), then combine
    y = torch.empty_like(d.recv_x)
    for r in range(w.R):
        y[r:r + 1] = gpu_expert(d.recv_x[r:r + 1], d.recv_topk_w[r:r + 1])
    out = host_bits(ep.combine(y, lay, M))
    del y, d
    for b0 in range(0, w.T, 512):
        tok = np.arange(b0, min(w.T, b0 + 512))
        Ls = oracle.layout(w.topk_idx[tok], w.E, w.R)
        Ds = oracle.dispatch(w.x[tok], w.topk_idx[tok], w.topk_w[tok], Ls["slot"], w.E, w.R, len(tok))
        Ys = oracle.expert_scale(Ds["recv_x"], Ds["recv_topk_w"], Ls["tokens_per_rank"])
        ref, _ = oracle.combine(Ys, Ls["slot"], len(tok))
        assert np.array_equal(out[tok], ref), b0
    assert ep.read_flags(lay.status) == 0


def _tiled_routing(name, copies, seed=7, **over):
    """A large batch made of `copies` copies of a seeded routing, each copy with its experts
    renamed by its own random permutation (so rows stay distinct and copies differ)."""
    w = workloads.make(name, **over)
    rng = np.random.Generator(np.random.PCG64(seed))
    parts = [rng.permutation(w.E)[w.topk_idx] for _ in range(copies)]
    return w, np.ascontiguousarray(np.concatenate(parts).astype(np.int64))


def test_layout_multi_wave_grid_matches_oracle():
    """1,000,000 tokens at R=32 (3907 tiles, several waves of resident CTAs): the rank
    layout with a workspace and without one (noalloc) both match the oracle in full, and
    no bounded wait of the look-back runs out."""
    w, topk_np = _tiled_routing("dsv3", 16, T=62500, H=8)
    T, E, R, rpn = topk_np.shape[0], w.E, w.R, w.ranks_per_node
    assert T == 1_000_000
    L = oracle.layout(topk_np, E, R, rpn)
    topk = torch.from_numpy(topk_np).cuda()
    lay = ep.alloc_layout(T, E, R, rpn)
    ep.get_layout(topk, E, R, rpn, out=lay)
    got = layout_to_host(lay)
    for key, v in got.items():
        assert np.array_equal(v, L[key]), key
    assert ep.read_flags(lay.status) == 0
    assert ep.ep_layout_workspace_size(T, E, R, rpn) <= ep.LAYOUT_NOALLOC_SCRATCH_BYTES
    nl = ep.alloc_layout(T, E, R, rpn)
    ep.ep_get_layout_noalloc(topk, E, R, rpn, nl.tokens_per_expert, nl.tokens_per_rank, nl.tokens_per_node,
                             nl.is_token_in_rank, nl.is_token_in_node, nl.slot, nl.status)
    got = layout_to_host(nl)
    for key, v in got.items():
        assert np.array_equal(v, L[key]), ("noalloc", key)
    assert ep.read_flags(nl.status) == 0


def test_expert_layout_multi_wave_grid_matches_oracle():
    """262,144 tokens, E=256 (1024 tiles, several waves of resident CTAs): the expert layout
    matches the oracle in full and no bounded wait runs out."""
    w, topk_np = _tiled_routing("dsv3", 8, T=32768, H=8)
    T, k, E = topk_np.shape[0], w.k, w.E
    EL = oracle.expert_layout(topk_np, E)
    topk = torch.from_numpy(topk_np).cuda()
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    eslot = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = torch.zeros(ep.ep_expert_layout_workspace_size(T, E), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the workspace is left at rest: a second call gives the same
        ep.ep_get_expert_layout(topk, E, off, eslot, ws, st)
        assert np.array_equal(host_bits(off), EL["expert_offsets"])
        assert np.array_equal(host_bits(eslot), EL["expert_slot"])
        assert ep.read_flags(st) == 0


# ----------------------------------------------------------------------------- FP8 rounding edges

def test_fp8_ties_subnormals_and_signed_zeros():
    """Blocks with amax = 448 (scale exactly 1) whose other elements sit on E4M3 midpoints
    (normal and subnormal), an all-zero block with -0 entries, and +-0 entries inside
    blocks whose amax is not zero (E4M3 codes 0x00 / 0x80)."""
    mids = []
    vals = sorted({oracle.e4m3_to_f32(c) for c in range(0x7F) if c != 0x7F})
    for a, b in zip(vals[:-1], vals[1:]):
        mids.append((a + b) / 2)
    mids = np.array(mids, np.float32)
    rows = []
    rng = np.random.Generator(np.random.PCG64(21))
    for i in range(6):
        blocks = []
        for b in range(4):
            v = rng.choice(mids, 128).astype(np.float32) * rng.choice(np.array([-1, 1], np.float32), 128)
            v[rng.integers(0, 128)] = 448.0 * (1 if b % 2 == 0 else -1)
            blocks.append(v)
        if i == 3:
            blocks[2] = np.zeros(128, np.float32)
            blocks[2][::3] = -0.0
        if i == 4:  # signed zeros inside blocks whose amax is not zero
            blocks[1][::5] = -0.0
            blocks[3][1::7] = 0.0
        rows.append(np.concatenate(blocks))
    xf = np.stack(rows).astype(np.float32)
    bits = workloads.bf16_bits(xf)
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(back, xf)  # E4M3 midpoints are exact in bf16
    T, H = bits.shape
    w = workloads.make("tiny", T=T, H=H, E=4, k=1, R=4)
    w.x = bits
    w.topk_idx = np.arange(T, dtype=np.int64)[:, None] % 4
    w.topk_w = np.ones((T, 1), np.float32)
    w.fp8 = True
    w.expert = "scale"
    run_rank_path(w)


def test_combine_order_crafted():
    """2^24, 1, -2^24 from ranks 0, 1, 2: ascending fp32 order gives 0, descending 1."""
    H, R = 64, 3
    y = np.stack([workloads.bf16_bits(np.full((1, H), v, np.float32)) for v in (2.0 ** 24, 1.0, -(2.0 ** 24))])
    slot = np.zeros((1, R), np.int32)
    out = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(dev_bf16(y), torch.from_numpy(slot).cuda(), 1, out)
    ref, _ = oracle.combine(y, slot, 1)
    assert np.array_equal(host_bits(out), ref)
    assert np.all(ref == 0)


# ----------------------------------------------------------------------------- restripe + node dispatch

def run_node_path(w, chunk=None, P_override=None):
    chunk = chunk or w.chunk_tokens
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    topk, lay = gpu_layout(w)
    _assert_layout(w, lay, L)
    N, T, M, H = w.num_nodes, w.T, w.max_tokens, w.H
    prob = torch.from_numpy(w.prob).cuda()
    P = w.prob.shape[2]
    staging, bst = guarded((N, M, P), torch.float32, SENT_F32)
    ep.ep_restripe_prob(prob, M, staging)
    ref_st = oracle.restripe_prob(w.prob, M, fill=SENT_F32)
    assert np.array_equal(host_bits(staging).view(np.uint32), ref_st.view(np.uint32))
    check_guards(bst, staging.numel(), SENT_F32)
    x = dev_bf16(w.x)
    nchunks = (T + chunk - 1) // chunk
    for mode, dense in ((ep.NODES_DENSE, True), (ep.NODES_SPARSE, False)):
        rx, brx = guarded((N, M, H), torch.bfloat16, SENT_BF16)
        rp, brp = guarded((N, M, P), torch.float32, SENT_F32)
        runs = torch.full((N, nchunks), SENT_I32, dtype=torch.int32, device="cuda")
        ep.ep_dispatch_nodes(x, staging, lay.is_token_in_node, N, M, chunk, mode, rx, rp, runs)
        ref = oracle.dispatch_nodes(w.x, ref_st, L["is_token_in_node"], M, chunk, dense=dense, fill_x=SENT_BF16,
                                    fill_prob=SENT_F32)
        assert np.array_equal(host_bits(rx), ref["recv_x_node"])
        assert np.array_equal(host_bits(rp).view(np.uint32), ref["recv_prob_node"].view(np.uint32))
        assert np.array_equal(host_bits(runs), ref["num_runs"])
        check_guards(brx, rx.numel(), SENT_BF16)
        check_guards(brp, rp.numel(), SENT_F32)


@pytest.mark.parametrize("over,chunk", [
    ({"T": 700, "H": 512}, 256),
    ({"T": 1000, "H": 64, "P": 4}, 100),
    ({"T": 33, "H": 8, "P": 8, "N": 1, "ranks_per_node": 2}, 7),
    ({"T": 4097, "H": 128, "P": 128, "N": 16, "ranks_per_node": 2}, 256),
    ({"T": 600, "H": 256, "max_tokens": 1000}, 64),
    ({"T": 40, "H": 36864, "P": 8}, 16),  # rows too large for the bulk-copy scatter
])
def test_node_path_matches_oracle(over, chunk):
    run_node_path(workloads.make("restripe", **over), chunk=chunk)


@pytest.mark.parametrize("T,N,P,M", [
    (1000, 40, 128, 1200),  # node blocks of 32 (tiles cover 2 node blocks, the second ragged)
    (333, 3, 256, 333),     # the widest slice the tensor maps take
    (77, 100, 4, 80),       # tiny slices, many nodes
    (257, 8, 128, 300),     # ragged last token block; rows [T, M) untouched
    (1, 1, 4, 1),
    (500, 2, 260, 600),     # P > 256: the warp kernel
    (3000, 300, 8, 3001),   # N > 256: node blocks of 256
])
def test_restripe_shapes_match_oracle(T, N, P, M):
    rng = np.random.Generator(np.random.PCG64(T * 7 + N))
    prob = rng.random((T, N, P), dtype=np.float32)
    out, back = guarded((N, M, P), torch.float32, SENT_F32)
    ep.ep_restripe_prob(torch.from_numpy(prob).cuda(), M, out)
    ref = oracle.restripe_prob(prob, M, fill=SENT_F32)
    assert np.array_equal(host_bits(out).view(np.uint32), ref.view(np.uint32))
    check_guards(back, out.numel(), SENT_F32)


def test_node_path_full_size():
    """T=8192, H=7168, 8 nodes, P=128, chunks of 256: restripe, dense and sparse, in full."""
    run_node_path(workloads.make("restripe"))


# ----------------------------------------------------------------------------- layout specifics

@pytest.mark.parametrize("T,E,k,R,rpn", [
    (1000, 14, 3, 7, 7),      # R = 7: row widths that are no multiple of 4 or 16 bytes
    (777, 66, 5, 33, 3),      # R = 33, 11 nodes of 3: vectors wrap across token rows
    (5000, 96, 8, 96, 32),    # several tiles on fewer parts each; ragged last tile
    (39 * 256 + 5, 160, 6, 160, 5),  # 40 tiles (parts = 1 or 2), N = 32
    (300, 256, 9, 256, 256),  # the largest R, one node
    (20000, 256, 8, 32, 4),   # 79 tiles: one CTA per tile
])
def test_layout_odd_widths_and_tile_splits_match_oracle(T, E, k, R, rpn):
    w = workloads.make("tiny", T=T, H=8, E=E, k=k, R=R, ranks_per_node=rpn)
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    topk, lay = gpu_layout(w)
    _assert_layout(w, lay, L)
    # the same workspace again (the epoch advances, the counters are back at rest)
    ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
    _assert_layout(w, lay, L)


def test_layout_empty_batch_and_workspace_reuse():
    lay = ep.alloc_layout(5000, 256, 32, 4)
    for T in (0, 1, 300, 5000, 17, 4096):
        w = workloads.make("dsv3", T=T if T else 1, H=8)
        topk = torch.from_numpy(w.topk_idx[:T]).cuda()
        sub = ep.Layout(lay.tokens_per_expert, lay.tokens_per_rank, lay.tokens_per_node,
                        lay.is_token_in_rank[:T], lay.is_token_in_node[:T], lay.slot[:T], lay.workspace, lay.status,
                        256, 32, 4)
        ep.get_layout(topk, 256, 32, 4, out=sub)
        L = oracle.layout(w.topk_idx[:T], 256, 32, 4)
        got = layout_to_host(sub)
        for key, v in got.items():
            assert np.array_equal(v, L[key]), (T, key)
    # the same workspace, now for other E, R and node counts
    for name, T in (("restripe", 2000), ("skewed", 1500), ("tiny", 128)):
        w = workloads.make(name, T=T, H=8)
        other = ep.alloc_layout(w.T, w.E, w.R, w.ranks_per_node)
        assert lay.workspace.numel() >= ep.ep_layout_workspace_size(w.T, w.E, w.R, w.ranks_per_node)
        other.workspace = lay.workspace
        other.status = lay.status
        ep.get_layout(torch.from_numpy(w.topk_idx).cuda(), w.E, w.R, w.ranks_per_node, out=other)
        _assert_layout(w, other, oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node))
    assert ep.read_flags(lay.status) == 0


def test_path_captured_in_a_cuda_graph():
    """layout -> dispatch -> combine captured once in a CUDA graph and replayed: same results."""
    w = workloads.make("dsv3", T=1000, H=1024)
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    topk = torch.from_numpy(w.topk_idx).cuda()
    x = dev_bf16(w.x)
    tw = torch.from_numpy(w.topk_w).cuda()
    M = w.max_tokens
    lay = ep.get_layout(topk, w.E, w.R, w.ranks_per_node)
    d = ep.dispatch(x, topk, tw, lay, M)
    out = ep.combine(d.recv_x, lay, M)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
        ep.dispatch(x, topk, tw, lay, M, out=d)
        ep.combine(d.recv_x, lay, M, out=out)
    for _ in range(3):
        lay.slot.fill_(-5)
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    _assert_layout(w, lay, L)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, M)
    ref, _ = oracle.combine(D["recv_x"], L["slot"], M)
    assert np.array_equal(host_bits(out), ref)


def test_layout_bounded_wait_times_out_without_hanging():
    """Tile 1 never publishes (test hook): its successors give up after about a second,
    raise EP_FLAG_TIMEOUT, and the workspace still works for the next call."""
    w = workloads.make("dsv3", T=256 * 6, H=8)
    topk = torch.from_numpy(w.topk_idx).cuda()
    lay = ep.alloc_layout(w.T, w.E, w.R, w.ranks_per_node)
    lay.workspace[12:16].copy_(torch.tensor([2, 0, 0, 0], dtype=torch.uint8))  # stall_tile = 1 + 1
    ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
    assert ep.read_flags(lay.status) & ep.FLAG_TIMEOUT
    lay.workspace[12:16].zero_()
    lay.status.zero_()
    ep.get_layout(topk, w.E, w.R, w.ranks_per_node, out=lay)
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    _assert_layout(w, lay, L)


def test_outputs_are_deterministic():
    w = workloads.make("dsv3", T=2048, H=2048)
    _, a = run_rank_path(w)
    _, b = run_rank_path(w)
    assert np.array_equal(a, b)
