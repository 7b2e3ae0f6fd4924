"""GPU parity of the expert-major path against the oracle, bit for bit: the expert
layout, the fused dispatch + permute, the receive-side permute of a split dispatch
(whose result must equal the fused one), the combine from expert-major slabs (normal
and low-latency forms), weighted and unweighted, and the split combine (send phase back
into the rank slabs, then the rank-level combine). Output buffers sit between guard
regions."""
import numpy as np
import pytest
import torch

import combine_ep_get_05_gb300 as ep
import oracle
import workloads
from gpu_helpers import SENT_BF16, SENT_F32, SENT_I32, check_guards, dev_bf16, gpu_layout, guarded, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.build_library()
    ep.lib()


def gpu_expert_layout(topk, E, ws=None):
    T, k = topk.shape
    off = torch.full((E + 1,), -9, dtype=torch.int32, device="cuda")
    slot = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = torch.zeros(max(256, ep.ep_expert_layout_workspace_size(T, E)), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_get_expert_layout(topk, E, off, slot, ws, status)
    return off, slot, ws, status


def check_expert_layout(w, topk_np=None):
    topk_np = w.topk_idx if topk_np is None else topk_np
    EL = oracle.expert_layout(topk_np, w.E)
    off, slot, ws, status = gpu_expert_layout(torch.from_numpy(topk_np).cuda(), w.E)
    assert np.array_equal(host_bits(off), EL["expert_offsets"])
    assert np.array_equal(host_bits(slot), EL["expert_slot"])
    assert int(status.item()) == EL["flags"]
    return EL, off, slot


def run_permuted(w, max_rows=None, weighted=True):
    E, R, T, H, k = w.E, w.R, w.T, w.H, w.k
    EL, off, slot = check_expert_layout(w)
    rows = oracle.rows_per_rank(EL["expert_offsets"], E, R)
    M = max_rows if max_rows is not None else max(1, int(rows.max()))
    x = dev_bf16(w.x)
    topk = torch.from_numpy(w.topk_idx).cuda()
    tw = torch.from_numpy(w.topk_w).cuda()

    # fused dispatch + permute
    px, bpx = guarded((R, M, H), torch.bfloat16, SENT_BF16)
    ps, bps = guarded((R, M), torch.int32, SENT_I32)
    pw, bpw = guarded((R, M), torch.float32, SENT_F32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_permuted(x, topk, tw, off, slot, E, R, M, px, ps, pw, st)
    ref = oracle.dispatch_permuted(w.x, w.topk_idx, w.topk_w, EL, E, R, M, fill_x=SENT_BF16, fill_idx=SENT_I32,
                                   fill_w=SENT_F32)
    assert int(st.item()) == ref["flags"]
    assert np.array_equal(host_bits(px), ref["perm_x"])
    assert np.array_equal(host_bits(ps), ref["perm_src"])
    assert np.array_equal(host_bits(pw).view(np.uint32), ref["perm_w"].view(np.uint32))
    for b, v, f in ((bpx, px, SENT_BF16), (bps, ps, SENT_I32), (bpw, pw, SENT_F32)):
        check_guards(b, v.numel(), f)

    # split: rank-level dispatch (send), then the receive-side permute
    L = oracle.layout(w.topk_idx, E, R, w.ranks_per_node)
    Mr = max(1, int(L["tokens_per_rank"].max()))
    topk_d, lay = gpu_layout(w)
    d = ep.alloc_dispatch(R, Mr, H, k)
    ep.dispatch(x, topk_d, tw, lay, Mr, out=d)
    sx, bsx = guarded((R, M, H), torch.bfloat16, SENT_BF16)
    ss, bss = guarded((R, M), torch.int32, SENT_I32)
    sw, bsw = guarded((R, M), torch.float32, SENT_F32)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_permute_received(d.recv_x, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w, lay.tokens_per_rank, off, slot,
                           E, M, sx, ss, sw, st2)
    assert int(st2.item()) == ref["flags"]
    assert np.array_equal(host_bits(sx), ref["perm_x"])
    assert np.array_equal(host_bits(ss), ref["perm_src"])
    assert np.array_equal(host_bits(sw).view(np.uint32), ref["perm_w"].view(np.uint32))
    for b, v, f in ((bsx, sx, SENT_BF16), (bss, ss, SENT_I32), (bsw, sw, SENT_F32)):
        check_guards(b, v.numel(), f)

    # combine from the slabs: random expert outputs (seeded), weighted and plain; some
    # entries are -0 (a sum that starts from +0 turns a lone -0 term into +0)
    y_np = workloads.random_bf16_rows(17, (R, M, H))
    y_np.reshape(-1)[::97] = 0x8000
    y = dev_bf16(y_np)
    for wts in (((tw, w.topk_w),) if weighted else ()) + ((None, None),):
        out, bout = guarded((T, H), torch.bfloat16, SENT_BF16)
        st3 = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_combine_permuted(y, topk, wts[0], off, slot, E, out, st3)
        exp, flags = oracle.combine_permuted(y_np, w.topk_idx, wts[1], EL, E, R)
        assert int(st3.item()) == flags
        assert np.array_equal(host_bits(out), exp)
        check_guards(bout, out.numel(), SENT_BF16)
        if T <= 1024 and E <= 1024:  # the low-latency form: the same bits
            out_ll, bll = guarded((T, H), torch.bfloat16, SENT_BF16)
            st5 = torch.zeros(1, dtype=torch.int32, device="cuda")
            ep.ep_combine_permuted_ll(y, topk, wts[0], off, slot, E, out_ll, st5)
            assert int(st5.item()) == flags
            assert np.array_equal(host_bits(out_ll), exp)
            check_guards(bll, out_ll.numel(), SENT_BF16)

    # split combine: send phase (expert-major rows back into the rank slabs), then the
    # receive phase (the rank-level combine)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], E, R, Mr, rows=False)
    for weighted_send in ((True, False) if weighted else (False,)):
        yr, byr = guarded((R, Mr, H), torch.bfloat16, SENT_BF16)
        st4 = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_combine_send(y, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w if weighted_send else None,
                           lay.tokens_per_rank, off, slot, E, yr, st4)
        exp_r, f_send = oracle.combine_send(y_np, D, L["tokens_per_rank"], EL, T, E, R, weighted=weighted_send,
                                            fill=SENT_BF16)
        assert int(st4.item()) == f_send
        assert np.array_equal(host_bits(yr), exp_r)
        check_guards(byr, yr.numel(), SENT_BF16)
        out, bout = guarded((T, H), torch.bfloat16, SENT_BF16)
        ep.ep_combine(yr, lay.slot, Mr, out)
        exp_c, _ = oracle.combine(exp_r, L["slot"], Mr)
        assert np.array_equal(host_bits(out), exp_c)
        check_guards(bout, out.numel(), SENT_BF16)


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("tiny", {"T": 1}),
    ("dsv3", {"T": 1000, "H": 1024}),
    ("dsv3", {"T": 777, "H": 7168}),
    ("skewed", {"T": 3000, "H": 256}),
    ("restripe", {"T": 600, "H": 128}),
    ("dsv3", {"T": 40, "H": 36864}),  # rows too large for the bulk-copy scatter
    ("dsv3", {"T": 128}),             # a decode batch at the full hidden size
    ("tiny", {"T": 1000, "H": 8, "k": 32, "E": 64, "R": 4}),  # k = 32: sources in several batches
])
def test_permuted_path_matches_oracle(name, over):
    run_permuted(workloads.make(name, **over))


def test_permuted_path_full_size_dsv3():
    run_permuted(workloads.make("dsv3"))


def test_permuted_capacity_overflow():
    w = workloads.make("skewed", T=2000, H=64)
    EL = oracle.expert_layout(w.topk_idx, w.E)
    rows = oracle.rows_per_rank(EL["expert_offsets"], w.E, w.R)
    run_permuted(w, max_rows=int(rows.max()) // 2)


def test_expert_layout_edge_cases():
    rng = np.random.Generator(np.random.PCG64(31))
    # repeats, out-of-range ids and empty slots are dropped and flagged
    w = workloads.make("tiny", T=700, H=8)
    t = w.topk_idx.copy()
    t[3, 1] = t[3, 0]
    t[10, 2] = w.E + 5
    t[20, :] = -1
    check_expert_layout(w, t)
    # the largest expert count, k = 32, several tiles with a ragged tail
    topk = workloads.routing_uniform(rng, 1537, 1024, 32)
    w2 = workloads.make("tiny", T=1537, H=8, E=1024, k=32, R=4)
    check_expert_layout(w2, topk)
    # empty batch
    off, slot, ws, status = gpu_expert_layout(torch.zeros((0, 4), dtype=torch.int64, device="cuda"), 16)
    assert np.all(host_bits(off) == 0) and int(status.item()) == 0


def test_expert_layout_workspace_reuse_and_bounded_wait():
    w = workloads.make("dsv3", T=256 * 5, H=8)
    topk = torch.from_numpy(w.topk_idx).cuda()
    EL = oracle.expert_layout(w.topk_idx, w.E)
    off, slot, ws, status = gpu_expert_layout(topk, w.E)
    ws[12:16].copy_(torch.tensor([3, 0, 0, 0], dtype=torch.uint8))  # tile 2 never publishes
    status.zero_()
    ep.ep_get_expert_layout(topk, w.E, off, slot, ws, status)
    assert int(status.item()) & ep.FLAG_TIMEOUT
    ws[12:16].zero_()
    for T in (1280, 300, 1):  # the same workspace keeps working, whatever T
        status.zero_()
        ep.ep_get_expert_layout(topk[:T], w.E, off, slot[:T], ws, status)
        ELT = oracle.expert_layout(w.topk_idx[:T], w.E)
        assert np.array_equal(host_bits(off), ELT["expert_offsets"])
        assert np.array_equal(host_bits(slot[:T]), ELT["expert_slot"])
        assert int(status.item()) == 0


def run_ll(w, topk_np=None, max_rows=None):
    """The single-launch decode-sized dispatch + permute against the oracle's layout and
    dispatch + permute, every output compared bit for bit, between guard regions."""
    topk_np = w.topk_idx if topk_np is None else topk_np
    E, R, T, H, k = w.E, w.R, w.T, w.H, topk_np.shape[1]
    EL = oracle.expert_layout(topk_np, E)
    rows = oracle.rows_per_rank(EL["expert_offsets"], E, R)
    M = max_rows if max_rows is not None else max(1, int(rows.max()))
    off, boff = guarded((E + 1,), torch.int32, SENT_I32)
    slot, bslot = guarded((T, k), torch.int32, SENT_I32)
    px, bpx = guarded((R, M, H), torch.bfloat16, SENT_BF16)
    ps, bps = guarded((R, M), torch.int32, SENT_I32)
    pw, bpw = guarded((R, M), torch.float32, SENT_F32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_permuted_ll(dev_bf16(w.x), torch.from_numpy(topk_np).cuda(), torch.from_numpy(w.topk_w).cuda(), E, R,
                               M, off, slot, px, ps, pw, st)
    ref = oracle.dispatch_permuted(w.x, topk_np, w.topk_w, EL, E, R, M, fill_x=SENT_BF16, fill_idx=SENT_I32,
                                   fill_w=SENT_F32)
    assert int(st.item()) == (EL["flags"] | ref["flags"])
    assert np.array_equal(host_bits(off), EL["expert_offsets"])
    assert np.array_equal(host_bits(slot), EL["expert_slot"])
    assert np.array_equal(host_bits(px), ref["perm_x"])
    assert np.array_equal(host_bits(ps), ref["perm_src"])
    assert np.array_equal(host_bits(pw).view(np.uint32), ref["perm_w"].view(np.uint32))
    for b, v, f in ((boff, off, SENT_I32), (bslot, slot, SENT_I32), (bpx, px, SENT_BF16), (bps, ps, SENT_I32),
                    (bpw, pw, SENT_F32)):
        check_guards(b, v.numel(), f)


@pytest.mark.parametrize("name,over", [
    ("dsv3", {"T": 128}),              # a decode batch at the full hidden size
    ("dsv3", {"T": 1, "H": 1024}),
    ("dsv3", {"T": 256, "H": 1024}),
    ("dsv3", {"T": 257, "H": 512}),    # a second chunk of one token
    ("dsv3", {"T": 1024, "H": 256}),   # the largest batch
    ("skewed", {"T": 1000, "H": 256}),
    ("restripe", {"T": 600, "H": 128}),  # E = 1024, empty slots
])
def test_low_latency_dispatch_permuted_matches_oracle(name, over):
    run_ll(workloads.make(name, **over))


def test_low_latency_dispatch_permuted_edge_cases():
    rng = np.random.Generator(np.random.PCG64(33))
    w = workloads.make("tiny", T=300, H=64)
    t = w.topk_idx.copy()
    t[3, 1] = t[3, 0]   # repeat
    t[10, 2] = w.E + 5  # out of range
    t[20, :] = -1       # routed nowhere
    run_ll(w, t)
    # k = 32 at the entry limit (T * k = 8192), E = 1024
    w2 = workloads.make("tiny", T=256, H=32, E=1024, k=32, R=4)
    run_ll(w2, workloads.routing_uniform(rng, 256, 1024, 32))
    # capacity drops
    w3 = workloads.make("skewed", T=800, H=64)
    EL = oracle.expert_layout(w3.topk_idx, w3.E)
    run_ll(w3, max_rows=int(oracle.rows_per_rank(EL["expert_offsets"], w3.E, w3.R).max()) // 2)
    # empty batch: zero offsets; over the limits: refused
    off = torch.full((17,), -9, dtype=torch.int32, device="cuda")
    z = torch.zeros((0, 4), dtype=torch.int64, device="cuda")
    ep.ep_dispatch_permuted_ll(torch.zeros((0, 8), dtype=torch.bfloat16, device="cuda"), z, None, 16, 4, 1, off,
                               torch.zeros((0, 4), dtype=torch.int32, device="cuda"),
                               torch.zeros((4, 1, 8), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert np.all(host_bits(off) == 0)
    lib = ep.lib()
    assert lib.ep_dispatch_permuted_ll(None, None, None, 1025, 8, 1, 16, 4, 1, None, None, None, None, None, None,
                                       None) == ep.EP_ERR_INVALID


def test_split_combine_equals_fused_when_it_must():
    """Unweighted, one expert per rank per token, ids ascending: the send phase copies rows
    and the receive phase adds them in the fused combine's order, so the split combine
    equals ep_combine_permuted bit for bit."""
    rng = np.random.Generator(np.random.PCG64(12))
    T, H, E, R, k = 2000, 1024, 64, 64, 8
    w = workloads.make("tiny", T=T, H=H, E=E, k=k, R=R, ranks_per_node=R)
    w.topk_idx = np.sort(workloads.routing_uniform(rng, T, E, k), axis=1)
    topk = torch.from_numpy(w.topk_idx).cuda()
    EL, off, slot = check_expert_layout(w)
    Mp = max(1, int(oracle.rows_per_rank(EL["expert_offsets"], E, R).max()))
    y = dev_bf16(workloads.random_bf16_rows(5, (R, Mp, H)))
    fused = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine_permuted(y, topk, None, off, slot, E, fused)
    _, lay = gpu_layout(w)
    Mr = T
    d = ep.alloc_dispatch(R, Mr, 8, k)  # only the metadata is needed
    ep.ep_dispatch(dev_bf16(w.x[:, :8].copy()), ep.DTYPE_BF16, topk, torch.from_numpy(w.topk_w).cuda(), lay.slot, E, R,
                   Mr, d.recv_x, None, d.recv_src_idx, d.recv_topk_idx, d.recv_topk_w)
    yr = torch.empty((R, Mr, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine_send(y, d.recv_src_idx, d.recv_topk_idx, None, lay.tokens_per_rank, off, slot, E, yr)
    split = ep.combine(yr, lay, Mr)
    assert torch.equal(split, fused)


def test_low_latency_combine_edge_cases():
    """Routed-nowhere tokens (+0 rows), repeated and out-of-range ids, experts with no
    tokens, capacity drops, the largest batch, an empty batch and the refusals."""
    w = workloads.make("tiny", T=300, H=64)
    t = w.topk_idx.copy()
    t[3, 1] = t[3, 0]   # repeat
    t[10, 2] = w.E + 5  # out of range
    t[20, :] = -1       # routed nowhere
    t[:, :][t == 7] = 6  # expert 7 gets no token
    t[np.arange(300) % 5 == 0, 3] = -1
    w.topk_idx = t
    for over_rows in (None, 0.5):
        EL = oracle.expert_layout(t, w.E)
        rows = oracle.rows_per_rank(EL["expert_offsets"], w.E, w.R)
        M = max(1, int(rows.max())) if over_rows is None else max(1, int(rows.max() * over_rows))
        y_np = workloads.random_bf16_rows(23, (w.R, M, w.H))
        off = torch.from_numpy(EL["expert_offsets"]).cuda()
        slot = torch.from_numpy(EL["expert_slot"]).cuda()
        for tw_np in (w.topk_w, None):
            out, bout = guarded((w.T, w.H), torch.bfloat16, SENT_BF16)
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            ep.ep_combine_permuted_ll(dev_bf16(y_np), torch.from_numpy(t).cuda(),
                                      None if tw_np is None else torch.from_numpy(tw_np).cuda(), off, slot, w.E, out, st)
            exp, flags = oracle.combine_permuted(y_np, t, tw_np, EL, w.E, w.R)
            assert int(st.item()) == flags
            assert np.array_equal(host_bits(out), exp)
            assert np.all(host_bits(out)[20] == 0)
            check_guards(bout, out.numel(), SENT_BF16)
    # the largest batch (T = 1024) at a ragged width
    w2 = workloads.make("dsv3", T=1024, H=264)
    EL = oracle.expert_layout(w2.topk_idx, w2.E)
    Mp = int(oracle.rows_per_rank(EL["expert_offsets"], w2.E, w2.R).max())
    y_np = workloads.random_bf16_rows(29, (w2.R, Mp, w2.H))
    out = torch.empty((w2.T, w2.H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine_permuted_ll(dev_bf16(y_np), torch.from_numpy(w2.topk_idx).cuda(), torch.from_numpy(w2.topk_w).cuda(),
                              torch.from_numpy(EL["expert_offsets"]).cuda(), torch.from_numpy(EL["expert_slot"]).cuda(),
                              w2.E, out)
    exp, _ = oracle.combine_permuted(y_np, w2.topk_idx, w2.topk_w, EL, w2.E, w2.R)
    assert np.array_equal(host_bits(out), exp)
    # empty batch: nothing launched; over the limits: refused before any launch
    lib = ep.lib()
    assert lib.ep_combine_permuted_ll(None, None, None, None, None, 0, 8, 4, 16, 4, 1, 4096, None, None) == ep.EP_OK
    assert lib.ep_combine_permuted_ll(None, None, None, None, None, 1025, 8, 4, 16, 4, 1, 4096, None,
                                      None) == ep.EP_ERR_INVALID
    assert lib.ep_combine_permuted_ll(None, None, None, None, None, 8, 8, 4, 2048, 4, 1, 4096, None,
                                      None) == ep.EP_ERR_INVALID
