"""Pins for the oracle's send phase of a split (hook-mode) combine, oracle_combine_send:
each rank reduces, per received row, its local experts' expert-major rows into one bf16
row of its rank-level slab, which the combine's receive phase (oracle_combine) reads.

Pinned by a round trip through the receive-side permute, closed forms (identity rows:
bf16(n * x); power-of-two weights: every partial sum exact), a crafted row whose result
depends on the order of its terms, the equality of the split and the fused combine where
it must hold, and the capacity rule.
"""
import numpy as np
import torch

import oracle
import workloads


def _bf16_round(v64):
    """float64 values exactly representable in fp32 -> bf16 bits (one rounding, torch)."""
    t = torch.from_numpy(np.asarray(v64, np.float64).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _pipeline(w, M=None):
    L = oracle.layout(w.topk_idx, w.E, w.R)
    M = M or w.T
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, M)
    EL = oracle.expert_layout(w.topk_idx, w.E)
    Mp = int(oracle.rows_per_rank(EL["expert_offsets"], w.E, w.R).max())
    return L, D, EL, Mp, M


def _received(L, M, R):
    return np.arange(M)[None, :] < np.minimum(L["tokens_per_rank"], M)[:, None]


def test_combine_send_inverts_the_receive_side_permute():
    """One expert per rank per token: the expert-major rows are copies of the rank rows,
    so the unweighted send phase gives the rank rows back bit for bit."""
    rng = np.random.Generator(np.random.PCG64(5))
    T, H, E, R, k = 150, 48, 16, 16, 4  # one expert per rank: ranks of a token are distinct
    w = workloads.make("tiny", T=T, H=H, E=E, k=k, R=R)
    w.topk_idx = workloads.routing_uniform(rng, T, E, k)
    L, D, EL, Mp, M = _pipeline(w)
    y = workloads.random_bf16_rows(11, (R, M, H))  # any rank-level expert outputs
    Dy = dict(D, recv_x=y)
    P = oracle.permute_received(Dy, L["tokens_per_rank"], EL, T, E, R, Mp)
    back, flags = oracle.combine_send(P["perm_x"], D, L["tokens_per_rank"], EL, T, E, R, weighted=False, fill=7)
    rec = _received(L, M, R)
    assert flags == 0
    assert np.array_equal(back[rec], y[rec])
    assert np.all(back[~rec] == 7)  # rows nobody received are not written


def test_combine_send_identity_rows_closed_form():
    """Expert-major rows = x[t] (the fused dispatch's rows, identity expert), unweighted:
    the rank row of token t is bf16(n * x[t]), n = the token's experts on that rank (n * x
    is exact in fp32, so the one rounding is torch's)."""
    for name, over in (("tiny", {"T": 200, "H": 64}), ("dsv3", {"T": 120, "H": 32})):
        w = workloads.make(name, **over)
        L, D, EL, Mp, M = _pipeline(w)
        PX = oracle.dispatch_permuted(w.x, w.topk_idx, w.topk_w, EL, w.E, w.R, Mp)
        y, flags = oracle.combine_send(PX["perm_x"], D, L["tokens_per_rank"], EL, w.T, w.E, w.R, weighted=False)
        assert flags == 0
        epr = w.E // w.R
        xs = _f(w.x)
        rec = _received(L, M, w.R)
        several = 0
        for r in range(w.R):
            for s in range(int(L["tokens_per_rank"][r])):
                t = int(D["recv_src_idx"][r, s])
                n = int(np.sum((w.topk_idx[t] >= 0) & (w.topk_idx[t] // epr == r)))
                several += n > 1
                assert np.array_equal(y[r, s], _bf16_round(n * xs[t])), (name, r, s)
        assert several > 0  # the workload does put several experts of a token on one rank
        assert rec.sum() == int(L["tokens_per_rank"].sum())


def test_combine_send_power_of_two_weights_closed_form():
    """Weights 2^-j: every product and partial sum of a bf16 value is exact in fp32, so the
    rank row is bf16 of the exact sum x * (sum of the local slots' weights)."""
    w = workloads.make("tiny", T=180, H=40)
    k = w.k
    w.topk_w = np.tile((2.0 ** -np.arange(k)).astype(np.float32), (w.T, 1))
    L, D, EL, Mp, M = _pipeline(w)
    PX = oracle.dispatch_permuted(w.x, w.topk_idx, w.topk_w, EL, w.E, w.R, Mp)
    y, _ = oracle.combine_send(PX["perm_x"], D, L["tokens_per_rank"], EL, w.T, w.E, w.R, weighted=True)
    epr = w.E // w.R
    xs = _f(w.x)
    for r in range(w.R):
        for s in range(int(L["tokens_per_rank"][r])):
            t = int(D["recv_src_idx"][r, s])
            on = (w.topk_idx[t] >= 0) & (w.topk_idx[t] // epr == r)
            wsum = float(np.sum(2.0 ** -np.arange(k)[on]))
            assert np.array_equal(y[r, s], _bf16_round(wsum * xs[t])), (r, s)


def test_combine_send_term_order_is_the_slot_order():
    """A token with three experts on rank 0 whose expert-major rows hold 2^24, 1, -2^24 in
    slot order: adding in slot order gives 0 (2^24 + 1 rounds back to 2^24), the reverse
    order gives 1."""
    H, E, R = 16, 8, 2
    topk = np.array([[0, 1, 2]], np.int64)  # experts 0, 1, 2 all on rank 0
    x = np.zeros((1, H), np.uint16)
    w = np.ones((1, 3), np.float32)
    L = oracle.layout(topk, E, R)
    D = oracle.dispatch(x, topk, w, L["slot"], E, R, 1)
    EL = oracle.expert_layout(topk, E)
    vals = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    yp = np.zeros((R, 3, H), np.uint16)
    for j, v in enumerate(vals):  # row of (t=0, j) on rank 0 is expert_offsets[j] + 0 = j
        yp[0, j] = _bf16_round(np.full(H, v))
    y, _ = oracle.combine_send(yp, D, L["tokens_per_rank"], EL, 1, E, R, weighted=False)
    assert np.all(y[0, 0] == 0)


def test_split_combine_equals_fused_where_it_must():
    """Unweighted, one expert per rank per token, top-k ids ascending (so slot order is rank
    order): the send phase copies rows and the receive phase sums them in the same order
    as the fused combine from the expert-major slabs -- equal bit for bit."""
    rng = np.random.Generator(np.random.PCG64(9))
    T, H, E, R, k = 300, 64, 32, 32, 6
    w = workloads.make("tiny", T=T, H=H, E=E, k=k, R=R)
    w.topk_idx = np.sort(workloads.routing_uniform(rng, T, E, k), axis=1)
    L, D, EL, Mp, M = _pipeline(w)
    yp = workloads.random_bf16_rows(3, (R, Mp, H))  # any expert outputs
    y, f1 = oracle.combine_send(yp, D, L["tokens_per_rank"], EL, T, E, R, weighted=False)
    split, f2 = oracle.combine(y, L["slot"], M)
    fused, f3 = oracle.combine_permuted(yp, w.topk_idx, None, EL, E, R)
    assert f1 == f2 == f3 == 0
    assert np.array_equal(split, fused)


def test_combine_send_capacity_drops_and_flags():
    w = workloads.make("tiny", T=100, H=16)
    L, D, EL, Mp, M = _pipeline(w)
    yp = workloads.random_bf16_rows(4, (w.R, Mp, w.H))
    full, f_full = oracle.combine_send(yp, D, L["tokens_per_rank"], EL, w.T, w.E, w.R, weighted=False)
    small = Mp // 2
    part, f_part = oracle.combine_send(np.ascontiguousarray(yp[:, :small]), D, L["tokens_per_rank"], EL, w.T, w.E,
                                       w.R, weighted=False)
    assert f_full == 0 and f_part == oracle.FLAG_CAPACITY
    # a row whose local experts all sit below the cut is unchanged; others lose terms
    assert not np.array_equal(full, part)
