"""Pins for the oracle's expert-major routines: expert layout, fused dispatch+permute,
receive-side permute and combine from the expert-major slabs.

Checked against numpy restatements (stable argsort, bincount/cumsum), the equality of
the fused and the split (dispatch, then receive-side permute) paths, a closed form for
the unweighted combine, a sequential fp32 brute force for the weighted one, and a crafted
token whose result depends on the order of its terms.
"""
import numpy as np
import torch

import oracle
import workloads


def _restate_layout(topk, E):
    """Stable counting sort by expert, restated with numpy (first occurrence per row only)."""
    T, k = topk.shape
    valid = (topk >= 0) & (topk < E)
    for j in range(k):  # a repeat of an earlier id in the same row does not count
        for jj in range(j):
            valid[:, j] &= topk[:, j] != topk[:, jj]
    flat = np.where(valid, topk, E).ravel()  # invalid entries sort last
    order = np.argsort(flat, kind="stable")  # (t, j) order within each expert
    counts = np.bincount(flat[valid.ravel()], minlength=E)[:E]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    slot = np.full(T * k, -1, np.int32)
    pos_in_sorted = np.empty(T * k, np.int64)
    pos_in_sorted[order] = np.arange(T * k)
    idx = np.nonzero(valid.ravel())[0]
    slot[idx] = pos_in_sorted[idx] - offsets[flat[idx]]
    return offsets, slot.reshape(T, k)


def _work(seed=3, T=97, H=64, E=24, R=4, k=4):
    rng = np.random.Generator(np.random.PCG64(seed))
    topk = workloads.routing_uniform(rng, T, E, k)
    x = workloads.bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    w = rng.random((T, k), dtype=np.float32)
    return x, topk, w


def test_expert_layout_matches_stable_sort_restatement():
    for seed, E, k in ((1, 24, 4), (2, 256, 8), (3, 8, 8), (4, 16, 1)):
        x, topk, w = _work(seed=seed, E=E, k=k, R=4 if E % 4 == 0 else 1)
        topk[3, k - 1] = -1
        topk[5, :] = -1
        EL = oracle.expert_layout(topk, E)
        off, slot = _restate_layout(topk, E)
        assert np.array_equal(EL["expert_offsets"], off)
        assert np.array_equal(EL["expert_slot"], slot)
        assert EL["flags"] == 0


def test_expert_layout_repeats_and_out_of_range_are_dropped_and_flagged():
    topk = np.array([[0, 2, 2], [5, 1, 0], [2, -1, 9]], np.int64)  # E = 6
    EL = oracle.expert_layout(topk, 6)
    assert EL["flags"] == oracle.FLAG_BAD_EXPERT
    assert EL["expert_slot"].tolist() == [[0, 0, -1], [0, 0, 1], [1, -1, -1]]
    assert EL["expert_offsets"].tolist() == [0, 2, 3, 5, 5, 5, 6]


def test_dispatch_permuted_groups_rows_by_local_expert_in_token_order():
    x, topk, w = _work()
    E, R = 24, 4
    epr = E // R
    EL = oracle.expert_layout(topk, E)
    rows = oracle.rows_per_rank(EL["expert_offsets"], E, R)
    M = int(rows.max())
    Pm = oracle.dispatch_permuted(x, topk, w, EL, E, R, M, fill_x=0xFFFF, fill_idx=-5, fill_w=-1.0)
    assert Pm["flags"] == 0
    for r in range(R):
        p = 0
        for l in range(epr):
            e = r * epr + l
            toks, js = np.nonzero(topk == e)  # ascending token order
            n = len(toks)
            assert np.array_equal(Pm["perm_src"][r, p:p + n], toks)
            assert np.array_equal(Pm["perm_x"][r, p:p + n], x[toks])
            assert np.array_equal(Pm["perm_w"][r, p:p + n], w[toks, js])
            p += n
        assert p == rows[r]
        assert np.all(Pm["perm_src"][r, p:] == -5)


def test_split_path_equals_fused_path_and_capacity():
    x, topk, w = _work(seed=8, T=150, E=32, R=8, k=6)
    E, R, T = 32, 8, 150
    L = oracle.layout(topk, E, R)
    EL = oracle.expert_layout(topk, E)
    M = int(oracle.rows_per_rank(EL["expert_offsets"], E, R).max())
    fused = oracle.dispatch_permuted(x, topk, w, EL, E, R, M, fill_idx=-3)
    D = oracle.dispatch(x, topk, w, L["slot"], E, R, T)
    split = oracle.permute_received(D, L["tokens_per_rank"], EL, T, E, R, M, fill_idx=-3)
    for key in ("perm_x", "perm_src", "perm_w"):
        assert np.array_equal(fused[key], split[key]), key
    small = oracle.dispatch_permuted(x, topk, w, EL, E, R, M - 2, fill_idx=-3)
    assert small["flags"] == oracle.FLAG_CAPACITY
    assert np.array_equal(small["perm_x"], fused["perm_x"][:, :M - 2])


def test_combine_permuted_closed_form_and_brute_force():
    x, topk, w = _work(seed=11, T=60, H=32, E=16, R=4, k=4)
    E, R = 16, 4
    topk[7, 2] = -1
    EL = oracle.expert_layout(topk, E)
    M = int(oracle.rows_per_rank(EL["expert_offsets"], E, R).max())
    Pm = oracle.dispatch_permuted(x, topk, w, EL, E, R, M)
    # unweighted, identity expert: bf16(n * x), exact
    out, flags = oracle.combine_permuted(Pm["perm_x"], topk, None, EL, E, R)
    n = (EL["expert_slot"] >= 0).sum(1).astype(np.float32)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    exp = (xt * torch.from_numpy(n)[:, None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert flags == 0 and np.array_equal(out, exp)
    # weighted: sequential fp32 in j order, each product and sum rounded once
    rng = np.random.Generator(np.random.PCG64(5))
    y = workloads.bf16_bits(rng.standard_normal(Pm["perm_x"].shape, dtype=np.float32) * 100)
    out, _ = oracle.combine_permuted(y, topk, w, EL, E, R)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).float().numpy()
    epr = E // R
    for t in range(60):
        acc = np.zeros(32, np.float32)
        for j in range(4):
            s = EL["expert_slot"][t, j]
            if s < 0:
                continue
            e = topk[t, j]
            r = e // epr
            p = EL["expert_offsets"][e] - EL["expert_offsets"][r * epr] + s
            acc = (acc + (yf[r, p] * np.float32(w[t, j])).astype(np.float32)).astype(np.float32)
        ref = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[t], ref)


def test_combine_permuted_term_order_is_the_topk_order():
    """Slots j = 0, 1, 2 carry 2^24, 1, -2^24: j order gives 0, any other order can give 1."""
    E, R, H = 3, 1, 8
    topk = np.array([[0, 1, 2]], np.int64)
    EL = oracle.expert_layout(topk, E)
    y = np.stack([workloads.bf16_bits(np.full((1, H), v, np.float32))[0]
                  for v in (2.0 ** 24, 1.0, -(2.0 ** 24))])[None]  # [1][3][H], rows in expert order
    out, _ = oracle.combine_permuted(y, topk, None, EL, E, R)
    assert np.all(out == 0)
    topk_rev = np.array([[2, 1, 0]], np.int64)
    EL2 = oracle.expert_layout(topk_rev, E)
    out2, _ = oracle.combine_permuted(y, topk_rev, None, EL2, E, R)
    assert np.all(out2 == 0x3F80)
