"""Pins for the oracle's path routines: layout, dispatch, restripe, node dispatch, combine.

Each routine is checked against what the definitions and mathematics fix,
never against a retyping of its own loop: exhaustive brute force on tiny
routings, numpy set/cumsum/bincount restatements, stable-partition invariants,
closed forms (identity-expert combine = bf16(n_ranks * x), restripe inverse)
and special cases (R = 1 combine is a copy).
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads


def _defs(topk, E, R, rpn=0):
    """Layout restated with numpy set operations and cumulative sums."""
    T, k = topk.shape
    epr = E // R
    valid = (topk >= 0) & (topk < E)
    tpe = np.bincount(topk[valid], minlength=E)
    in_rank = np.zeros((T, R), np.uint8)
    for t in range(T):
        for r in {int(e) // epr for e in topk[t] if 0 <= e < E}:
            in_rank[t, r] = 1
    before = np.cumsum(in_rank.astype(np.int64), axis=0) - in_rank
    slot = np.where(in_rank == 1, before, -1)
    out = dict(tokens_per_expert=tpe, tokens_per_rank=in_rank.sum(0), is_token_in_rank=in_rank, slot=slot)
    if rpn:
        in_node = in_rank.reshape(T, R // rpn, rpn).max(axis=2)
        out.update(is_token_in_node=in_node, tokens_per_node=in_node.sum(0))
    return out


def _check_layout(topk, E, R, rpn=0):
    got = oracle.layout(topk, E, R, rpn)
    exp = _defs(topk, E, R, rpn)
    for key, v in exp.items():
        assert np.array_equal(got[key], v), key
    return got


# ----------------------------------------------------------------------------- layout

def test_layout_exhaustive_tiny():
    """Every routing of 3 tokens, 2 distinct experts of 4, 2 ranks (and 2 nodes of 1 rank)."""
    pairs = list(itertools.permutations(range(4), 2))
    for combo in itertools.product(pairs, repeat=3):
        topk = np.array(combo, np.int64)
        _check_layout(topk, E=4, R=2, rpn=1)


def test_layout_exhaustive_with_empty_slots():
    choices = [(-1, -1), (0, -1), (-1, 3), (1, 2), (2, 3), (0, 1)]
    for combo in itertools.product(choices, repeat=3):
        _check_layout(np.array(combo, np.int64), E=4, R=4, rpn=2)


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("dsv3", {"T": 1000}),
    ("restripe", {"T": 700}),
    ("skewed", {"T": 900}),
])
def test_layout_random_workloads(name, over):
    w = workloads.make(name, **over)
    got = _check_layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    valid = int((w.topk_idx >= 0).sum())
    assert got["tokens_per_expert"].sum() == valid
    assert got["tokens_per_rank"].sum() == got["is_token_in_rank"].sum()
    assert got["flags"] == 0


def test_layout_counts_duplicate_rank_once_and_flags_bad_expert():
    topk = np.array([[0, 1, 5], [3, 3, -1], [7, 2, 9]], np.int64)  # E=8, R=2 -> 4 experts/rank
    got = oracle.layout(topk, 8, 2)
    assert got["flags"] == oracle.FLAG_BAD_EXPERT
    assert list(got["tokens_per_expert"]) == [1, 1, 1, 2, 0, 1, 0, 1]
    assert got["is_token_in_rank"].tolist() == [[1, 1], [1, 0], [1, 1]]
    assert got["slot"].tolist() == [[0, 0], [1, -1], [2, 1]]
    assert list(got["tokens_per_rank"]) == [3, 2]


# ----------------------------------------------------------------------------- dispatch

def _small(seed=3, T=37, H=256, E=12, R=3, k=3, drop=0.15):
    rng = np.random.Generator(np.random.PCG64(seed))
    topk = workloads.routing_uniform(rng, T, E, k)
    topk[rng.random(topk.shape) < drop] = -1
    x = workloads.bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    w = rng.random((T, k), dtype=np.float32)
    return x, topk, w


def test_dispatch_is_a_stable_partition():
    x, topk, w = _small()
    E, R, T, k = 12, 3, x.shape[0], topk.shape[1]
    L = oracle.layout(topk, E, R)
    D = oracle.dispatch(x, topk, w, L["slot"], E, R, T, fill_x=0xFFFF, fill_idx=-7, fill_w=-9.0)
    assert D["flags"] == 0
    for r in range(R):
        dest = np.nonzero(L["is_token_in_rank"][:, r])[0]          # tokens in ascending order
        n = len(dest)
        assert np.array_equal(D["recv_src_idx"][r, :n], dest)
        assert np.all(D["recv_src_idx"][r, n:] == -7)
        assert np.array_equal(D["recv_x"][r, :n], x[dest])
        assert np.all(D["recv_x"][r, n:] == 0xFFFF)
        for s, t in enumerate(dest):
            for j in range(k):
                e = topk[t, j]
                local = e - r * (E // R) if (e >= 0 and e // (E // R) == r) else -1
                assert D["recv_topk_idx"][r, s, j] == local
                assert D["recv_topk_w"][r, s, j] == (w[t, j] if local >= 0 else 0.0)
    # every (t, r) pair delivered exactly once
    pairs = [(int(D["recv_src_idx"][r, s]), r) for r in range(R) for s in range(L["tokens_per_rank"][r])]
    assert len(pairs) == len(set(pairs)) == int(L["is_token_in_rank"].sum())


def test_dispatch_capacity_drops_and_flags():
    x, topk, w = _small(seed=4)
    E, R = 12, 3
    L = oracle.layout(topk, E, R)
    cap = int(L["tokens_per_rank"].max()) - 3
    D = oracle.dispatch(x, topk, w, L["slot"], E, R, cap, fill_x=0xABCD)
    assert D["flags"] == oracle.FLAG_CAPACITY
    full = oracle.dispatch(x, topk, w, L["slot"], E, R, int(L["tokens_per_rank"].max()))
    for r in range(R):
        n = min(cap, int(L["tokens_per_rank"][r]))
        assert np.array_equal(D["recv_x"][r, :n], full["recv_x"][r, :n])
        assert np.all(D["recv_x"][r, n:] == 0xABCD)


def test_dispatch_fp8_rows_are_quantised_sources():
    x, topk, w = _small(seed=5, H=384)
    E, R, T = 12, 3, x.shape[0]
    L = oracle.layout(topk, E, R)
    D = oracle.dispatch(x, topk, w, L["slot"], E, R, T, fp8=True)
    for r in range(R):
        for s in range(int(L["tokens_per_rank"][r])):
            q, sc = oracle.quantize_row_e4m3(x[D["recv_src_idx"][r, s]])
            assert np.array_equal(D["recv_x"][r, s], q)
            assert np.array_equal(D["recv_scales"][r, s], sc)


# ----------------------------------------------------------------------------- restripe

def test_restripe_is_an_index_swap_with_inverse():
    rng = np.random.Generator(np.random.PCG64(9))
    T, N, P, M = 53, 5, 12, 64
    prob = rng.random((T, N, P), dtype=np.float32)
    out = oracle.restripe_prob(prob, M, fill=-1.0)
    assert np.array_equal(out[:, :T, :], prob.transpose(1, 0, 2))
    assert np.all(out[:, T:, :] == -1.0)
    # same bytes: the multiset of values is unchanged
    assert np.array_equal(np.sort(out[:, :T].ravel()), np.sort(prob.ravel()))
    # restriping the [N][T][P] staging rows back (N "tokens" of T "nodes", capacity N) is the inverse
    back = oracle.restripe_prob(np.ascontiguousarray(out[:, :T, :]), N)
    assert np.array_equal(back, prob)


# ----------------------------------------------------------------------------- node dispatch

def test_node_dispatch_dense_sparse_and_runs():
    w = workloads.make("restripe", T=300, H=64, P=8, chunk_tokens=32)
    T, N = w.T, w.num_nodes
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    in_node = L["is_token_in_node"]
    assert np.all((in_node.sum(1) >= 1) & (in_node.sum(1) <= 4))
    staging = oracle.restripe_prob(w.prob, T)
    dense = oracle.dispatch_nodes(w.x, staging, in_node, T, 32, dense=True, fill_x=0x7777, fill_prob=-2.0)
    sparse = oracle.dispatch_nodes(w.x, staging, in_node, T, 32, dense=False, fill_x=0x7777, fill_prob=-2.0)
    for n in range(N):
        assert np.array_equal(dense["recv_x_node"][n], w.x)
        assert np.array_equal(dense["recv_prob_node"][n], w.prob[:, n, :])
        m = in_node[:, n].astype(bool)
        assert np.array_equal(sparse["recv_x_node"][n][m], w.x[m])
        assert np.all(sparse["recv_x_node"][n][~m] == 0x7777)
        assert np.array_equal(sparse["recv_prob_node"][n][m], w.prob[m, n, :])
        assert np.all(sparse["recv_prob_node"][n][~m] == -2.0)
        for c in range(dense["num_runs"].shape[1]):
            seg = in_node[c * 32:(c + 1) * 32, n].astype(np.int64)
            starts = int(np.sum(np.diff(np.concatenate([[0], seg])) == 1))
            assert sparse["num_runs"][n, c] == starts
            assert dense["num_runs"][n, c] == 1


# ----------------------------------------------------------------------------- combine

def _bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_combine_identity_expert_closed_form():
    """y = recv_x (identity) => out = bf16(n_ranks(t) * x), exact since n <= 8."""
    w = workloads.make("tiny")
    L = oracle.layout(w.topk_idx, w.E, w.R)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, w.max_tokens)
    out, flags = oracle.combine(D["recv_x"], L["slot"], w.max_tokens)
    n = L["is_token_in_rank"].sum(1).astype(np.float32)
    exp = (_bf16_tensor(w.x).float() * torch.from_numpy(n)[:, None]).to(torch.bfloat16)
    assert flags == 0
    assert np.array_equal(out, exp.view(torch.int16).numpy().view(np.uint16))


def test_combine_sums_in_ascending_rank_order():
    rng = np.random.Generator(np.random.PCG64(12))
    T, H, R, M = 9, 32, 4, 9
    slot = np.full((T, R), -1, np.int32)
    cnt = [0] * R
    for t in range(T):
        for r in range(R):
            if rng.random() < 0.6:
                slot[t, r] = cnt[r]
                cnt[r] += 1
    slot[0, :] = -1  # a token routed nowhere
    # magnitudes spread so that the order of the fp32 additions matters
    y = workloads.bf16_bits((rng.standard_normal((R, M, H)) * 10.0 ** rng.integers(-3, 4, (R, M, H))).astype(np.float32))
    out, flags = oracle.combine(y, slot, M)
    yf = _bf16_tensor(y).float().numpy()
    for t in range(T):
        acc = np.zeros(H, np.float32)
        for r in range(R):
            if slot[t, r] >= 0:
                acc = (acc + yf[r, slot[t, r]]).astype(np.float32)
        exp = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[t], exp)
    assert np.all(out[0] == 0)
    assert flags == 0


def test_combine_order_is_ascending_on_a_crafted_token():
    """(2^24 + 1) rounds to 2^24 in fp32 (tie to even), so the rank order shows in the result:
    ascending ((0 + 2^24) + 1) + -2^24 = 0, descending ((0 - 2^24) + 1) + 2^24 = 1."""
    H, R = 8, 3
    vals = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    y = np.stack([workloads.bf16_bits(np.full((1, H), v, np.float32)) for v in vals])  # [R][1][H]
    slot = np.zeros((1, R), np.int32)
    out, _ = oracle.combine(y, slot, 1)
    assert np.all(out == 0x0000)
    # reversing the rank roles (the same rows fed as ranks 2, 1, 0) gives 1.0
    out_rev, _ = oracle.combine(np.ascontiguousarray(y[::-1]), slot, 1)
    assert np.all(out_rev == 0x3F80)


def test_combine_single_rank_is_a_copy_and_capacity_flag():
    rng = np.random.Generator(np.random.PCG64(13))
    T, H = 20, 64
    y = workloads.bf16_bits(rng.standard_normal((1, T, H), dtype=np.float32))
    slot = np.arange(T, dtype=np.int32)[:, None]
    out, flags = oracle.combine(y, slot, T)
    assert np.array_equal(out, y[0]) and flags == 0
    out, flags = oracle.combine(y[:, :10], slot, 10)
    assert flags == oracle.FLAG_CAPACITY
    assert np.array_equal(out[:10], y[0, :10]) and np.all(out[10:] == 0)


def test_pipeline_with_weighted_expert_returns_x():
    """With the x * sum(w) expert and weights summing to 1, combine returns x to a few bf16 ulp."""
    w = workloads.make("dsv3", T=256, H=512)
    L = oracle.layout(w.topk_idx, w.E, w.R, w.ranks_per_node)
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, w.max_tokens)
    y = oracle.expert_scale(D["recv_x"], D["recv_topk_w"], L["tokens_per_rank"])
    # the expert restated with torch: bf16(x * w_r), w_r summed in j order
    for r in range(w.R):
        n = int(L["tokens_per_rank"][r])
        wr = torch.zeros(n)
        for j in range(w.k):
            wr = wr + torch.from_numpy(D["recv_topk_w"][r, :n, j])
        exp = (_bf16_tensor(D["recv_x"][r, :n]).float() * wr[:, None]).to(torch.bfloat16)
        assert np.array_equal(y[r, :n], exp.view(torch.int16).numpy().view(np.uint16))
    out, _ = oracle.combine(y, L["slot"], w.max_tokens)
    xo = _bf16_tensor(out).float()
    xi = _bf16_tensor(w.x).float()
    assert torch.all((xo - xi).abs() <= 4 * 2.0 ** -8 * xi.abs() + 1e-30)
