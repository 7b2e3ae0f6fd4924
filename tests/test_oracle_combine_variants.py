"""Pins for the oracle's combine variants: the combine of FP8 rows and the combined top-k
weights.

FP8 rows: with power-of-two block scales and codes whose values lie in [2^-2, 60], every
dequantised value and every partial sum of up to 32 of them is exact in fp32, so the
result is the exact (float64) sum of the values, rounded once to bf16; the values are
decoded by torch's float8_e4m3fn, not by the oracle. A crafted token shows the rank
order; random rows are checked against a numpy float32 running sum; dropped slots are
flagged.

Weights: after a dispatch, the combined weights of every token are the router's
weights, bit for bit (exactly one rank holds each slot's weight, the others hold +0),
and 0 where a slot was empty or its rank was dropped for capacity.
"""
import numpy as np
import torch

import oracle
import workloads


def _e4m3_values(codes):
    """float64 values of E4M3 codes, decoded by torch."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _bf16_of_f64(v):
    """bf16 bits of float64 values that are exact in fp32 (one rounding, by torch)."""
    f = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64)).to(torch.float32)
    assert torch.equal(f.to(torch.float64), torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64)))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _random_slots(rng, T, R, p=0.5):
    slot = np.full((T, R), -1, np.int32)
    cnt = [0] * R
    for t in range(T):
        for r in range(R):
            if rng.random() < p:
                slot[t, r] = cnt[r]
                cnt[r] += 1
    return slot, max(cnt + [1])


def test_combine_fp8_exact_closed_form_with_power_of_two_scales():
    rng = np.random.Generator(np.random.PCG64(41))
    T, H, R = 40, 384, 32
    slot, M = _random_slots(rng, T, R)
    slot[3, :] = -1  # a token routed nowhere
    # normal codes with exponent field 5..12 (values 2^-2 .. 60), either sign
    exp_field = rng.integers(5, 13, (R, M, H))
    mant = rng.integers(0, 8, (R, M, H))
    sign = rng.integers(0, 2, (R, M, H))
    codes = ((sign << 7) | (exp_field << 3) | mant).astype(np.uint8)
    scales = (2.0 ** rng.integers(-1, 2, (R, M, H // 128))).astype(np.float32)
    out, flags = oracle.combine_fp8(codes, scales, slot, M)
    vals = _e4m3_values(codes) * np.repeat(scales.astype(np.float64), 128, axis=2)
    exp = np.zeros((T, H), np.float64)
    for t in range(T):
        for r in range(R):
            if slot[t, r] >= 0:
                exp[t] += vals[r, slot[t, r]]
    assert flags == 0
    assert np.array_equal(out, _bf16_of_f64(exp))
    assert np.all(out[3] == 0)


def test_combine_fp8_order_is_ascending_on_a_crafted_token():
    """256 * 2^16 = 2^24: ascending ((0 + 2^24) + 1) - 2^24 = 0 (2^24 + 1 ties to 2^24),
    descending ((0 - 2^24) + 1) + 2^24 = 1."""
    H, R = 128, 3
    codes = np.stack([np.full((1, H), c, np.uint8) for c in (0x78, 0x38, 0xF8)])  # 256, 1, -256
    scales = np.array([[[65536.0]], [[1.0]], [[65536.0]]], np.float32)
    assert np.array_equal(_e4m3_values(codes[:, 0, 0]), [256.0, 1.0, -256.0])
    slot = np.zeros((1, R), np.int32)
    out, _ = oracle.combine_fp8(codes, scales, slot, 1)
    assert np.all(out == 0x0000)
    out_rev, _ = oracle.combine_fp8(np.ascontiguousarray(codes[::-1]), np.ascontiguousarray(scales[::-1]), slot, 1)
    assert np.all(out_rev == 0x3F80)


def test_combine_fp8_random_rows_match_a_float32_running_sum_and_flag_capacity():
    rng = np.random.Generator(np.random.PCG64(42))
    T, H, R = 25, 256, 6
    slot, M = _random_slots(rng, T, R, p=0.7)
    codes = rng.integers(0, 256, (R, M, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x40  # no NaN codes
    scales = np.exp(rng.uniform(-12, 4, (R, M, H // 128))).astype(np.float32)
    out, flags = oracle.combine_fp8(codes, scales, slot, M)
    vals = (_e4m3_values(codes).astype(np.float32) * np.repeat(scales, 128, axis=2)).astype(np.float32)
    for t in range(T):
        acc = np.zeros(H, np.float32)
        for r in range(R):
            if slot[t, r] >= 0:
                acc = (acc + vals[r, slot[t, r]]).astype(np.float32)
        assert np.array_equal(out[t], torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    assert flags == 0
    cap = max(1, M // 2)
    _, flags = oracle.combine_fp8(codes[:, :cap], scales[:, :cap], slot, cap)
    assert flags == oracle.FLAG_CAPACITY


def test_combined_weights_return_the_router_weights():
    for name, over in (("restripe", {"T": 300, "H": 8}), ("dsv3", {"T": 300, "H": 8}), ("skewed", {"T": 300, "H": 8})):
        w = workloads.make(name, **over)
        L = oracle.layout(w.topk_idx, w.E, w.R)
        M = w.max_tokens or w.T  # the skewed workload sizes its slabs from the layout
        D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, M)
        got, flags = oracle.combine_weights(D["recv_topk_w"], L["slot"], M)
        exp = np.where((w.topk_idx >= 0) & (w.topk_idx < w.E), w.topk_w, np.float32(0)).astype(np.float32)
        assert flags == 0
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), name


def test_combined_weights_drop_capacity_and_sum_in_rank_order():
    w = workloads.make("skewed", T=400, H=8)
    L = oracle.layout(w.topk_idx, w.E, w.R)
    M = int(L["tokens_per_rank"].max()) // 2
    D = oracle.dispatch(w.x, w.topk_idx, w.topk_w, L["slot"], w.E, w.R, M)
    got, flags = oracle.combine_weights(D["recv_topk_w"], L["slot"], M)
    assert flags == oracle.FLAG_CAPACITY
    epr = w.E // w.R
    for t in range(w.T):
        for j in range(w.k):
            e = int(w.topk_idx[t, j])
            kept = 0 <= e < w.E and 0 <= L["slot"][t, e // epr] < M
            assert got[t, j] == (w.topk_w[t, j] if kept else 0.0)
    # three ranks holding 2^24, 1, -2^24 for one slot: the ascending sum is 0, not 1
    rw = np.array([[[2.0 ** 24]], [[1.0]], [[-(2.0 ** 24)]]], np.float32)
    got, _ = oracle.combine_weights(rw, np.zeros((1, 3), np.int32), 1)
    assert got[0, 0] == 0.0
    got, _ = oracle.combine_weights(np.ascontiguousarray(rw[::-1]), np.zeros((1, 3), np.int32), 1)
    assert got[0, 0] == 1.0
