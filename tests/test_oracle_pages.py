"""Pin the oracle's byte accounting to figures the DeepEP pages print.

The pages print dispatch/combine kernel times and bandwidths (fixture:
tests/golden/pages_dispatch_bytes.json, each case with its citation). time x
bandwidth is the bytes one call moved. The oracle must reproduce it as
(number of (token, destination node) pairs from its layout) x (bytes of one
receive row from its dispatch output: 2H for bf16, H + 4 H/128 for the FP8
row with its per-128-channel fp32 scales), within the precision of the
printed digits. A token sent once per expert instead of once per node, or a
different FP8 scale granularity, misses by several percent.
"""
import json
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_dispatch_bytes.json")


def _half_unit(s: str) -> float:
    """Half a unit of the last printed digit, relative to the printed value."""
    dec = len(s.split(".")[1]) if "." in s else 0
    return 0.5 * 10.0 ** (-dec) / float(s)


def _row_bytes(H: int, fp8: bool) -> int:
    """Bytes of one receive row, read off the oracle's dispatch output buffers."""
    x = np.zeros((1, H), np.uint16)
    topk = np.array([[0]], np.int64)
    L = oracle.layout(topk, 1, 1)
    D = oracle.dispatch(x, topk, np.ones((1, 1), np.float32), L["slot"], 1, 1, 1, fp8=fp8)
    n = D["recv_x"][0, 0].nbytes
    if fp8:
        n += D["recv_scales"][0, 0].nbytes
    return n


def test_dispatch_bytes_match_printed_time_times_bandwidth():
    g = json.load(open(GOLDEN))
    T_sim = 16 * g["tokens"]  # a larger sample keeps routing noise near 0.1 %
    rng = np.random.Generator(np.random.PCG64(2024))
    topk = workloads.routing_uniform(rng, T_sim, g["experts"], g["topk"])
    for case in g["cases"]:
        R = case["nodes"] * g["ranks_per_node"]
        L = oracle.layout(topk, g["experts"], R, g["ranks_per_node"])
        pairs_per_token = L["tokens_per_node"].sum() / T_sim
        ours = pairs_per_token * g["tokens"] * _row_bytes(g["hidden"], case["dtype"] == "fp8")
        page = float(case["time_us"]) * 1e-6 * float(case["bw_gbs"]) * 1e9
        tol = _half_unit(case["time_us"]) + _half_unit(case["bw_gbs"]) + 0.002
        assert abs(ours - page) / page <= tol, (case["cite"], ours, page)


def test_fp8_row_is_h_plus_per_128_scales():
    assert _row_bytes(7168, True) == 7168 + 56 * 4
    assert _row_bytes(7168, False) == 7168 * 2
