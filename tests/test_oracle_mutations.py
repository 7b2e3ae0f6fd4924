"""Plant plausible mistakes in a copy of the oracle and check the pins catch each one.

Every mutation is compiled from a patched copy of oracle/ep_oracle.c into a
temporary library (CPU only) and swapped in for the real one while the named
pin tests run; each pin set must fail on its mutant.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_formats as F
import test_oracle_pages as G
import test_oracle_path as PTH
import test_oracle_permuted as PERM
import test_oracle_combine_variants as CV
import test_oracle_split_combine as SPL

MUTATIONS = [
    ("bf16 ties away from even",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
     "if (lower >= 0x8000u) upper += 1u;",
     [F.test_bf16_special_values]),
    ("e4m3 ties round up",
     "if (frac > 0.5 || (frac == 0.5 && (nn & 1u))) nn += 1u;",
     "if (frac >= 0.5) nn += 1u;",
     [F.test_e4m3_encode_brute_force_on_midpoints_and_neighbours]),
    ("e4m3 exponent bias off by one",
     "code = ((uint32_t)(ex + 7) << 3) | (nn - 8u);",
     "code = ((uint32_t)(ex + 8) << 3) | (nn - 8u);",
     [F.test_e4m3_encode_matches_torch_on_random_in_range_values]),
    ("fp8 scale uses 447",
     "float scale = amax / 448.0f;",
     "float scale = amax / 447.0f;",
     [F.test_fp8_row_matches_torch_restatement]),
    ("fp8 quantises with x * (1/scale)",
     "code = oracle_f32_to_e4m3(v / scale);",
     "code = oracle_f32_to_e4m3(v * (1.0f / scale));",
     [F.test_fp8_row_matches_torch_restatement]),
    ("layout slot is inclusive",
     "slot[i] = tokens_per_rank[r]; /* tokens already counted before t */",
     "slot[i] = tokens_per_rank[r] + 1;",
     [PTH.test_layout_exhaustive_tiny]),
    ("layout counts a rank once per expert",
     "hit[e / experts_per_rank] = 1;",
     "hit[e / experts_per_rank] = 1; if (0) {}",
     None),  # not a behaviour change: control that the harness itself passes
    ("dispatch local id off by one rank",
     "? (int32_t)(e - (int64_t)r * experts_per_rank) : -1;",
     "? (int32_t)(e - (int64_t)(r + 1) * experts_per_rank) : -1;",
     [PTH.test_dispatch_is_a_stable_partition]),
    ("dispatch ignores capacity",
     "if (s >= max_tokens) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            size_t row",
     "if (s >= max_tokens) {\n                flags |= 0;\n                continue;\n            }\n            size_t row",
     [PTH.test_dispatch_capacity_drops_and_flags]),
    ("restripe transposed",
     "out[((size_t)n * max_tokens + t) * P + p] = prob[((size_t)t * N + n) * P + p];",
     "out[((size_t)n * max_tokens + t) * P + p] = prob[((size_t)n * T + t) * P + p];",
     [PTH.test_restripe_is_an_index_swap_with_inverse]),
    ("sparse path counts tokens instead of runs",
     "runs += 1;",
     "runs += t - start;",
     [PTH.test_node_dispatch_dense_sparse_and_runs]),
    ("sparse run drops its last token",
     "copy_token_range(x, prob_staging, H, P, max_tokens, n, start, t, recv_x_node,",
     "copy_token_range(x, prob_staging, H, P, max_tokens, n, start, t - 1, recv_x_node,",
     [PTH.test_node_dispatch_dense_sparse_and_runs]),
    ("combine in descending rank order",
     "for (int32_t r = 0; r < R; ++r) {\n            int32_t s = slot[(size_t)t * R + r];\n            if (s < 0) continue;\n            if (s >= max_tokens) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            const uint16_t* row",
     "for (int32_t r = R - 1; r >= 0; --r) {\n            int32_t s = slot[(size_t)t * R + r];\n            if (s < 0) continue;\n            if (s >= max_tokens) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            const uint16_t* row",
     [PTH.test_combine_order_is_ascending_on_a_crafted_token]),
    ("combine accumulates in bf16",
     "for (int32_t h = 0; h < H; ++h) acc[h] = acc[h] + oracle_bf16_to_f32(row[h]);",
     "for (int32_t h = 0; h < H; ++h) acc[h] = oracle_bf16_to_f32(oracle_f32_to_bf16(acc[h] + oracle_bf16_to_f32(row[h])));",
     [PTH.test_combine_sums_in_ascending_rank_order]),
    ("expert slot counts from 1",
     "out = cnt[e];",
     "out = cnt[e] + 1;",
     [PERM.test_expert_layout_matches_stable_sort_restatement]),
    ("expert layout keeps repeated ids",
     "if (topk_idx[(size_t)t * k + jj] == e) repeat = 1;",
     "if (0) repeat = 1;",
     [PERM.test_expert_layout_repeats_and_out_of_range_are_dropped_and_flagged]),
    ("permuted row ignores the rank's first expert offset",
     "return expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];",
     "return expert_offsets[e] - expert_offsets[0 * epr + r * 0] + expert_slot[(size_t)t * k + j];",
     [PERM.test_dispatch_permuted_groups_rows_by_local_expert_in_token_order]),
    ("weighted combine drops the weight",
     "if (topk_w != NULL) term = term * topk_w[(size_t)t * k + j];",
     "if (topk_w != NULL) term = term * 1.0f;",
     [PERM.test_combine_permuted_closed_form_and_brute_force]),
    ("combine from expert slabs sums slots in reverse",
     "        for (int32_t j = 0; j < k; ++j) {\n            if (expert_slot[(size_t)t * k + j] < 0) continue;\n            int64_t e = topk_idx[(size_t)t * k + j];\n            int32_t r = (int32_t)(e / (E / R));\n            int32_t p = permuted_row(expert_offsets, expert_slot, t, j, k, e, E, R);\n            if (p >= max_rows) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            const uint16_t* row",
     "        for (int32_t j = k - 1; j >= 0; --j) {\n            if (expert_slot[(size_t)t * k + j] < 0) continue;\n            int64_t e = topk_idx[(size_t)t * k + j];\n            int32_t r = (int32_t)(e / (E / R));\n            int32_t p = permuted_row(expert_offsets, expert_slot, t, j, k, e, E, R);\n            if (p >= max_rows) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            const uint16_t* row",
     [PERM.test_combine_permuted_term_order_is_the_topk_order]),
    ("fp8 combine reads the next block's scale",
     "float v = oracle_e4m3_to_f32(y[yr * H + h]) * y_scales[yr * nb + h / 128];",
     "float v = oracle_e4m3_to_f32(y[yr * H + h]) * y_scales[yr * nb + (h / 128 + 1) % nb];",
     [CV.test_combine_fp8_exact_closed_form_with_power_of_two_scales]),
    ("fp8 combine in descending rank order",
     "for (int32_t r = 0; r < R; ++r) {\n            int32_t s = slot[(size_t)t * R + r];\n            if (s < 0) continue;\n            if (s >= max_tokens) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            size_t yr = (size_t)r * max_tokens + s;\n            for (int32_t h = 0; h < H; ++h) {\n                float v",
     "for (int32_t r = R - 1; r >= 0; --r) {\n            int32_t s = slot[(size_t)t * R + r];\n            if (s < 0) continue;\n            if (s >= max_tokens) {\n                flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            size_t yr = (size_t)r * max_tokens + s;\n            for (int32_t h = 0; h < H; ++h) {\n                float v",
     [CV.test_combine_fp8_order_is_ascending_on_a_crafted_token]),
    ("combined weights keep the last rank's row",
     "out[(size_t)t * k + j] = out[(size_t)t * k + j] + w[j];",
     "out[(size_t)t * k + j] = w[j];",
     [CV.test_combined_weights_return_the_router_weights]),
    ("combined weights lose the capacity flag",
     "flags |= ORACLE_FLAG_CAPACITY;\n                continue;\n            }\n            const float* w",
     "flags |= 0;\n                continue;\n            }\n            const float* w",
     [CV.test_combined_weights_drop_capacity_and_sum_in_rank_order]),
    ("combine send drops the weight",
     "if (recv_topk_w != NULL) term = term * recv_topk_w[row * k + j];",
     "if (recv_topk_w != NULL) term = term * 1.0f;",
     [SPL.test_combine_send_power_of_two_weights_closed_form]),
    ("combine send sums slots in reverse",
     "            for (int32_t j = 0; j < k; ++j) {\n                int32_t l = recv_topk_idx[row * k + j];\n                if (l < 0 || expert_slot[(size_t)t * k + j] < 0) continue;\n                int32_t e = r * epr + l;\n                int32_t p = expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];\n                if (p >= max_rows) {\n                    flags |= ORACLE_FLAG_CAPACITY;\n                    continue;\n                }\n                const uint16_t* src",
     "            for (int32_t j = k - 1; j >= 0; --j) {\n                int32_t l = recv_topk_idx[row * k + j];\n                if (l < 0 || expert_slot[(size_t)t * k + j] < 0) continue;\n                int32_t e = r * epr + l;\n                int32_t p = expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];\n                if (p >= max_rows) {\n                    flags |= ORACLE_FLAG_CAPACITY;\n                    continue;\n                }\n                const uint16_t* src",
     [SPL.test_combine_send_term_order_is_the_slot_order]),
    ("combine send indexes rank 0's expert offsets",
     "int32_t p = expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];\n                if (p >= max_rows) {\n                    flags |= ORACLE_FLAG_CAPACITY;\n                    continue;\n                }\n                const uint16_t* src",
     "int32_t p = expert_offsets[e] - expert_offsets[0] + expert_slot[(size_t)t * k + j];\n                if (p >= max_rows) {\n                    flags |= ORACLE_FLAG_CAPACITY;\n                    continue;\n                }\n                const uint16_t* src",
     [SPL.test_combine_send_inverts_the_receive_side_permute, SPL.test_combine_send_identity_rows_closed_form]),
    ("combine send accumulates in bf16",
     "if (recv_topk_w != NULL) term = term * recv_topk_w[row * k + j];\n                    acc[h] = acc[h] + term;",
     "if (recv_topk_w != NULL) term = term * recv_topk_w[row * k + j];\n                    acc[h] = oracle_bf16_to_f32(oracle_f32_to_bf16(acc[h] + term));",
     [SPL.test_combine_send_power_of_two_weights_closed_form]),
    ("combine send loses the capacity flag",
     "flags |= ORACLE_FLAG_CAPACITY;\n                    continue;\n                }\n                const uint16_t* src",
     "flags |= 0;\n                    continue;\n                }\n                const uint16_t* src",
     [SPL.test_combine_send_capacity_drops_and_flags]),
    ("expert drops the last weight",
     "for (int32_t j = 0; j < k; ++j) w = w + recv_topk_w[row * k + j];",
     "for (int32_t j = 0; j + 1 < k; ++j) w = w + recv_topk_w[row * k + j];",
     [PTH.test_pipeline_with_weighted_expert_returns_x]),
]


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    d = tmp_path / "mut"
    d.mkdir(exist_ok=True)
    (d / "ep_oracle.h").write_text(open(os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.h")).read())
    (d / "ep_oracle.c").write_text(src.replace(old, new))
    so = d / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(d / "ep_oracle.c"), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new, pins):
    real = oracle._load()
    so = _build_mutant(tmp_path, old, new)
    mutant = ctypes.CDLL(so)
    # give the mutant the same signatures as the real library
    for sym in ("oracle_f32_to_bf16", "oracle_bf16_to_f32", "oracle_f32_to_e4m3", "oracle_e4m3_to_f32",
                "oracle_quantize_row_e4m3", "oracle_layout", "oracle_dispatch", "oracle_restripe_prob",
                "oracle_dispatch_nodes", "oracle_combine", "oracle_expert_scale", "oracle_expert_layout",
                "oracle_dispatch_permuted", "oracle_permute_received", "oracle_combine_permuted",
                "oracle_combine_fp8", "oracle_combine_weights", "oracle_combine_send"):
        f_real, f_mut = getattr(real, sym), getattr(mutant, sym)
        f_mut.restype, f_mut.argtypes = f_real.restype, f_real.argtypes
    monkeypatch.setattr(oracle, "_lib", mutant)
    if pins is None:  # control: an equivalent rewrite passes the layout pins
        PTH.test_layout_exhaustive_tiny()
        G.test_dispatch_bytes_match_printed_time_times_bandwidth()
        return
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()
