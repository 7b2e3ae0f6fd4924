/*
 * ep_oracle.c -- the oracle for the expert-parallel (EP) dispatch/combine path.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg load it; nothing on the product path
 * does. It shares no code with the CUDA library.
 *
 * Every routine is the plain definition of its step, written as slowly and
 * plainly as possible: one token at a time, one rank at a time, one element at
 * a time, in the order the definition states. Floating point is IEEE-754
 * binary32 with round-to-nearest-even and no contraction (built with
 * -ffp-contract=off; FLT_EVAL_METHOD must be 0).
 *
 * Sources (DeepEP pull-request pages):
 *   [PR #347] "Feature/sm free normal kernel": section 2.1 Feature (dispatch
 *     sends each token to the ranks it routes to, combine brings the expert
 *     outputs back), section 3.1 Experiment Setup (4096 tokens, hidden 7168,
 *     top-8), section 3.2.1 tables (FP8 and BF16 dispatch, BF16 combine), and
 *     the commit "add arg return_recv_hook for get_dispatch_layout" (the
 *     routing-layout step).
 *   [PR #634] "Hybrid ep nixl restripe": sections "Baseline problem" and "Fix"
 *     (prob layouts, the restripe, dense puts per (chunk, destination) and one
 *     put per run on the sparse path, NUM_OF_TOKENS_PER_CHUNK = 256), section
 *     "Receive-side and DOCA path are unchanged" (local slice at
 *     node_rank x MAX_TOKENS, per-token stride prob_per_token), and the commit
 *     "fix scan permute-fusion local-experts sum array sizing" (the scan).
 *   [PR #453] "Higher Performance with Lower SM Occupancy through Zero-Copy and
 *     TMA Offloading": commit "Add assertion against too large recv token
 *     count" (the capacity check).
 * Readings where the pages are silent are stated at each routine.
 */
#include "ep_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bfloat16 is the upper half of a binary32. Rounding keeps the upper 16 bits
 * and rounds on the lower 16: up when they exceed half, to the even upper half
 * on an exact tie. A carry out of the mantissa correctly bumps the exponent
 * (the largest finite values round up to infinity). NaN stays NaN (quiet bit
 * set). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Value of an OCP E4M3 code: sign, 4-bit exponent with bias 7, 3-bit mantissa.
 * Exponent field 0 holds the subnormals m * 2^-9; field 15 with mantissa 7 is
 * NaN (there are no infinities). */
float oracle_e4m3_to_f32(uint8_t q) {
    int s = q >> 7;
    int e = (q >> 3) & 0xF;
    int m = q & 0x7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 7 - 3);
    return (float)(s ? -v : v);
}

/* binary32 -> E4M3, round to nearest (ties to the even code), saturating:
 * every finite or infinite magnitude above the largest finite value 448 gives
 * +-448; NaN gives the NaN code. The result is found by scaling |f| by the
 * quantum of its binade (a power of two, so the scaling is exact in double)
 * and rounding the quotient to an integer by hand. */
uint8_t oracle_f32_to_e4m3(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    if (f != f) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)f);
    if (a > 448.0) return (uint8_t)(sign | 0x7E);

    int subnormal = a < ldexp(1.0, -6);
    int ex = -6; /* binade exponent: 2^ex <= a < 2^(ex+1) for normals */
    double quantum;
    if (subnormal) {
        quantum = ldexp(1.0, -9);
    } else {
        int e2;
        (void)frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1) */
        ex = e2 - 1;
        quantum = ldexp(1.0, ex - 3);
    }
    double n = a / quantum; /* exact */
    double fl = floor(n);
    double frac = n - fl;
    uint32_t nn = (uint32_t)fl;
    if (frac > 0.5 || (frac == 0.5 && (nn & 1u))) nn += 1u;

    uint32_t code;
    if (subnormal) {
        code = nn; /* 0..8; 8 is the smallest normal 2^-6, whose code is also 8 */
    } else {
        if (nn == 16u) { /* rounded up into the next binade */
            ex += 1;
            nn = 8u;
        }
        code = ((uint32_t)(ex + 7) << 3) | (nn - 8u);
    }
    return (uint8_t)(sign | code);
}

/* Per-token 1x128 quantisation of one row (the FP8 dispatch row format: H
 * e4m3 bytes plus one fp32 scale per 128 channels, the 7168 + 56 x 4 bytes a
 * token that the FP8 dispatch rows of [PR #347] section 3.2.1 move):
 *   amax  = max |x_i| over the 128 channels of the block (exact in fp32)
 *   scale = amax / 448                   (one binary32 division)
 *   q_i   = e4m3_rn_satfinite(x_i / scale) (one division, one rounding)
 * Reading: a block whose amax is 0 stores scale 0 and the signed zero code of
 * each element (0x00 for +0, 0x80 for -0), which is what x_i / scale gives for
 * a zero x_i in any block with a positive scale. */
void oracle_quantize_row_e4m3(const uint16_t* x, int32_t H, uint8_t* q, float* scales) {
    int32_t nb = H / 128;
    for (int32_t b = 0; b < nb; ++b) {
        float amax = 0.0f;
        for (int32_t i = 0; i < 128; ++i) {
            float v = fabsf(oracle_bf16_to_f32(x[b * 128 + i]));
            if (v > amax) amax = v;
        }
        float scale = amax / 448.0f;
        scales[b] = scale;
        for (int32_t i = 0; i < 128; ++i) {
            float v = oracle_bf16_to_f32(x[b * 128 + i]);
            uint8_t code;
            if (amax == 0.0f)
                code = signbit(v) ? 0x80 : 0x00;
            else
                code = oracle_f32_to_e4m3(v / scale);
            q[b * 128 + i] = code;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Routing layout                                                            */
/* ------------------------------------------------------------------------- */

/* The layout step ("get_dispatch_layout", [PR #347] commit list) reads the
 * router's top-k expert ids and produces, in token order:
 *   tokens_per_expert[e] = number of (t, j) with topk_idx[t][j] == e
 *   is_token_in_rank[t][r] = 1 when any of token t's experts lives on rank r
 *   tokens_per_rank[r] = number of tokens t with is_token_in_rank[t][r]
 *   slot[t][r] = #{t' < t : is_token_in_rank[t'][r]} (a stable exclusive prefix
 *                sum down the tokens), or -1 when token t does not go to rank r
 *   is_token_in_node / tokens_per_node likewise at node granularity (only when
 *   ranks_per_node > 0).
 * Readings: experts sit on ranks in contiguous blocks (rank = e / (E/R)); a
 * token with several experts on one rank goes to that rank once. */
int32_t oracle_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                      int32_t ranks_per_node, int32_t* tokens_per_expert,
                      int32_t* tokens_per_rank, int32_t* tokens_per_node,
                      uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot) {
    int32_t flags = 0;
    int32_t experts_per_rank = E / R;
    int32_t N = ranks_per_node > 0 ? R / ranks_per_node : 0;
    uint8_t* hit = (uint8_t*)calloc((size_t)R, 1);

    for (int32_t e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int32_t r = 0; r < R; ++r) tokens_per_rank[r] = 0;
    for (int32_t n = 0; n < N; ++n) tokens_per_node[n] = 0;

    for (int32_t t = 0; t < T; ++t) {
        memset(hit, 0, (size_t)R);
        for (int32_t j = 0; j < k; ++j) {
            int64_t e = topk_idx[(size_t)t * k + j];
            if (e < 0) continue;
            if (e >= E) {
                flags |= ORACLE_FLAG_BAD_EXPERT;
                continue;
            }
            tokens_per_expert[e] += 1;
            hit[e / experts_per_rank] = 1;
        }
        for (int32_t r = 0; r < R; ++r) {
            size_t i = (size_t)t * R + r;
            is_token_in_rank[i] = hit[r];
            if (hit[r]) {
                slot[i] = tokens_per_rank[r]; /* tokens already counted before t */
                tokens_per_rank[r] += 1;
            } else {
                slot[i] = -1;
            }
        }
        for (int32_t n = 0; n < N; ++n) {
            uint8_t any = 0;
            for (int32_t r = n * ranks_per_node; r < (n + 1) * ranks_per_node; ++r) any |= hit[r];
            is_token_in_node[(size_t)t * N + n] = any;
            if (any) tokens_per_node[n] += 1;
        }
    }
    free(hit);
    return flags;
}

/* ------------------------------------------------------------------------- */
/* Rank-level dispatch                                                       */
/* ------------------------------------------------------------------------- */

/* Dispatch sends each token once to every rank it routes to ([PR #347] 2.1):
 * for every (t, r) with s = slot[t][r] >= 0, into the destination-major receive
 * buffers of rank r at row s:
 *   recv_x[r][s]           = x[t]          (bf16), or its e4m3 quantisation
 *   recv_scales[r][s][b]   = the block scales     (FP8 only)
 *   recv_src_idx[r][s]     = t
 *   recv_topk_idx[r][s][j] = e_j - r * (E/R) when expert e_j lives on r, else -1
 *   recv_topk_w[r][s][j]   = w_j when expert e_j lives on r, else 0
 * A slot at or beyond max_tokens is dropped and raises ORACLE_FLAG_CAPACITY
 * (the too-large receive-count assertion of [PR #453], as a flag). Rows a rank
 * does not receive are left untouched. */
int32_t oracle_dispatch(const uint16_t* x, int32_t out_fp8, const int64_t* topk_idx,
                        const float* topk_w, const int32_t* slot, int32_t T, int32_t H,
                        int32_t k, int32_t E, int32_t R, int32_t max_tokens, void* recv_x,
                        float* recv_scales, int32_t* recv_src_idx, int32_t* recv_topk_idx,
                        float* recv_topk_w) {
    int32_t flags = 0;
    int32_t experts_per_rank = E / R;
    int32_t nb = H / 128;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j)
            if (topk_idx[(size_t)t * k + j] >= E) flags |= ORACLE_FLAG_BAD_EXPERT;
        for (int32_t r = 0; r < R; ++r) {
            int32_t s = slot[(size_t)t * R + r];
            if (s < 0) continue;
            if (s >= max_tokens) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            size_t row = (size_t)r * max_tokens + (size_t)s;
            if (recv_x != NULL) {
                if (out_fp8) {
                    uint8_t* q = (uint8_t*)recv_x + row * (size_t)H;
                    oracle_quantize_row_e4m3(x + (size_t)t * H, H, q, recv_scales + row * nb);
                } else {
                    uint16_t* dst = (uint16_t*)recv_x + row * (size_t)H;
                    for (int32_t h = 0; h < H; ++h) dst[h] = x[(size_t)t * H + h];
                }
            }
            if (recv_src_idx != NULL) recv_src_idx[row] = t;
            for (int32_t j = 0; j < k; ++j) {
                int64_t e = topk_idx[(size_t)t * k + j];
                int on_rank = e >= 0 && e < E && e / experts_per_rank == r;
                if (recv_topk_idx != NULL)
                    recv_topk_idx[row * k + j] = on_rank ? (int32_t)(e - (int64_t)r * experts_per_rank) : -1;
                if (recv_topk_w != NULL) recv_topk_w[row * k + j] = on_rank ? topk_w[(size_t)t * k + j] : 0.0f;
            }
        }
    }
    return flags;
}

/* ------------------------------------------------------------------------- */
/* Prob restripe                                                             */
/* ------------------------------------------------------------------------- */

/* [PR #634] "Baseline problem" / "Fix": the prob tensor arrives as
 * [num_tokens][num_of_nodes][prob_per_token]; the restripe writes the
 * destination-major staging layout [num_of_nodes][max_tokens][prob_per_token],
 * an index swap that moves every byte once:
 *   out[n][t][p] = prob[t][n][p]   for all t < T, n < N, p < P.
 * Rows t in [T, max_tokens) are not written. All (t, n) slices are copied,
 * routed or not, as the memcpy the restripe replaced did. */
void oracle_restripe_prob(const float* prob, int32_t T, int32_t N, int32_t P,
                          int32_t max_tokens, float* out) {
    for (int32_t t = 0; t < T; ++t)
        for (int32_t n = 0; n < N; ++n)
            for (int32_t p = 0; p < P; ++p)
                out[((size_t)n * max_tokens + t) * P + p] = prob[((size_t)t * N + n) * P + p];
}

/* ------------------------------------------------------------------------- */
/* Node-level dense / sparse dispatch                                        */
/* ------------------------------------------------------------------------- */

static void copy_token_range(const uint16_t* x, const float* prob_staging, int32_t H, int32_t P,
                             int32_t max_tokens, int32_t n, int32_t t0, int32_t t1,
                             uint16_t* recv_x_node, float* recv_prob_node) {
    for (int32_t t = t0; t < t1; ++t) {
        size_t row = (size_t)n * max_tokens + t;
        for (int32_t h = 0; h < H; ++h) recv_x_node[row * H + h] = x[(size_t)t * H + h];
        if (prob_staging != NULL && recv_prob_node != NULL)
            for (int32_t p = 0; p < P; ++p) recv_prob_node[row * P + p] = prob_staging[row * P + p];
    }
}

/* [PR #634] "Fix": per (chunk of chunk_tokens consecutive tokens, destination
 * node n) the dense path moves the chunk's whole token range of hidden rows and
 * of staged prob slices in one copy each; the sparse path moves one copy per
 * maximal run of consecutive tokens of the chunk that route to n.
 * Reading of the receive layout: token-indexed, so destination positions follow
 * source positions (recv_x_node[n][t] = x[t], recv_prob_node[n][t] =
 * prob_staging[n][t]); that is what makes one copy per chunk or per run
 * coherent, and it matches the receive side keeping token-major strides.
 * num_runs[n][c] counts the copies of the hidden rows for (n, chunk c): 1 for
 * every non-empty chunk on the dense path, the number of runs on the sparse
 * path. Requires T <= max_tokens (returns -1 otherwise, writing nothing). */
int32_t oracle_dispatch_nodes(const uint16_t* x, const float* prob_staging,
                              const uint8_t* is_token_in_node, int32_t T, int32_t H, int32_t N,
                              int32_t P, int32_t max_tokens, int32_t chunk_tokens, int32_t mode,
                              uint16_t* recv_x_node, float* recv_prob_node, int32_t* num_runs) {
    if (T > max_tokens || chunk_tokens <= 0) return -1;
    int32_t nchunks = (T + chunk_tokens - 1) / chunk_tokens;
    for (int32_t n = 0; n < N; ++n) {
        for (int32_t c = 0; c < nchunks; ++c) {
            int32_t t0 = c * chunk_tokens;
            int32_t t1 = t0 + chunk_tokens < T ? t0 + chunk_tokens : T;
            int32_t runs = 0;
            if (mode == 0) {
                copy_token_range(x, prob_staging, H, P, max_tokens, n, t0, t1, recv_x_node, recv_prob_node);
                runs = t1 > t0 ? 1 : 0;
            } else {
                int32_t t = t0;
                while (t < t1) {
                    if (!is_token_in_node[(size_t)t * N + n]) {
                        ++t;
                        continue;
                    }
                    int32_t start = t;
                    while (t < t1 && is_token_in_node[(size_t)t * N + n]) ++t;
                    copy_token_range(x, prob_staging, H, P, max_tokens, n, start, t, recv_x_node,
                                     recv_prob_node);
                    runs += 1;
                }
            }
            if (num_runs != NULL) num_runs[(size_t)n * nchunks + c] = runs;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Combine                                                                   */
/* ------------------------------------------------------------------------- */

/* Combine brings every rank's expert output for a token back to the token's
 * position and reduces ([PR #347] 2.1 and the BF16 combine table of 3.2.1):
 *   acc = 0 (fp32); for r = 0, 1, ..., R-1 with s = slot[t][r] >= 0:
 *       acc = acc + float(y[r][s][h])
 *   out[t][h] = bf16_rn(acc)
 * Readings: the sum is unweighted (weights belong to the expert), it runs in
 * ascending rank order, and a token routed nowhere gets +0. A slot at or beyond
 * max_tokens was never received; it is skipped and raises
 * ORACLE_FLAG_CAPACITY. */
int32_t oracle_combine(const uint16_t* y, const int32_t* slot, int32_t T, int32_t H, int32_t R,
                       int32_t max_tokens, uint16_t* out) {
    int32_t flags = 0;
    float* acc = (float*)malloc((size_t)H * sizeof(float) + 1);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int32_t r = 0; r < R; ++r) {
            int32_t s = slot[(size_t)t * R + r];
            if (s < 0) continue;
            if (s >= max_tokens) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            const uint16_t* row = y + ((size_t)r * max_tokens + s) * H;
            for (int32_t h = 0; h < H; ++h) acc[h] = acc[h] + oracle_bf16_to_f32(row[h]);
        }
        for (int32_t h = 0; h < H; ++h) out[(size_t)t * H + h] = oracle_f32_to_bf16(acc[h]);
    }
    free(acc);
    return flags;
}

/* Combine of FP8 expert outputs. The pages show only the BF16 combine ([PR #347]
 * 3.2.1) and, for FP8, the dispatch row format (H E4M3 codes and one fp32 scale per
 * 128 channels). Reading: a received FP8 row is dequantised exactly as the dispatch
 * wrote it, v[h] = fp32(e4m3(q[h]) * scale[h / 128]) (one fp32 rounding), and reduced
 * as oracle_combine does:
 *   acc = 0 (fp32); for r = 0, 1, ..., R-1 with s = slot[t][r] >= 0: acc = acc + v
 *   out[t][h] = bf16_rn(acc)
 * Slots at or beyond max_tokens are skipped and raise ORACLE_FLAG_CAPACITY. */
int32_t oracle_combine_fp8(const uint8_t* y, const float* y_scales, const int32_t* slot, int32_t T,
                           int32_t H, int32_t R, int32_t max_tokens, uint16_t* out) {
    int32_t flags = 0;
    int32_t nb = H / 128;
    float* acc = (float*)malloc((size_t)H * sizeof(float) + 1);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int32_t r = 0; r < R; ++r) {
            int32_t s = slot[(size_t)t * R + r];
            if (s < 0) continue;
            if (s >= max_tokens) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            size_t yr = (size_t)r * max_tokens + s;
            for (int32_t h = 0; h < H; ++h) {
                float v = oracle_e4m3_to_f32(y[yr * H + h]) * y_scales[yr * nb + h / 128];
                acc[h] = acc[h] + v;
            }
        }
        for (int32_t h = 0; h < H; ++h) out[(size_t)t * H + h] = oracle_f32_to_bf16(acc[h]);
    }
    free(acc);
    return flags;
}

/* Combined top-k weights: the combine also brings the received weight rows back to
 * token order ([PR #347] 2.1: the combine returns what the dispatch sent out). Each
 * rank's copy of a token carries w_j for the slots whose expert it holds and 0 for
 * the others, so
 *   out[t][j] = sum over r ascending with s = slot[t][r] >= 0 of recv_topk_w[r][s][j]
 * (fp32 from +0) gives back the router's weight of every slot (0 where the slot was
 * empty, out of range or dropped). Slots at or beyond max_tokens are skipped and raise
 * ORACLE_FLAG_CAPACITY. */
int32_t oracle_combine_weights(const float* recv_topk_w, const int32_t* slot, int32_t T, int32_t k,
                               int32_t R, int32_t max_tokens, float* out) {
    int32_t flags = 0;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) out[(size_t)t * k + j] = 0.0f;
        for (int32_t r = 0; r < R; ++r) {
            int32_t s = slot[(size_t)t * R + r];
            if (s < 0) continue;
            if (s >= max_tokens) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            const float* w = recv_topk_w + ((size_t)r * max_tokens + s) * k;
            for (int32_t j = 0; j < k; ++j) out[(size_t)t * k + j] = out[(size_t)t * k + j] + w[j];
        }
    }
    return flags;
}

/* ------------------------------------------------------------------------- */
/* Expert-major layout, permuted dispatch, receive-side permute, combine       */
/* ------------------------------------------------------------------------- */

/* [PR #634] "Hybrid ep nixl restripe", commit "hybrid_ep: fix scan permute-fusion
 * local-experts sum array sizing" and the "dispatch+permute" rows of its B300 results:
 * after dispatch the tokens a rank receives are permuted into local-expert order, from a
 * scan over tokens and a per-local-expert sum array. Written out:
 *   count[e]          = number of (t, j) whose expert is e (each token's ids distinct)
 *   expert_offsets[e] = sum of count[e'] for e' < e   (expert_offsets[E] = total)
 *   expert_slot[t][j] = number of (t', j') before (t, j), in token-then-slot order,
 *                       with the same expert; -1 for an empty slot (< 0), an id >= E, or a
 *                       repeat of an id earlier in the same row (the last two raise
 *                       ORACLE_FLAG_BAD_EXPERT).
 * Experts of a rank are contiguous, so expert order is rank-major: rank r's entries are
 * expert_offsets[r*(E/R)] .. expert_offsets[(r+1)*(E/R)], grouped by local expert. */
int32_t oracle_expert_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E,
                             int32_t* expert_offsets, int32_t* expert_slot) {
    int32_t flags = 0;
    int32_t* cnt = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int64_t e = topk_idx[(size_t)t * k + j];
            int32_t out = -1;
            if (e >= E) {
                flags |= ORACLE_FLAG_BAD_EXPERT;
            } else if (e >= 0) {
                int repeat = 0;
                for (int32_t jj = 0; jj < j; ++jj)
                    if (topk_idx[(size_t)t * k + jj] == e) repeat = 1;
                if (repeat) {
                    flags |= ORACLE_FLAG_BAD_EXPERT;
                } else {
                    out = cnt[e];
                    cnt[e] += 1;
                }
            }
            expert_slot[(size_t)t * k + j] = out;
        }
    }
    expert_offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) expert_offsets[e + 1] = expert_offsets[e] + cnt[e];
    free(cnt);
    return flags;
}

/* row of (t, j) inside its rank's expert-major slab */
static int32_t permuted_row(const int32_t* expert_offsets, const int32_t* expert_slot, int32_t t,
                            int32_t j, int32_t k, int64_t e, int32_t E, int32_t R) {
    int32_t epr = E / R;
    int32_t r = (int32_t)(e / epr);
    return expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];
}

/* Dispatch and permute fused: for every (t, j) with expert_slot[t][j] >= 0, expert e on
 * rank r = e / (E/R), and p = expert_offsets[e] - expert_offsets[r*(E/R)] + expert_slot:
 *   perm_x[r][p] = x[t], perm_src[r][p] = t, perm_w[r][p] = topk_w[t][j].
 * A token with two experts on one rank occupies two rows. p >= max_rows is dropped and
 * raises ORACLE_FLAG_CAPACITY. Other rows are not written. */
int32_t oracle_dispatch_permuted(const uint16_t* x, const int64_t* topk_idx, const float* topk_w,
                                 const int32_t* expert_offsets, const int32_t* expert_slot,
                                 int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                 int32_t max_rows, uint16_t* perm_x, int32_t* perm_src,
                                 float* perm_w) {
    int32_t flags = 0;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            if (expert_slot[(size_t)t * k + j] < 0) continue;
            int64_t e = topk_idx[(size_t)t * k + j];
            int32_t r = (int32_t)(e / (E / R));
            int32_t p = permuted_row(expert_offsets, expert_slot, t, j, k, e, E, R);
            if (p >= max_rows) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            size_t row = (size_t)r * max_rows + (size_t)p;
            for (int32_t h = 0; h < H; ++h) perm_x[row * H + h] = x[(size_t)t * H + h];
            if (perm_src != NULL) perm_src[row] = t;
            if (perm_w != NULL) perm_w[row] = topk_w[(size_t)t * k + j];
        }
    }
    return flags;
}

/* The receive phase of a split (hook-mode) dispatch ([PR #347] 2.1: the send phase
 * returns first, the receive phase runs later): every row s < min(tokens_per_rank[r],
 * max_tokens) that rank r received from a rank-level dispatch, for every slot j whose
 * local expert id l = recv_topk_idx[r][s][j] >= 0, goes to the same expert-major row the
 * fused dispatch uses (t = recv_src_idx[r][s], e = r*(E/R) + l):
 *   perm_x[r][p] = recv_x[r][s], perm_src[r][p] = t, perm_w[r][p] = recv_topk_w[r][s][j]. */
int32_t oracle_permute_received(const uint16_t* recv_x, const int32_t* recv_src_idx,
                                const int32_t* recv_topk_idx, const float* recv_topk_w,
                                const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                                const int32_t* expert_slot, int32_t T, int32_t H, int32_t k,
                                int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                                uint16_t* perm_x, int32_t* perm_src, float* perm_w) {
    int32_t flags = 0;
    int32_t epr = E / R;
    (void)T;
    for (int32_t r = 0; r < R; ++r) {
        int32_t n = tokens_per_rank[r] < max_tokens ? tokens_per_rank[r] : max_tokens;
        for (int32_t s = 0; s < n; ++s) {
            size_t in_row = (size_t)r * max_tokens + s;
            int32_t t = recv_src_idx[in_row];
            for (int32_t j = 0; j < k; ++j) {
                int32_t l = recv_topk_idx[in_row * k + j];
                if (l < 0 || expert_slot[(size_t)t * k + j] < 0) continue;
                int32_t e = r * epr + l;
                int32_t p = expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];
                if (p >= max_rows) {
                    flags |= ORACLE_FLAG_CAPACITY;
                    continue;
                }
                size_t row = (size_t)r * max_rows + (size_t)p;
                for (int32_t h = 0; h < H; ++h) perm_x[row * H + h] = recv_x[in_row * H + h];
                if (perm_src != NULL) perm_src[row] = t;
                if (perm_w != NULL) perm_w[row] = recv_topk_w[in_row * k + j];
            }
        }
    }
    return flags;
}

/* Combine from the expert-major slabs:
 *   acc = 0 (fp32); for j = 0, 1, ..., k-1 with expert_slot[t][j] >= 0:
 *       term = float(y[r][p][h]), times topk_w[t][j] (one fp32 multiply) when weighted
 *       acc  = acc + term
 *   out[t][h] = bf16_rn(acc)
 * Reading: the token's own top-k order fixes the order of the terms; rows p >= max_rows
 * were never written and are skipped with ORACLE_FLAG_CAPACITY. */
int32_t oracle_combine_permuted(const uint16_t* y, const int64_t* topk_idx, const float* topk_w,
                                const int32_t* expert_offsets, const int32_t* expert_slot,
                                int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                int32_t max_rows, uint16_t* out) {
    int32_t flags = 0;
    float* acc = (float*)malloc((size_t)H * sizeof(float) + 1);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int32_t j = 0; j < k; ++j) {
            if (expert_slot[(size_t)t * k + j] < 0) continue;
            int64_t e = topk_idx[(size_t)t * k + j];
            int32_t r = (int32_t)(e / (E / R));
            int32_t p = permuted_row(expert_offsets, expert_slot, t, j, k, e, E, R);
            if (p >= max_rows) {
                flags |= ORACLE_FLAG_CAPACITY;
                continue;
            }
            const uint16_t* row = y + ((size_t)r * max_rows + p) * H;
            for (int32_t h = 0; h < H; ++h) {
                float term = oracle_bf16_to_f32(row[h]);
                if (topk_w != NULL) term = term * topk_w[(size_t)t * k + j];
                acc[h] = acc[h] + term;
            }
        }
        for (int32_t h = 0; h < H; ++h) out[(size_t)t * H + h] = oracle_f32_to_bf16(acc[h]);
    }
    free(acc);
    return flags;
}

/* The send phase of a split (hook-mode) combine ([PR #347] 2.1: in hook mode the send
 * phase runs first and returns, the receive phase runs later as its own step). The
 * combine's receive phase is oracle_combine: it reads one row per (token, rank) from
 * the rank-level slabs. The send phase fills those rows: rank r takes, for every row
 * s < min(tokens_per_rank[r], max_tokens) it received (t = recv_src_idx[r][s]), the
 * expert-major rows of that token's local experts -- the rows the receive-side permute
 * wrote, p = expert_offsets[e] - expert_offsets[r*(E/R)] + expert_slot[t][j] for every
 * slot j with local id l = recv_topk_idx[r][s][j] >= 0, e = r*(E/R) + l -- and reduces
 * them into its rank-level row:
 *   acc = 0 (fp32); for j = 0, 1, ..., k-1 with such a row p:
 *       term = float(y_perm[r][p][h]), times recv_topk_w[r][s][j] (one fp32 multiply)
 *              when weights are given
 *       acc  = acc + term
 *   y_rank[r][s][h] = bf16_rn(acc)
 * Reading: the pages split the combine into send and receive without fixing where a
 * rank's local experts are reduced; the rank-level receive rows are bf16 like every other
 * combine input, so each rank rounds its partial sum once. Rows p >= max_rows were never
 * written: skipped with ORACLE_FLAG_CAPACITY. Rows s beyond the count are not written. */
int32_t oracle_combine_send(const uint16_t* y_perm, const int32_t* recv_src_idx,
                            const int32_t* recv_topk_idx, const float* recv_topk_w,
                            const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                            const int32_t* expert_slot, int32_t T, int32_t H, int32_t k,
                            int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                            uint16_t* y_rank) {
    int32_t flags = 0;
    int32_t epr = E / R;
    float* acc = (float*)malloc((size_t)H * sizeof(float) + 1);
    (void)T;
    for (int32_t r = 0; r < R; ++r) {
        int32_t n = tokens_per_rank[r] < max_tokens ? tokens_per_rank[r] : max_tokens;
        for (int32_t s = 0; s < n; ++s) {
            size_t row = (size_t)r * max_tokens + s;
            int32_t t = recv_src_idx[row];
            for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int32_t l = recv_topk_idx[row * k + j];
                if (l < 0 || expert_slot[(size_t)t * k + j] < 0) continue;
                int32_t e = r * epr + l;
                int32_t p = expert_offsets[e] - expert_offsets[r * epr] + expert_slot[(size_t)t * k + j];
                if (p >= max_rows) {
                    flags |= ORACLE_FLAG_CAPACITY;
                    continue;
                }
                const uint16_t* src = y_perm + ((size_t)r * max_rows + p) * H;
                for (int32_t h = 0; h < H; ++h) {
                    float term = oracle_bf16_to_f32(src[h]);
                    if (recv_topk_w != NULL) term = term * recv_topk_w[row * k + j];
                    acc[h] = acc[h] + term;
                }
            }
            for (int32_t h = 0; h < H; ++h) y_rank[row * H + h] = oracle_f32_to_bf16(acc[h]);
        }
    }
    free(acc);
    return flags;
}

/* ------------------------------------------------------------------------- */
/* Harness expert (between dispatch and combine; not a step of the path)      */
/* ------------------------------------------------------------------------- */

/* y[r][s][h] = bf16_rn(v * w) with w = sum over j, in j order from 0, of
 * recv_topk_w[r][s][j] and v = float(recv_x[r][s][h]) for bf16 rows, or
 * (float(q) * scale) for e4m3 rows. Only rows s < min(tokens_per_rank[r],
 * max_tokens) are written. */
void oracle_expert_scale(const void* recv_x, int32_t in_fp8, const float* recv_scales,
                         const float* recv_topk_w, const int32_t* tokens_per_rank, int32_t R,
                         int32_t max_tokens, int32_t H, int32_t k, uint16_t* y) {
    int32_t nb = H / 128;
    for (int32_t r = 0; r < R; ++r) {
        int32_t count = tokens_per_rank[r] < max_tokens ? tokens_per_rank[r] : max_tokens;
        for (int32_t s = 0; s < count; ++s) {
            size_t row = (size_t)r * max_tokens + s;
            float w = 0.0f;
            for (int32_t j = 0; j < k; ++j) w = w + recv_topk_w[row * k + j];
            for (int32_t h = 0; h < H; ++h) {
                float v;
                if (in_fp8) {
                    uint8_t q = ((const uint8_t*)recv_x)[row * H + h];
                    v = oracle_e4m3_to_f32(q) * recv_scales[row * nb + h / 128];
                } else {
                    v = oracle_bf16_to_f32(((const uint16_t*)recv_x)[row * H + h]);
                }
                y[row * H + h] = oracle_f32_to_bf16(v * w);
            }
        }
    }
}
