/*
 * ep_oracle.h -- the oracle: a plain, slow, single-threaded C99 statement of
 * what the expert-parallel dispatch/combine path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg may load this library. The
 * CUDA library shares no code, header, table or helper with it.
 *
 * Conventions (the same contract the CUDA library states, written out here
 * independently):
 *   - bf16 values are passed as their raw uint16 bit patterns.
 *   - e4m3 values are raw uint8 bit patterns (OCP OFP8 E4M3: bias 7, no
 *     infinities, NaN = S.1111.111, largest finite 448).
 *   - topk_idx entries < 0 mean "no expert"; entries >= E are invalid: they are
 *     skipped and raise ORACLE_FLAG_BAD_EXPERT.
 *   - Expert e lives on virtual rank e / (E / R); rank r lives on node
 *     r / ranks_per_node.
 *   - Return values are a bit mask of ORACLE_FLAG_* (0 = clean).
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_FLAG_CAPACITY 1   /* a slot >= max_tokens was dropped */
#define ORACLE_FLAG_BAD_EXPERT 2 /* a topk_idx entry >= E was skipped */

/* number formats */
uint16_t oracle_f32_to_bf16(float f);
float oracle_bf16_to_f32(uint16_t b);
uint8_t oracle_f32_to_e4m3(float f);
float oracle_e4m3_to_f32(uint8_t q);
/* one token row of H bf16 -> H e4m3 codes + H/128 fp32 scales */
void oracle_quantize_row_e4m3(const uint16_t* x, int32_t H, uint8_t* q, float* scales);

/* routing layout */
int32_t oracle_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                      int32_t ranks_per_node, int32_t* tokens_per_expert,
                      int32_t* tokens_per_rank, int32_t* tokens_per_node,
                      uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot);

/* rank-level dispatch; out_fp8 = 0: recv_x is bf16, 1: recv_x is e4m3 + recv_scales.
 * Any of recv_x / recv_scales / recv_src_idx / recv_topk_idx / recv_topk_w may be
 * NULL, in which case that output is not produced. */
int32_t oracle_dispatch(const uint16_t* x, int32_t out_fp8, const int64_t* topk_idx,
                        const float* topk_w, const int32_t* slot, int32_t T, int32_t H,
                        int32_t k, int32_t E, int32_t R, int32_t max_tokens, void* recv_x,
                        float* recv_scales, int32_t* recv_src_idx, int32_t* recv_topk_idx,
                        float* recv_topk_w);

/* prob restripe [T][N][P] -> [N][max_tokens][P] */
void oracle_restripe_prob(const float* prob, int32_t T, int32_t N, int32_t P,
                          int32_t max_tokens, float* out);

/* node-level dispatch, token-indexed receive; mode 0 = dense, 1 = sparse (runs) */
int32_t oracle_dispatch_nodes(const uint16_t* x, const float* prob_staging,
                              const uint8_t* is_token_in_node, int32_t T, int32_t H, int32_t N,
                              int32_t P, int32_t max_tokens, int32_t chunk_tokens, int32_t mode,
                              uint16_t* recv_x_node, float* recv_prob_node, int32_t* num_runs);

/* combine: fp32 sum in ascending rank order, one rounding to bf16 */
int32_t oracle_combine(const uint16_t* y, const int32_t* slot, int32_t T, int32_t H, int32_t R,
                       int32_t max_tokens, uint16_t* out);

/* combine of FP8 rows (codes [R][max][H], scales [R][max][H/128]): each row dequantised
 * to fp32(e4m3(q) * scale), then as oracle_combine */
int32_t oracle_combine_fp8(const uint8_t* y, const float* y_scales, const int32_t* slot, int32_t T,
                           int32_t H, int32_t R, int32_t max_tokens, uint16_t* out);

/* combined top-k weights: out[t][j] = fp32 sum over ranks ascending of recv_topk_w[r][slot][j] */
int32_t oracle_combine_weights(const float* recv_topk_w, const int32_t* slot, int32_t T, int32_t k,
                               int32_t R, int32_t max_tokens, float* out);

/* expert-major layout: offsets [E+1] (exclusive sums of the per-expert counts, in
 * expert order) and expert_slot [T][k] = the stable position of (t, j) among the
 * entries of its expert, or -1. A repeated id in one token's row keeps only its
 * first occurrence (the repeat gets -1 and raises ORACLE_FLAG_BAD_EXPERT). */
int32_t oracle_expert_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E,
                             int32_t* expert_offsets, int32_t* expert_slot);

/* fused dispatch + permute into expert-major rank slabs [R][max_rows][H] */
int32_t oracle_dispatch_permuted(const uint16_t* x, const int64_t* topk_idx, const float* topk_w,
                                 const int32_t* expert_offsets, const int32_t* expert_slot,
                                 int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                 int32_t max_rows, uint16_t* perm_x, int32_t* perm_src,
                                 float* perm_w);

/* receive-side permute of rank-level dispatch output into the same expert-major slabs */
int32_t oracle_permute_received(const uint16_t* recv_x, const int32_t* recv_src_idx,
                                const int32_t* recv_topk_idx, const float* recv_topk_w,
                                const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                                const int32_t* expert_slot, int32_t T, int32_t H, int32_t k,
                                int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                                uint16_t* perm_x, int32_t* perm_src, float* perm_w);

/* combine from expert-major slabs: out[t] = bf16(sum over j ascending of w_j * y), weighted
 * when topk_w is not NULL (one fp32 multiply and one fp32 add per term), plain sum otherwise */
int32_t oracle_combine_permuted(const uint16_t* y, const int64_t* topk_idx, const float* topk_w,
                                const int32_t* expert_offsets, const int32_t* expert_slot,
                                int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                int32_t max_rows, uint16_t* out);

/* send phase of a split combine: each rank reduces, per received row, its local experts'
 * expert-major rows (slot order, weighted by recv_topk_w when not NULL) into one bf16 row
 * of its rank-level slab y_rank [R][max_tokens][H]; oracle_combine is the receive phase */
int32_t oracle_combine_send(const uint16_t* y_perm, const int32_t* recv_src_idx,
                            const int32_t* recv_topk_idx, const float* recv_topk_w,
                            const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                            const int32_t* expert_slot, int32_t T, int32_t H, int32_t k,
                            int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                            uint16_t* y_rank);

/* the test harness's stand-in expert (not part of the path): every received row
 * scaled by the sum, in j order, of its top-k weights on that rank */
void oracle_expert_scale(const void* recv_x, int32_t in_fp8, const float* recv_scales,
                         const float* recv_topk_w, const int32_t* tokens_per_rank, int32_t R,
                         int32_t max_tokens, int32_t H, int32_t k, uint16_t* y);

#ifdef __cplusplus
}
#endif
#endif
