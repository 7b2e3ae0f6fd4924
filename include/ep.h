/*
 * ep.h -- C ABI of the GB300 (sm_103a) expert-parallel dispatch/combine library.
 *
 * One GPU holds R "virtual" expert-parallel ranks as partitions of its HBM: a
 * rank's receive buffer is its slab [max_tokens][...] of a destination-major
 * [R][max_tokens][...] array. Sending a token to a rank is a store into that
 * slab; receiving is a load from it. The operations follow the expert-parallel
 * dispatch/combine described on the DeepEP pull-request pages:
 *   [PR #347] "Feature/sm free normal kernel" (sections 2.1 Feature,
 *     3.1 Experiment Setup, 3.2.1 tables, 3.3.1 HBM Cost; the commit that adds
 *     return_recv_hook to get_dispatch_layout),
 *   [PR #634] "Hybrid ep nixl restripe" (sections Baseline problem, Fix,
 *     Receive-side and DOCA path are unchanged; the scan permute-fusion commit),
 *   [PR #453] "Higher Performance with Lower SM Occupancy through Zero-Copy and
 *     TMA Offloading" (commits: recv-count assertion, separate dispatch/combine
 *     buffer sizes, buffer alignment).
 *
 * General contract (every entry point):
 *   - Pointers named d_* / device arrays are CUDA device pointers on the
 *     current device; the library reads and writes them only from kernels
 *     launched on `stream`. The caller owns every buffer; the library never
 *     allocates, frees or synchronises, and returns as soon as its kernels are
 *     queued.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Arrays are dense, row-major, in the layout stated per argument. Every
 *     array pointer must be 16-byte aligned (rows are moved in 16-byte vectors).
 *   - Sizes are int32; products of sizes are computed in 64 bits.
 *   - The return value is synchronous: EP_OK when the kernels were queued,
 *     EP_ERR_INVALID when an argument is rejected (nothing was launched),
 *     EP_ERR_CUDA when a launch failed (ep_last_cuda_error() gives the code).
 *   - Errors found by the kernels are reported asynchronously by OR-ing
 *     EP_FLAG_* bits into `*status` (a device int32, zeroed by the caller;
 *     status may be NULL to ignore them). Kernels never trap: an out-of-range
 *     write is skipped, never performed.
 *   - Calls on one stream run in order; two calls that share an output or a
 *     workspace must not run concurrently on different streams.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EP_ABI_VERSION 1

typedef int32_t ep_status_t;
#define EP_OK 0
#define EP_ERR_INVALID 1
#define EP_ERR_CUDA 2
#define EP_ERR_SCRATCH 3 /* ep_get_layout_noalloc: the sizes need more than its fixed scratch */

/* asynchronous error bits OR-ed into *status by the kernels */
#define EP_FLAG_CAPACITY 1   /* a receive slot >= max_tokens was dropped ([PR #453] commit
                                "Add assertion against too large recv token count", as a flag) */
#define EP_FLAG_BAD_EXPERT 2 /* a topk_idx entry >= E was skipped */
#define EP_FLAG_TIMEOUT 4    /* a bounded wait gave up: a layout scan's look-back, or a
                                bulk-copy row load of a BF16 dispatch (its copy is then
                                incomplete) */
#define EP_FLAG_WORKSPACE 8  /* the layout workspace was not at rest: zero-fill it and call again */

typedef int32_t ep_dtype_t;
#define EP_DTYPE_BF16 0 /* bfloat16 rows, 2 bytes per element */
#define EP_DTYPE_E4M3 1 /* OCP E4M3 rows (1 byte per element) + one fp32 scale per 128 elements */

typedef int32_t ep_node_mode_t;
#define EP_NODES_DENSE 0  /* copy every chunk's whole token range to every node */
#define EP_NODES_SPARSE 1 /* copy only the runs of consecutive tokens routed to the node */

/* ABI version of the loaded library (EP_ABI_VERSION at build time). */
int32_t ep_abi_version(void);

/* Static string describing a synchronous status (EP_OK, EP_ERR_*). Never NULL. */
const char* ep_status_str(ep_status_t s);

/* cudaError_t code behind the most recent EP_ERR_CUDA returned on the calling
 * host thread (0 if there was none). */
int32_t ep_last_cuda_error(void);

/* ------------------------------------------------------------------------- */
/* Routing layout                                                            */
/* ------------------------------------------------------------------------- */

/* Bytes of device workspace ep_get_layout needs for these sizes. */
size_t ep_layout_workspace_size(int32_t T, int32_t E, int32_t R, int32_t ranks_per_node);

/* First bytes of the layout workspace. The workspace must be zero-filled once
 * before its first use; every completed call leaves it ready for the next call
 * (the counter returns to zero and the epoch advances). `stall_tile` is a test
 * hook: when it holds i + 1, tile i never publishes its counts, so that the
 * bounded waits of its successors run out and raise EP_FLAG_TIMEOUT. Keep it 0. */
typedef struct {
    uint32_t reserved;   /* unused, left as found */
    uint32_t done;       /* tiles that have added their counts */
    uint32_t epoch;      /* calls completed on this workspace */
    uint32_t stall_tile; /* test hook, 0 = off */
} ep_layout_ws_header_t;

/* ep_get_layout -- the routing layout of a batch (get_dispatch_layout,
 * [PR #347] commit list; the scan of [PR #634] "fix scan permute-fusion
 * local-experts sum array sizing").
 *
 * Inputs
 *   topk_idx        int64 [T][k]  router output: expert ids; < 0 = no expert;
 *                                 >= E is skipped and raises EP_FLAG_BAD_EXPERT
 *   T >= 0 tokens, 1 <= k <= 32, 1 <= R <= 256 ranks, E experts with E % R == 0
 *   and E <= 8192 (expert e lives on rank e / (E/R)); ranks_per_node = 0 (no
 *   node outputs) or a divisor of R (rank r lives on node r / ranks_per_node).
 * Outputs (all overwritten, in token order)
 *   tokens_per_expert int32 [E]   number of (t, j) with topk_idx[t][j] == e
 *   tokens_per_rank   int32 [R]   tokens sent to each rank (a token with several
 *                                 experts on one rank is sent once)
 *   tokens_per_node   int32 [N]   likewise per node (NULL when ranks_per_node = 0)
 *   is_token_in_rank  uint8 [T][R] 1 when token t goes to rank r
 *   is_token_in_node  uint8 [T][N] likewise per node (NULL when ranks_per_node = 0)
 *   slot              int32 [T][R] stable exclusive prefix sum down the tokens:
 *                                 #{t' < t : is_token_in_rank[t'][r]}, or -1
 *   workspace         device, >= ep_layout_workspace_size(...) bytes, 256-byte
 *                     aligned, zero-filled before its first use (see above)
 *   status            device int32 or NULL; EP_FLAG_BAD_EXPERT, EP_FLAG_TIMEOUT,
 *                     EP_FLAG_WORKSPACE (outputs not written)
 */
ep_status_t ep_get_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                          int32_t ranks_per_node, int32_t* tokens_per_expert,
                          int32_t* tokens_per_rank, int32_t* tokens_per_node,
                          uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot,
                          void* workspace, size_t workspace_bytes, int32_t* status,
                          void* stream);

/* ep_get_layout_noalloc -- ep_get_layout for callers that cannot allocate.
 * The pages have no counterpart: this entry point exists for callers that have
 * no way to provide the layout workspace -- code that must not allocate device
 * memory where it runs (a fixed, pre-planned memory budget with no allocator of
 * its own), or a host runtime that can only pass pointers to arrays it already
 * owns. It computes exactly what ep_get_layout computes, with the same inputs,
 * outputs, argument rules and flags, but takes no workspace: it uses a
 * fixed-size array inside the library (EP_LAYOUT_NOALLOC_SCRATCH_BYTES of
 * device memory that every GPU which loads the library keeps until the process
 * exits). It never calls cudaMalloc, cudaFree or any allocating routine.
 *   - Each call looks up that array's device address (cudaGetSymbolAddress,
 *     with the device current) and remembers it per device; a call made while
 *     `stream` is capturing uses the remembered address instead, and returns
 *     EP_ERR_INVALID (nothing queued) when none has been remembered yet.
 *   - Each call zero-fills the part of the array it uses (an async memset on
 *     `stream`), then launches the layout kernel.
 *   - Sizes whose workspace (ep_layout_workspace_size) exceeds
 *     EP_LAYOUT_NOALLOC_SCRATCH_BYTES are rejected with EP_ERR_SCRATCH before
 *     anything is launched (T up to 126,720 tokens at R = 256, 1,014,528 at R = 32).
 *   - All calls on a device share the array: calls whose work can overlap on the
 *     GPU (different streams without ordering) race. Keep them on one stream.
 */
#define EP_LAYOUT_NOALLOC_SCRATCH_BYTES (1u << 20)
ep_status_t ep_get_layout_noalloc(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                                  int32_t ranks_per_node, int32_t* tokens_per_expert,
                                  int32_t* tokens_per_rank, int32_t* tokens_per_node,
                                  uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot,
                                  int32_t* status, void* stream);

/* ------------------------------------------------------------------------- */
/* Rank-level dispatch                                                       */
/* ------------------------------------------------------------------------- */

/* ep_dispatch -- send every token once to every rank it routes to ([PR #347]
 * 2.1 Feature; workload of 3.1: 4096 tokens, hidden 7168, top-8; FP8 and BF16
 * dispatch of 3.2.1). For every (t, r) with s = slot[t][r] >= 0:
 *   recv_x[r][s][:]        = x[t][:]                  (out_dtype BF16), or
 *                            e4m3(x[t][:] / scale_b)  (out_dtype E4M3) with
 *   recv_scales[r][s][b]   = scale_b = amax_b / 448, amax_b = max |x| over the
 *                            128 elements of block b (fp32, correctly rounded
 *                            division; q rounded once to nearest-even and
 *                            saturated to +-448; a block with amax 0 stores
 *                            scale 0 and the signed zero code of each element)
 *   recv_src_idx[r][s]     = t
 *   recv_topk_idx[r][s][j] = e_j - r*(E/R) when expert e_j lives on r, else -1
 *   recv_topk_w[r][s][j]   = topk_w[t][j] when expert e_j lives on r, else 0
 * A slot >= max_tokens is dropped and raises EP_FLAG_CAPACITY. Rows a rank does
 * not receive are not written.
 *
 *   x             bf16 [T][H], H % 8 == 0 (H % 128 == 0 for E4M3)
 *   topk_idx      int64 [T][k], topk_w fp32 [T][k] (topk_w may be NULL when
 *                 recv_topk_w is NULL)
 *   slot          int32 [T][R] from ep_get_layout
 *   recv_x        [R][max_tokens][H] of out_dtype (required); R * max_tokens < 2^31
 *   recv_scales   fp32 [R][max_tokens][H/128]               (E4M3 only, else NULL)
 *   recv_src_idx  int32 [R][max_tokens]                     (nullable)
 *   recv_topk_idx int32 [R][max_tokens][k]                  (nullable)
 *   recv_topk_w   fp32 [R][max_tokens][k]                   (nullable)
 *   status        EP_FLAG_CAPACITY, EP_FLAG_BAD_EXPERT; EP_FLAG_TIMEOUT (BF16, rows
 *                 moved by bulk copies: a row load that never completed)
 */
ep_status_t ep_dispatch(const void* x, ep_dtype_t out_dtype, const int64_t* topk_idx,
                        const float* topk_w, const int32_t* slot, int32_t T, int32_t H, int32_t k,
                        int32_t E, int32_t R, int32_t max_tokens, void* recv_x,
                        float* recv_scales, int32_t* recv_src_idx, int32_t* recv_topk_idx,
                        float* recv_topk_w, int32_t* status, void* stream);

/* ------------------------------------------------------------------------- */
/* Prob restripe                                                             */
/* ------------------------------------------------------------------------- */

/* ep_restripe_prob -- [PR #634] "Baseline problem" / "Fix": copy the prob
 * tensor from its token-major layout [T][num_nodes][P] into the
 * destination-major staging layout [num_nodes][max_tokens][P], so that the
 * slices one destination needs for consecutive tokens are contiguous:
 *   out[n][t][p] = prob[t][n][p]   for all t < T, n < num_nodes, p < P.
 * Every (t, n) slice is copied (the same bytes as the plain copy it replaces);
 * rows t in [T, max_tokens) are not written.
 *   prob  fp32 [T][num_nodes][P], P % 4 == 0;  out fp32 [num_nodes][max_tokens][P]
 *   requires T <= max_tokens.
 */
ep_status_t ep_restripe_prob(const float* prob, int32_t T, int32_t num_nodes, int32_t P,
                             int32_t max_tokens, float* out, void* stream);

/* ------------------------------------------------------------------------- */
/* Node-level dense / sparse dispatch                                        */
/* ------------------------------------------------------------------------- */

/* ep_dispatch_nodes -- [PR #634] "Fix": per chunk of chunk_tokens consecutive
 * tokens (NUM_OF_TOKENS_PER_CHUNK = 256 on the page) and destination node n,
 *   EP_NODES_DENSE : the chunk's whole token range of hidden rows and of staged
 *                    prob slices goes to n in one contiguous copy each;
 *   EP_NODES_SPARSE: only the maximal runs of consecutive tokens of the chunk
 *                    with is_token_in_node[t][n] go, one copy per run.
 * The receive layout is token-indexed (destination positions follow source
 * positions; the receive side keeps token-major strides, [PR #634] "Receive-side
 * and DOCA path are unchanged"):
 *   recv_x_node[n][t][:]    = x[t][:]
 *   recv_prob_node[n][t][:] = prob_staging[n][t][:]
 *   num_runs[n][c]          = copies of hidden rows made for (n, chunk c):
 *                             1 per non-empty chunk (dense), runs (sparse)
 *   x bf16 [T][H] (H % 8 == 0); prob_staging fp32 [num_nodes][max_tokens][P]
 *   from ep_restripe_prob (P % 4 == 0; NULL together with recv_prob_node to
 *   move rows only); is_token_in_node uint8 [T][num_nodes] from ep_get_layout
 *   (read on the sparse path only; may be NULL on the dense path);
 *   recv_x_node bf16 [num_nodes][max_tokens][H]; recv_prob_node fp32
 *   [num_nodes][max_tokens][P]; num_runs int32 [num_nodes][ceil(T/chunk_tokens)]
 *   or NULL. Requires T <= max_tokens, chunk_tokens >= 1.
 */
ep_status_t ep_dispatch_nodes(const void* x, const float* prob_staging,
                              const uint8_t* is_token_in_node, int32_t T, int32_t H,
                              int32_t num_nodes, int32_t P, int32_t max_tokens,
                              int32_t chunk_tokens, ep_node_mode_t mode, void* recv_x_node,
                              float* recv_prob_node, int32_t* num_runs, void* stream);

/* ------------------------------------------------------------------------- */
/* Combine                                                                   */
/* ------------------------------------------------------------------------- */

/* ep_combine -- bring every rank's expert output for a token back to the
 * token's position and reduce ([PR #347] 2.1 Feature; BF16 combine of 3.2.1):
 *   out[t][h] = bf16_rn( sum over r = 0, 1, ..., R-1 ascending with
 *                        s = slot[t][r] >= 0 of float(y[r][s][h]) )
 * accumulated in fp32 from +0 in exactly that order (one IEEE addition per
 * term, one rounding to bf16 at the end), so the result is deterministic. The
 * sum is unweighted: top-k weights belong to the expert. A token routed
 * nowhere gets +0. A slot >= max_tokens was never received: it is skipped and
 * raises EP_FLAG_CAPACITY.
 *   y    bf16 [R][max_tokens][H], H % 8 == 0
 *   slot int32 [T][R] from ep_get_layout
 *   out  bf16 [T][H]
 */
ep_status_t ep_combine(const void* y, const int32_t* slot, int32_t T, int32_t H, int32_t R,
                       int32_t max_tokens, void* out, int32_t* status, void* stream);

/* ep_combine_fp8 -- ep_combine for expert outputs kept in the FP8 row format of the
 * dispatch ([PR #347] 3.2.1: H E4M3 codes and one fp32 scale per 128 channels). The
 * pages show only the BF16 combine; this call reads each received row as the dispatch
 * wrote it, dequantises every channel to fp32(e4m3(q) * scale) (one fp32 rounding) and
 * reduces exactly as ep_combine does:
 *   out[t][h] = bf16_rn( sum over r ascending with s = slot[t][r] >= 0 of
 *                        fp32(e4m3(y[r][s][h]) * y_scales[r][s][h / 128]) )
 *   y        E4M3 codes [R][max_tokens][H], H % 128 == 0
 *   y_scales fp32 [R][max_tokens][H/128]
 *   slot     int32 [T][R] from ep_get_layout;  out bf16 [T][H]
 * R * max_tokens < 2^31. A slot >= max_tokens is skipped and raises EP_FLAG_CAPACITY.
 * NaN codes (0x7F, 0xFF) are outside the contract. */
ep_status_t ep_combine_fp8(const uint8_t* y, const float* y_scales, const int32_t* slot, int32_t T,
                           int32_t H, int32_t R, int32_t max_tokens, void* out, int32_t* status,
                           void* stream);

/* ep_combine_weights -- the combined top-k weights: the combine also returns the weight
 * rows the dispatch sent out ([PR #347] 2.1: the combine brings back what the dispatch
 * sent), reduced to token order:
 *   combined_w[t][j] = sum over r ascending with s = slot[t][r] >= 0 of
 *                      recv_topk_w[r][s][j]            (fp32 from +0)
 * Each rank's copy carries w_j for the slots whose expert it holds and +0 for the rest,
 * so after ep_dispatch this is the router's weight (0 for empty, out-of-range or
 * dropped slots).
 *   recv_topk_w fp32 [R][max_tokens][k] (1 <= k <= 32); slot int32 [T][R];
 *   combined_w fp32 [T][k]. A slot >= max_tokens is skipped and raises EP_FLAG_CAPACITY. */
ep_status_t ep_combine_weights(const float* recv_topk_w, const int32_t* slot, int32_t T, int32_t k,
                               int32_t R, int32_t max_tokens, float* combined_w, int32_t* status,
                               void* stream);

/* ------------------------------------------------------------------------- */
/* Expert-major path: dispatch + permute (fused or split) and its combine     */
/* ------------------------------------------------------------------------- */

/* After dispatch, a rank's tokens are permuted into local-expert order for the
 * expert GEMMs ([PR #634] commit "hybrid_ep: fix scan permute-fusion local-experts
 * sum array sizing"; "dispatch+permute" rows of its B300 results). The expert-major
 * slab of rank r holds its rows grouped by local expert l = 0 .. E/R-1, each group
 * in token order; the row of (token t, top-k slot j) with expert e on rank r is
 *   p = expert_offsets[e] - expert_offsets[r*(E/R)] + expert_slot[t][j].
 * A token with two experts on one rank has two rows there. */

/* Bytes of device workspace ep_get_expert_layout needs. */
size_t ep_expert_layout_workspace_size(int32_t T, int32_t E);

/* ep_get_expert_layout -- the per-local-expert sum array and scan:
 *   expert_offsets[e] = number of counted (t, j) with expert e' < e   [E+1] int32
 *   expert_slot[t][j] = number of counted (t', j') before (t, j) in token-then-slot
 *                       order with the same expert, or -1           [T][k] int32
 * A (t, j) counts when 0 <= topk_idx[t][j] < E and the id does not repeat an earlier
 * slot of the same row; ids >= E and repeats get -1 and raise EP_FLAG_BAD_EXPERT.
 *   topk_idx int64 [T][k], 1 <= k <= 32, 1 <= E <= 1024
 *   workspace: >= ep_expert_layout_workspace_size(T, E) bytes, 256-byte aligned,
 *     zero-filled before its first use; each completed call leaves it ready for the
 *     next (same header and stall hook as the ep_get_layout workspace)
 *   status: EP_FLAG_BAD_EXPERT, EP_FLAG_TIMEOUT, EP_FLAG_WORKSPACE */
ep_status_t ep_get_expert_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E,
                                 int32_t* expert_offsets, int32_t* expert_slot, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream);

/* ep_dispatch_permuted -- dispatch and permute fused (one launch): for every counted
 * (t, j), into rank r = e / (E/R) at row p (above):
 *   perm_x[r][p] = x[t], perm_src[r][p] = t, perm_w[r][p] = topk_w[t][j].
 *   x bf16 [T][H] (H % 8 == 0); topk_idx int64 / topk_w fp32 [T][k];
 *   expert_offsets / expert_slot from ep_get_expert_layout;
 *   perm_x bf16 [R][max_rows][H]; perm_src int32 [R][max_rows] (nullable);
 *   perm_w fp32 [R][max_rows] (nullable; needs topk_w); R * max_rows < 2^31.
 * p >= max_rows is dropped with EP_FLAG_CAPACITY; other rows are not written;
 * EP_FLAG_TIMEOUT as for ep_dispatch (bulk-copy row loads). */
ep_status_t ep_dispatch_permuted(const void* x, const int64_t* topk_idx, const float* topk_w,
                                 const int32_t* expert_offsets, const int32_t* expert_slot,
                                 int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                 int32_t max_rows, void* perm_x, int32_t* perm_src, float* perm_w,
                                 int32_t* status, void* stream);

/* ep_permute_received -- the receive phase of a split ("hook mode", [PR #347] 2.1
 * Feature: the send phase returns, the receive phase runs later as its own launch)
 * dispatch: the send phase is ep_dispatch into rank slabs; this call moves each
 * received row s < min(tokens_per_rank[r], max_tokens) of rank r, for every slot j
 * with local id l = recv_topk_idx[r][s][j] >= 0, to the same expert-major row the
 * fused path uses (t = recv_src_idx[r][s], e = r*(E/R) + l):
 *   perm_x[r][p] = recv_x[r][s], perm_src[r][p] = t, perm_w[r][p] = recv_topk_w[r][s][j].
 * The result equals ep_dispatch_permuted's. recv_* are ep_dispatch's bf16 outputs
 * ([R][max_tokens][H], [R][max_tokens], [R][max_tokens][k] x2; recv_topk_w nullable
 * when perm_w is NULL); tokens_per_rank from ep_get_layout. */
ep_status_t ep_permute_received(const void* recv_x, const int32_t* recv_src_idx,
                                const int32_t* recv_topk_idx, const float* recv_topk_w,
                                const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                                const int32_t* expert_slot, int32_t T, int32_t H, int32_t k,
                                int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                                void* perm_x, int32_t* perm_src, float* perm_w, int32_t* status,
                                void* stream);

/* ep_dispatch_permuted_ll -- the low-latency (decode-sized) form of the expert-major
 * dispatch: one launch computes the expert layout and moves the rows, with the same
 * results as ep_get_expert_layout followed by ep_dispatch_permuted (expert_offsets,
 * expert_slot, perm_x, perm_src, perm_w and the status flags). The pages name a
 * low-latency mode for small decode batches ([PR #347] "low-latency" kernels beside the
 * normal ones) without defining it; this is its single-GPU reading: no workspace, no
 * second launch, every CTA recomputing the small layout in shared memory.
 *   T <= 1024, T * k <= 8192, E <= 1024, E % R == 0; other arguments as
 *   ep_get_expert_layout / ep_dispatch_permuted. expert_offsets int32 [E+1] and
 *   expert_slot int32 [T][k] are outputs. T = 0 writes zero offsets. */
ep_status_t ep_dispatch_permuted_ll(const void* x, const int64_t* topk_idx, const float* topk_w,
                                    int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                    int32_t max_rows, int32_t* expert_offsets, int32_t* expert_slot,
                                    void* perm_x, int32_t* perm_src, float* perm_w, int32_t* status,
                                    void* stream);

/* ep_combine_permuted -- combine from expert-major slabs back to token order:
 *   out[t][h] = bf16_rn(acc), acc = 0; for j = 0 .. k-1 with a counted (t, j):
 *       acc = acc + topk_w[t][j] * float(y[r][p][h])   (topk_w given: one fp32
 *                                                        multiply, one fp32 add)
 *       acc = acc + float(y[r][p][h])                  (topk_w NULL)
 * in exactly that order, so the result is deterministic. Rows p >= max_rows were
 * never written: skipped with EP_FLAG_CAPACITY. A token with no counted entry gets +0.
 *   y bf16 [R][max_rows][H]; out bf16 [T][H]. */
ep_status_t ep_combine_permuted(const void* y, const int64_t* topk_idx, const float* topk_w,
                                const int32_t* expert_offsets, const int32_t* expert_slot,
                                int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                int32_t max_rows, void* out, int32_t* status, void* stream);

/* ep_combine_send -- the send phase of a split ("hook mode", [PR #347] 2.1 Feature: the
 * send phase runs and returns, the receive phase runs later as its own launch) combine;
 * the receive phase is ep_combine. It is the inverse of ep_permute_received: every rank
 * r takes, for each row s < min(tokens_per_rank[r], max_tokens) it received (token
 * t = recv_src_idx[r][s]), the expert-major rows of the token's local experts -- row
 * p = expert_offsets[e] - expert_offsets[r*(E/R)] + expert_slot[t][j] for every slot j
 * with local id l = recv_topk_idx[r][s][j] >= 0, e = r*(E/R) + l -- and reduces them into
 * its rank-level row:
 *   y_rank[r][s][h] = bf16_rn(acc), acc = 0; for j = 0 .. k-1 with such a row p:
 *       acc = acc + recv_topk_w[r][s][j] * float(y_perm[r][p][h])  (weights given: one
 *                                                                   fp32 multiply, one add)
 *       acc = acc + float(y_perm[r][p][h])                        (recv_topk_w NULL)
 * in exactly that order. ep_combine(y_rank, slot, ...) then completes the combine. Each
 * rank rounds its partial sum to bf16 once (the rank-level rows are bf16, like every
 * combine input), so the split result can differ from ep_combine_permuted's single fp32
 * sum in the last bits; it equals it bit for bit when no token has two experts on one
 * rank, the sum is unweighted and every token's expert ids ascend.
 *   y_perm bf16 [R][max_rows][H] (H % 8 == 0); recv_src_idx int32 [R][max_tokens],
 *   recv_topk_idx int32 / recv_topk_w fp32 [R][max_tokens][k] from ep_dispatch;
 *   tokens_per_rank from ep_get_layout; expert_offsets / expert_slot from
 *   ep_get_expert_layout; y_rank bf16 [R][max_tokens][H] (other rows not written);
 *   R * max_rows < 2^31, R * max_tokens < 2^31. p >= max_rows is skipped with
 *   EP_FLAG_CAPACITY. */
ep_status_t ep_combine_send(const void* y_perm, const int32_t* recv_src_idx, const int32_t* recv_topk_idx,
                            const float* recv_topk_w, const int32_t* tokens_per_rank,
                            const int32_t* expert_offsets, const int32_t* expert_slot, int32_t T,
                            int32_t H, int32_t k, int32_t E, int32_t R, int32_t max_tokens,
                            int32_t max_rows, void* y_rank, int32_t* status, void* stream);

/* ep_combine_permuted_ll -- the low-latency (decode-sized) form of ep_combine_permuted
 * (the pages name low-latency kernels beside the normal ones, [PR #347]): the same
 * arguments and bit-identical results, for T <= 1024 and E <= 1024, shaped for latency --
 * one CTA per (token, 256-vector slice of its row), the expert offsets and the token's
 * slots fetched together, then every source vector of the slice in flight at once. */
ep_status_t ep_combine_permuted_ll(const void* y, const int64_t* topk_idx, const float* topk_w,
                                   const int32_t* expert_offsets, const int32_t* expert_slot,
                                   int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                   int32_t max_rows, void* out, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
