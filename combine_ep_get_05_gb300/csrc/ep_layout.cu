// ep_layout.cu -- routing layout: per-expert / per-rank / per-node counts,
// is_token_in_rank / is_token_in_node and the stable slot of every (token, rank).
//
// The layout step is DeepEP's get_dispatch_layout ("[PR #347] Feature/sm free
// normal kernel", commit "add arg return_recv_hook for get_dispatch_layout");
// the slots are the scan of "[PR #634] Hybrid ep nixl restripe" (commit "fix
// scan permute-fusion local-experts sum array sizing"): slot[t][r] is the
// number of earlier tokens that also go to rank r.
//
// One launch; a tile of 256 tokens (thread = token) is handled by 1, 2, 4 or 8 CTAs
// ("parts"), each computing the whole tile's masks and prefix and writing the rows of
// its own share of the tile's 32-token warp groups, so that small batches spread their
// row stores over many SMs:
//   1. each thread reads its token's k expert ids, bumps a shared-memory expert
//      histogram and forms its rank bit mask (R <= 256: four 64-bit words);
//   2. a warp-level bit-matrix transpose gives, per rank, the 32-token membership
//      mask of each warp; popcounts give per-warp counts and in-warp prefixes;
//   3. the tile's per-rank counts are scanned across tiles with a decoupled
//      look-back: every (tile, rank) publishes one 64-bit word holding
//      {epoch, state, count}; state 1 = this tile's count only, state 2 = the
//      inclusive prefix; part 0 publishes, every part reads. CTA i * parts + p is
//      part p of tile i: CTAs are dispatched in index order, so a tile waits only on
//      tiles whose CTAs already run (the order single-pass scans rely on); every
//      wait is bounded in time and raises EP_FLAG_TIMEOUT when it gives up;
//   4. each part writes its warp groups' rows of is_token_in_rank / slot /
//      is_token_in_node as 16-byte vectors (the rows are contiguous);
//   5. expert and node counts are accumulated with atomics in the workspace and
//      each CTA then bumps a counter (release); the CTA that bumps it last moves
//      the counts to the outputs, zeroes the accumulators and the counter and
//      advances the epoch, so the workspace is ready for the next call without a
//      memset. Nothing but that last CTA waits on the counter.
#include <mutex>

#include "ep_common.cuh"
#include "ep_lookback.cuh"

namespace {

using namespace ep;

constexpr int kTileTokens = 256;  // = threads per CTA
constexpr int kTileWarps = kTileTokens / 32;
constexpr int kMaxRanks = 256;
constexpr int kMaxExperts = 8192;
constexpr int kMaxTopk = 32;
constexpr int kLookbackBatch = 16;
constexpr int kIdsPerPass = 8;  // expert ids a thread holds in registers at once

struct LayoutArgs {
    const int64_t* topk_idx;
    int T, k, E, R, rpn, N, epr, num_tiles;
    int parts;  // CTAs per tile (1, 2, 4 or 8); CTA (tile, part) writes warp groups part*8/parts ...
    int32_t* tokens_per_expert;
    int32_t* tokens_per_rank;
    int32_t* tokens_per_node;
    uint8_t* in_rank;
    uint8_t* in_node;
    int32_t* slot;
    ep_layout_ws_header_t* hdr;
    unsigned long long* words;  // [num_tiles][R]
    int32_t* acc_expert;        // [E]
    int32_t* acc_node;          // [N]
    int32_t* status;
};

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

inline int num_tiles_for(int T) { return T > 0 ? (T + kTileTokens - 1) / kTileTokens : 1; }

// Transpose of a 32 x 32 bit matrix held one row per lane (bit j of lane i =
// A[i][j]): returns column `lane`, i.e. bit i of the result = A[i][lane]. Five
// levels swap the off-diagonal blocks of size 16, 8, 4, 2, 1 between lane pairs.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
    const uint32_t low_cols[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int level = 0; level < 5; ++level) {
        const int s = 16 >> level;
        const uint32_t m = low_cols[level];
        const uint32_t y = __shfl_xor_sync(kFullMask, x, s);
        x = (lane & s) ? ((x & ~m) | ((y >> s) & m)) : ((x & m) | ((y & m) << s));
    }
    return x;
}

__global__ void __launch_bounds__(kTileTokens) layout_kernel(LayoutArgs a) {
    // the next kernel (a dispatch launched as a dependent launch) may be scheduled now: its
    // CTAs settle on the SMs this grid leaves free and wait there for its completion
    allow_dependents();
    extern __shared__ int32_t s_hist[];  // [E]
    __shared__ uint32_t s_mask[kTileWarps][kMaxRanks];
    __shared__ int32_t s_wpref[kTileWarps][kMaxRanks];
    __shared__ uint32_t s_nmask[kTileWarps][kMaxRanks];
    __shared__ uint32_t s_epoch, s_stall, s_done;

    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int tile = static_cast<int>(blockIdx.x) / a.parts;
    const int part = static_cast<int>(blockIdx.x) - tile * a.parts;
    const int wpp = kTileWarps / a.parts;  // warp groups this CTA writes: [w0, w0 + wpp)
    const int w0 = part * wpp;
    const bool own = warp >= w0 && warp < w0 + wpp;
    const int t0 = tile * kTileTokens;
    const int t = t0 + tid;
    const long long* row = reinterpret_cast<const long long*>(a.topk_idx) + static_cast<size_t>(t < a.T ? t : 0) * a.k;

    // the token's first expert ids are requested before anything else waits
    long long ev[kIdsPerPass];
#pragma unroll
    for (int i = 0; i < kIdsPerPass; ++i) ev[i] = (t < a.T && i < a.k) ? __ldg(row + i) : -1ll;
    if (tid == 0) {
        s_epoch = ld_relaxed_u32(&a.hdr->epoch) + 1u;
        s_stall = ld_relaxed_u32(&a.hdr->stall_tile);
    }
    for (int e = tid; e < a.E; e += kTileTokens) s_hist[e] = 0;
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const bool stalled = s_stall == static_cast<uint32_t>(tile) + 1u;

    // 1. token -> rank mask; expert histogram of this CTA's own warp groups
    uint64_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    bool bad = false;
    for (int j0 = 0; j0 < a.k; j0 += kIdsPerPass) {
        if (j0 > 0) {
#pragma unroll
            for (int i = 0; i < kIdsPerPass; ++i) ev[i] = (t < a.T && j0 + i < a.k) ? __ldg(row + j0 + i) : -1ll;
        }
#pragma unroll
        for (int i = 0; i < kIdsPerPass; ++i) {
            const long long e = ev[i];
            if (e < 0) continue;
            if (e >= a.E) {
                bad = true;
                continue;
            }
            if (own) atomicAdd(&s_hist[e], 1);
            const int r = static_cast<int>(e) / a.epr;
            const uint64_t bit = 1ull << (r & 63);
            if (r < 64) m0 |= bit;
            else if (r < 128) m1 |= bit;
            else if (r < 192) m2 |= bit;
            else m3 |= bit;
        }
    }
    if (bad && own) raise_flag(a.status, EP_FLAG_BAD_EXPERT);

    // 2. per-rank warp membership masks: for each chunk of 32 ranks, the warp holds a
    //    32 x 32 bit matrix (lane = token, bit = rank); transposing it leaves in lane j
    //    the 32-token mask of rank 32c + j (what a ballot per rank would give).
    for (int c = 0; c * 32 < a.R; ++c) {
        const uint64_t word = c < 2 ? m0 : (c < 4 ? m1 : (c < 6 ? m2 : m3));
        const uint32_t m = transpose32(static_cast<uint32_t>(word >> ((c & 1) * 32)), lane);
        if (c * 32 + lane < a.R) s_mask[warp][c * 32 + lane] = m;
    }
    __syncthreads();

    // 3. the tile's per-rank counts; part 0 publishes them first (later tiles wait on them)
    uint32_t agg = 0;
    if (tid < a.R) {
        int run = 0;
        for (int w = 0; w < kTileWarps; ++w) {
            s_wpref[w][tid] = run;
            run += __popc(s_mask[w][tid]);
        }
        agg = static_cast<uint32_t>(run);
        if (part == 0 && !stalled)
            st_relaxed_u64(a.words + static_cast<size_t>(tile) * a.R + tid,
                           pack_word(epoch, tile == 0 ? kStatePrefix : kStateAggregate, agg));
    }
    // expert and node counts of the own warp groups -> workspace accumulators; the node
    // masks are formed by the highest threads, which take no part in the look-back when
    // R is small
    for (int e = tid; e < a.E; e += kTileTokens) {
        const int c = s_hist[e];
        if (c != 0) atomicAdd(&a.acc_expert[e], c);
    }
    {
        const int n = kTileTokens - 1 - tid;
        if (n < a.N) {
            int c = 0;
            for (int w = w0; w < w0 + wpp; ++w) {
                uint32_t m = 0;
                for (int q = 0; q < a.rpn; ++q) m |= s_mask[w][n * a.rpn + q];
                s_nmask[w][n] = m;
                c += __popc(m);
            }
            if (c != 0) atomicAdd(&a.acc_node[n], c);
        }
    }

    // this CTA's accumulator contributions are issued: the barrier orders every thread's
    // atomics before the release of the counter, which the last warp takes (off the
    // look-back's warps when R is small); the answer is needed only after the scan
    __syncthreads();
    uint32_t done_before = 0;
    if (tid == kTileTokens - 1) done_before = atom_add_acq_rel_u32(&a.hdr->done, 1u);

    // per-rank scan across tiles (decoupled look-back), thread r owns rank r; every part
    // of the tile reads the same words, part 0 alone publishes the inclusive prefix
    if (tid < a.R) {
        const int r = tid;
        bool timed_out = false;
        const uint32_t excl = lookback_exclusive<kLookbackBatch>(a.words, a.R, tile, r, epoch, timed_out);
        if (timed_out) raise_flag(a.status, EP_FLAG_TIMEOUT);
        if (part == 0 && tile > 0 && !stalled)
            st_relaxed_u64(a.words + static_cast<size_t>(tile) * a.R + r, pack_word(epoch, kStatePrefix, excl + agg));
        for (int w = w0; w < w0 + wpp; ++w) s_wpref[w][r] += static_cast<int32_t>(excl);
        if (part == 0 && tile == a.num_tiles - 1) a.tokens_per_rank[r] = static_cast<int32_t>(excl + agg);
    }
    if (tid == kTileTokens - 1) s_done = done_before;
    __syncthreads();
    const uint32_t done = s_done;
    const uint32_t ctas = static_cast<uint32_t>(a.num_tiles * a.parts);

    // 4. rows of is_token_in_rank / slot / is_token_in_node of the own warp groups: one
    //    contiguous run per array (the groups start at token t0 + 32 * w0), written as
    //    16-byte vectors, consecutive threads on consecutive vectors; entry f of the run
    //    is (token f / width, column f % width). The bytes past the last whole vector
    //    (only at the end of the batch) are written one by one.
    {
        const int first = t0 + 32 * w0;
        const int ntok = a.T - first < 32 * wpp ? a.T - first : 32 * wpp;
        if (ntok > 0) {
            // slot: 4 entries per vector; s_wpref holds the rank's slot of the first
            // token of each own warp group
            {
                int32_t* base = a.slot + static_cast<size_t>(first) * a.R;
                const int ne = ntok * a.R;
                for (int c = tid; c < ne / 4; c += kTileTokens) {
                    int u = (4 * c) / a.R;
                    int r = 4 * c - u * a.R;
                    int32_t v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int w = w0 + (u >> 5);
                        const uint32_t m = s_mask[w][r];
                        const uint32_t b = 1u << (u & 31);
                        v[q] = (m & b) ? s_wpref[w][r] + __popc(m & (b - 1u)) : -1;
                        if (++r == a.R) {
                            r = 0;
                            ++u;
                        }
                    }
                    st_v4(base + 4 * c, make_uint4(static_cast<uint32_t>(v[0]), static_cast<uint32_t>(v[1]),
                                                   static_cast<uint32_t>(v[2]), static_cast<uint32_t>(v[3])));
                }
                for (int f = (ne & ~3) + tid; f < ne; f += kTileTokens) {
                    const int u = f / a.R, r = f - (f / a.R) * a.R;
                    const int w = w0 + (u >> 5);
                    const uint32_t m = s_mask[w][r];
                    const uint32_t b = 1u << (u & 31);
                    base[f] = (m & b) ? s_wpref[w][r] + __popc(m & (b - 1u)) : -1;
                }
            }
            // membership bytes of one mask table, 16 entries per vector
            auto write_bits = [&](uint8_t* base, const uint32_t (*mask)[kMaxRanks], int width) {
                const int nb = ntok * width;
                for (int c = tid; c < nb / 16; c += kTileTokens) {
                    int u = (16 * c) / width;
                    int r = 16 * c - u * width;
                    uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        wd[q >> 2] |= ((mask[w0 + (u >> 5)][r] >> (u & 31)) & 1u) << (8 * (q & 3));
                        if (++r == width) {
                            r = 0;
                            ++u;
                        }
                    }
                    st_v4(base + 16 * c, make_uint4(wd[0], wd[1], wd[2], wd[3]));
                }
                for (int f = (nb & ~15) + tid; f < nb; f += kTileTokens) {
                    const int u = f / width, r = f - (f / width) * width;
                    base[f] = static_cast<uint8_t>((mask[w0 + (u >> 5)][r] >> (u & 31)) & 1u);
                }
            };
            write_bits(a.in_rank + static_cast<size_t>(first) * a.R, s_mask, a.R);
            if (a.in_node != nullptr) write_bits(a.in_node + static_cast<size_t>(first) * a.N, s_nmask, a.N);
        }
    }

    // 5. the CTA that counted itself last moves the accumulated counts out and resets
    //    the workspace (every CTA read the epoch before it counted itself)
    if (done >= ctas) {
        // the workspace was not at rest (not zero-filled, or shared by concurrent
        // calls): report it; the caller zero-fills it again
        if (tid == 0) raise_flag(a.status, EP_FLAG_WORKSPACE);
    } else if (done == ctas - 1u) {
        // the counter's acquire (last thread) and the barrier after the scan order the
        // other CTAs' accumulator atomics before these reads
        for (int e = tid; e < a.E; e += kTileTokens) a.tokens_per_expert[e] = atomicExch(&a.acc_expert[e], 0);
        for (int n = tid; n < a.N; n += kTileTokens) a.tokens_per_node[n] = atomicExch(&a.acc_node[n], 0);
        if (tid == 0) {
            atomicExch(&a.hdr->done, 0u);
            atomicExch(&a.hdr->epoch, epoch);
        }
    }
}

// CTAs per tile: the largest power of two (at most one CTA per warp group) that keeps
// the grid within one CTA per SM, so that the batch's row stores spread over most SMs
// (one SM issues scattered row stores at only a few tens of GB/s).
int parts_for(int num_tiles) {
    const long long sms = sm_count();
    int parts = 1;
    while (parts < kTileWarps && static_cast<long long>(num_tiles) * (2 * parts) <= sms) parts *= 2;
    return parts;
}

std::atomic<int> g_smem_attr_set[kMaxDevices];

}  // namespace

// Workspace layout: [header | expert accumulators (kMaxExperts) | node accumulators
// (kMaxRanks) | tile words (num_tiles x R)]. The accumulators sit at fixed offsets
// sized for the largest E and N, so a workspace that is at rest stays valid for
// any later call whatever its T, E, R; the tile words carry their epoch, so
// stale words of earlier calls are never mistaken for current ones.
constexpr size_t kOffExperts = 256;
constexpr size_t kOffNodes = kOffExperts + kMaxExperts * sizeof(int32_t);
constexpr size_t kOffWords = kOffNodes + kMaxRanks * sizeof(int32_t);

namespace {

// Argument checks common to both entry points (the workspace is checked by the caller).
bool layout_args_ok(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R, int32_t ranks_per_node,
                    const int32_t* tokens_per_expert, const int32_t* tokens_per_rank, const int32_t* tokens_per_node,
                    const uint8_t* is_token_in_rank, const uint8_t* is_token_in_node, const int32_t* slot) {
    using namespace ep;
    if (T < 0 || T >= (1 << 30) || k < 1 || k > kMaxTopk || R < 1 || R > kMaxRanks || E < R ||
        E > kMaxExperts || E % R != 0 || ranks_per_node < 0 || ranks_per_node > R ||
        (ranks_per_node > 0 && R % ranks_per_node != 0))
        return false;
    const bool nodes = ranks_per_node > 0;
    if (tokens_per_expert == nullptr || tokens_per_rank == nullptr) return false;
    if (T > 0 && (topk_idx == nullptr || is_token_in_rank == nullptr || slot == nullptr)) return false;
    if (nodes && (tokens_per_node == nullptr || (T > 0 && is_token_in_node == nullptr))) return false;
    return aligned16_or_null(topk_idx) && aligned16(tokens_per_expert) && aligned16(tokens_per_rank) &&
           aligned16_or_null(tokens_per_node) && aligned16_or_null(is_token_in_rank) &&
           aligned16_or_null(is_token_in_node) && aligned16_or_null(slot);
}

// Packs the arguments, points them into the workspace and launches the layout kernel.
ep_status_t launch_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R, int32_t ranks_per_node,
                          int32_t* tokens_per_expert, int32_t* tokens_per_rank, int32_t* tokens_per_node,
                          uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot, char* ws,
                          int32_t* status, cudaStream_t stream) {
    using namespace ep;
    const bool nodes = ranks_per_node > 0;
    LayoutArgs a{};
    a.topk_idx = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.R = R;
    a.rpn = nodes ? ranks_per_node : 1;
    a.N = nodes ? R / ranks_per_node : 0;
    a.epr = E / R;
    a.num_tiles = num_tiles_for(T);
    a.parts = parts_for(a.num_tiles);
    a.tokens_per_expert = tokens_per_expert;
    a.tokens_per_rank = tokens_per_rank;
    a.tokens_per_node = nodes ? tokens_per_node : nullptr;
    a.in_rank = is_token_in_rank;
    a.in_node = nodes ? is_token_in_node : nullptr;
    a.slot = slot;
    a.hdr = reinterpret_cast<ep_layout_ws_header_t*>(ws);
    a.acc_expert = reinterpret_cast<int32_t*>(ws + kOffExperts);
    a.acc_node = reinterpret_cast<int32_t*>(ws + kOffNodes);
    a.words = reinterpret_cast<unsigned long long*>(ws + kOffWords);
    a.status = status;
    const ep_status_t attr =
        ensure_dynamic_smem(g_smem_attr_set, layout_kernel, kMaxExperts * static_cast<int>(sizeof(int32_t)));
    if (attr != EP_OK) return attr;
    layout_kernel<<<a.num_tiles * a.parts, kTileTokens, static_cast<size_t>(E) * sizeof(int32_t), stream>>>(a);
    return check_launch();
}

}  // namespace

extern "C" size_t ep_layout_workspace_size(int32_t T, int32_t E, int32_t R, int32_t ranks_per_node) {
    (void)ranks_per_node;
    if (T < 0 || E <= 0 || R <= 0) return 0;
    return kOffWords + align256(static_cast<size_t>(num_tiles_for(T)) * R * sizeof(unsigned long long));
}

extern "C" ep_status_t ep_get_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                                     int32_t ranks_per_node, int32_t* tokens_per_expert,
                                     int32_t* tokens_per_rank, int32_t* tokens_per_node,
                                     uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot,
                                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    using namespace ep;
    if (!layout_args_ok(topk_idx, T, k, E, R, ranks_per_node, tokens_per_expert, tokens_per_rank, tokens_per_node,
                        is_token_in_rank, is_token_in_node, slot))
        return EP_ERR_INVALID;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < ep_layout_workspace_size(T, E, R, ranks_per_node))
        return EP_ERR_INVALID;
    return launch_layout(topk_idx, T, k, E, R, ranks_per_node, tokens_per_expert, tokens_per_rank, tokens_per_node,
                         is_token_in_rank, is_token_in_node, slot, static_cast<char*>(workspace), status,
                         as_stream(stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant: ep_get_layout_noalloc
// ---------------------------------------------------------------------------
// Some callers cannot hand the layout a workspace: code that runs where device
// allocation is forbidden or unavailable (a caller with a fixed, pre-planned
// memory budget and no allocator of its own, a host runtime that only passes
// pointers to tensors it already owns, or a plain C caller without a CUDA
// allocator). For them the workspace lives in this fixed-size device array
// instead. It is part of the library image: every GPU that loads the library
// holds these bytes until the process exits. All calls on a device share it,
// so calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race and must not be issued.
static __device__ __align__(256) unsigned char g_layout_scratch[EP_LAYOUT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoAllocScratchBytes = EP_LAYOUT_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes > kOffWords, "scratch must hold the fixed workspace part");

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device (host code must not use the
// symbol itself: on the host it names a host-side shadow, not device memory). The address
// is looked up on every call (cudaGetSymbolAddress is a cheap host call) and remembered,
// so a context created anew (after cudaDeviceReset) is picked up at once. A call made
// while `stream` is capturing does not look it up (the lookup may have to load the
// module) and uses the remembered address; with none remembered it is refused
// (EP_ERR_INVALID) before anything is queued.
ep_status_t scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err);
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_INVALID;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    err = cudaStreamIsCapturing(stream, &cap);
    if (err != cudaSuccess) return cuda_fail(err);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (err != cudaSuccess || p == nullptr) return cuda_fail(err != cudaSuccess ? err : cudaErrorInvalidSymbol);
        g_scratch_ptr[dev] = p;
    } else if (g_scratch_ptr[dev] == nullptr) {
        return EP_ERR_INVALID;
    }
    *out = g_scratch_ptr[dev];
    return EP_OK;
}

}  // namespace

extern "C" ep_status_t ep_get_layout_noalloc(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E, int32_t R,
                                             int32_t ranks_per_node, int32_t* tokens_per_expert,
                                             int32_t* tokens_per_rank, int32_t* tokens_per_node,
                                             uint8_t* is_token_in_rank, uint8_t* is_token_in_node, int32_t* slot,
                                             int32_t* status, void* stream) {
    using namespace ep;
    if (!layout_args_ok(topk_idx, T, k, E, R, ranks_per_node, tokens_per_expert, tokens_per_rank, tokens_per_node,
                        is_token_in_rank, is_token_in_node, slot))
        return EP_ERR_INVALID;
    const size_t need = ep_layout_workspace_size(T, E, R, ranks_per_node);
    if (need > kNoAllocScratchBytes) return EP_ERR_SCRATCH;

    void* scratch = nullptr;
    ep_status_t st = scratch_address(as_stream(stream), &scratch);
    if (st != EP_OK) return st;
    // the array keeps the previous call's contents: zero the part this call uses
    const cudaError_t err = cudaMemsetAsync(scratch, 0, need, as_stream(stream));
    if (err != cudaSuccess) return cuda_fail(err);
    return launch_layout(topk_idx, T, k, E, R, ranks_per_node, tokens_per_expert, tokens_per_rank, tokens_per_node,
                         is_token_in_rank, is_token_in_node, slot, static_cast<char*>(scratch), status,
                         as_stream(stream));
}
