// ep_permute.cu -- expert-major ("dispatch + permute") path: the expert layout,
// the fused permuted dispatch, the receive-side permute of a split (hook-mode)
// dispatch, and the combine from expert-major slabs.
//
// "[PR #634] Hybrid ep nixl restripe": commit "hybrid_ep: fix scan permute-fusion
// local-experts sum array sizing" and the dispatch+permute rows of its B300
// results -- after dispatch, each rank's tokens are permuted into local-expert
// order using a scan over the tokens and a per-local-expert sum array.
// "[PR #347] Feature/sm free normal kernel", 2.1 Feature: in hook mode the send
// phase runs first and the receive phase later, as its own launch.
//
// Expert-major slab of rank r: rows grouped by local expert l = 0, 1, ..., E/R-1,
// each group in token order; the row of (token t, top-k slot j) with expert e is
//   p = expert_offsets[e] - expert_offsets[r*(E/R)] + expert_slot[t][j].
#include <cstdio>

#include "ep_common.cuh"
#include "ep_lookback.cuh"
#include "ep_scatter.cuh"

namespace {

using namespace ep;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxExpertsPerm = 1024;  // expert layout: experts held per tile in shared memory
constexpr int kMaxTopk = 32;
constexpr int kUnroll = 8;
constexpr int kBatch = 8;
constexpr int kLookbackBatch = 8;

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }
inline int num_tiles_for(int T) { return T > 0 ? (T + kThreads - 1) / kThreads : 1; }

// ---------------------------------------------------------------------------
// Expert layout
// ---------------------------------------------------------------------------

struct ExpertLayoutArgs {
    const int64_t* topk_idx;
    int T, k, E, num_tiles;
    int32_t* offsets;  // [E+1]
    int32_t* eslot;    // [T][k]
    ep_layout_ws_header_t* hdr;
    unsigned long long* words;  // [num_tiles][E]
    int32_t* status;
};

// One tile of 256 tokens per CTA (thread = token); tile i is CTA i (CTAs are dispatched
// in index order, so a tile waits only on tiles whose CTAs already run). Each thread reads
// its token's ids (eight loads in flight at a time) and keeps, per top-k slot, the expert
// the entry counts for (in range and the first occurrence in the row) or -1, in shared
// memory. Each warp builds, per expert, the 32-bit mask of its tokens that chose the
// expert (shared-memory atomic ORs: the result does not depend on their order); a
// token's rank among the warp's tokens with the same expert is the popcount of the mask
// below its lane. Per-expert tile counts are scanned across tiles by a decoupled
// look-back over epoch-tagged words (bounded waits); the tile holding the last tokens,
// which ends up with every expert's total, writes the offsets.
__global__ void __launch_bounds__(kThreads, 2) expert_layout_kernel(ExpertLayoutArgs a) {
    extern __shared__ uint32_t smem[];
    uint32_t* s_emask = smem;                                              // [kWarps][E]
    int32_t* s_wpref = reinterpret_cast<int32_t*>(smem + kWarps * a.E);  // [kWarps][E]
    int32_t* s_tpref = s_wpref + kWarps * a.E;                           // [E]
    int32_t* s_total = s_tpref + a.E;                                    // [E]
    int32_t* s_ex = s_total + a.E;                                       // [k][kThreads]
    __shared__ uint32_t s_epoch, s_stall, s_done;
    __shared__ int32_t s_part[kThreads];

    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int tile = static_cast<int>(blockIdx.x);
    const int t = tile * kThreads + tid;
    const long long* row = reinterpret_cast<const long long*>(a.topk_idx) + static_cast<size_t>(t < a.T ? t : 0) * a.k;

    long long ev[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) ev[i] = (t < a.T && i < a.k) ? __ldg(row + i) : -1ll;
    if (tid == 0) {
        s_epoch = ld_relaxed_u32(&a.hdr->epoch) + 1u;
        s_stall = ld_relaxed_u32(&a.hdr->stall_tile);
    }
    for (int e = lane; e < a.E; e += 32) s_emask[warp * a.E + e] = 0u;
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const bool stalled = s_stall == static_cast<uint32_t>(tile) + 1u;

    bool bad = false;
    for (int j0 = 0; j0 < a.k; j0 += kBatch) {
        if (j0 > 0) {
#pragma unroll
            for (int i = 0; i < kBatch; ++i) ev[i] = (t < a.T && j0 + i < a.k) ? __ldg(row + j0 + i) : -1ll;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int j = j0 + i;
            if (j >= a.k) break;
            const long long e = ev[i];
            int x = -1;
            if (t < a.T && e >= 0) {
                if (e >= a.E) {
                    bad = true;
                } else {
                    // a repeat of an earlier slot of the row counts once
                    bool rep = false;
#pragma unroll
                    for (int ii = 0; ii < i; ++ii) rep |= ev[ii] == e;
                    for (int jj = 0; jj < j0; ++jj) rep |= s_ex[jj * kThreads + tid] == static_cast<int>(e);
                    if (rep) bad = true;
                    else x = static_cast<int>(e);
                }
            }
            s_ex[j * kThreads + tid] = x;
            if (x >= 0) atomicOr(&s_emask[warp * a.E + x], 1u << lane);
        }
    }
    if (bad) raise_flag(a.status, EP_FLAG_BAD_EXPERT);
    __syncthreads();

    for (int e = tid; e < a.E; e += kThreads) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            s_wpref[w * a.E + e] = run;
            run += __popc(s_emask[w * a.E + e]);
        }
        const uint32_t agg = static_cast<uint32_t>(run);
        unsigned long long* my_word = a.words + static_cast<size_t>(tile) * a.E + e;
        if (!stalled) st_relaxed_u64(my_word, pack_word(epoch, tile == 0 ? kStatePrefix : kStateAggregate, agg));
        bool timed_out = false;
        const uint32_t excl = lookback_exclusive<kLookbackBatch>(a.words, a.E, tile, e, epoch, timed_out);
        if (timed_out) raise_flag(a.status, EP_FLAG_TIMEOUT);
        if (tile > 0 && !stalled) st_relaxed_u64(my_word, pack_word(epoch, kStatePrefix, excl + agg));
        s_tpref[e] = static_cast<int32_t>(excl);
        s_total[e] = static_cast<int32_t>(excl + agg);
    }
    __syncthreads();

    // every CTA read the epoch before it counts itself here; the last one resets
    uint32_t done_before = 0;
    if (tid == kThreads - 1) done_before = atom_add_acq_rel_u32(&a.hdr->done, 1u);

    // the tile with the last tokens knows every expert's total: write the offsets
    if (tile == a.num_tiles - 1) {
        const int per = (a.E + kThreads - 1) / kThreads;
        const int e0 = tid * per;
        int sum = 0;
        for (int i = 0; i < per; ++i)
            if (e0 + i < a.E) sum += s_total[e0 + i];
        // block exclusive scan of the per-thread sums (warp shuffles, then warp totals)
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) s_part[warp] = incl;
        __syncthreads();
        int warp_base = 0;
        for (int w = 0; w < warp; ++w) warp_base += s_part[w];
        int run = warp_base + incl - sum;
        for (int i = 0; i < per; ++i) {
            if (e0 + i < a.E) {
                a.offsets[e0 + i] = run;
                run += s_total[e0 + i];
            }
        }
        if (tid == kThreads - 1) a.offsets[a.E] = warp_base + incl;
    }

    if (t < a.T) {
        const uint32_t below = (1u << lane) - 1u;
        for (int j = 0; j < a.k; ++j) {
            const int e = s_ex[j * kThreads + tid];
            int32_t v = -1;
            if (e >= 0) v = s_tpref[e] + s_wpref[warp * a.E + e] + __popc(s_emask[warp * a.E + e] & below);
            a.eslot[static_cast<size_t>(t) * a.k + j] = v;
        }
    }

    if (tid == kThreads - 1) s_done = done_before;
    __syncthreads();
    const uint32_t done = s_done;
    if (done >= static_cast<uint32_t>(a.num_tiles)) {
        if (tid == 0) raise_flag(a.status, EP_FLAG_WORKSPACE);
    } else if (done == static_cast<uint32_t>(a.num_tiles - 1) && tid == 0) {
        atomicExch(&a.hdr->done, 0u);
        atomicExch(&a.hdr->epoch, epoch);
    }
}

// ---------------------------------------------------------------------------
// Row copies shared by the permuted dispatch and the receive-side permute
// ---------------------------------------------------------------------------

// copy one row of nvec 16-byte vectors to nd destination rows (row indices in s_row)
__device__ __forceinline__ void copy_row(const uint4* src, uint4* base, const long long* s_row, int nd, int nvec) {
    const int lane = lane_id();
    for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) buf[u] = ld_stream_v4(src + v);
        }
        for (int d = 0; d < nd; ++d) {
            uint4* dst = base + static_cast<size_t>(s_row[d]) * nvec;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) st_v4(dst + v, buf[u]);
            }
        }
    }
}

// Destinations of (token t): the rows of its counted top-k entries, in slot order.
// Lane j handles slot j (k <= 32). Returns their number; s_row/s_j get row and slot.
__device__ __forceinline__ int permuted_destinations(const int64_t* topk_idx, const int32_t* offsets,
                                                     const int32_t* eslot, int t, int k, int E, int R,
                                                     int max_rows, long long* s_row, int* s_j, int32_t* status) {
    const int lane = lane_id();
    const int epr = E / R;
    bool ok = false, over = false;
    long long rowi = 0;
    if (lane < k) {
        const int32_t sl = eslot[static_cast<size_t>(t) * k + lane];
        const int64_t e = topk_idx[static_cast<size_t>(t) * k + lane];
        if (sl >= 0 && e >= 0 && e < E) {
            const int r = static_cast<int>(e) / epr;
            const int p = offsets[e] - offsets[r * epr] + sl;
            if (p >= 0 && p < max_rows) {
                ok = true;
                rowi = static_cast<long long>(r) * max_rows + p;
            } else {
                over = true;
            }
        }
    }
    const uint32_t m = __ballot_sync(kFullMask, ok);
    if (ok) {
        const int pos = __popc(m & lanemask_lt());
        s_row[pos] = rowi;
        s_j[pos] = lane;
    }
    if (__any_sync(kFullMask, over) && lane == 0) raise_flag(status, EP_FLAG_CAPACITY);
    __syncwarp();
    return __popc(m);
}

struct PermDispatchArgs {
    const uint16_t* x;
    const int64_t* topk_idx;
    const float* topk_w;
    const int32_t* offsets;
    const int32_t* eslot;
    int T, H, k, E, R, max_rows;
    uint16_t* perm_x;
    int32_t* perm_src;
    float* perm_w;
    int32_t* status;
};

// Fused dispatch + permute: warp per token, the row is read once and stored to the
// expert-major row of each of its counted top-k entries.
__global__ void __launch_bounds__(kThreads) dispatch_permuted_kernel(PermDispatchArgs a) {
    __shared__ long long s_row[kWarps][kMaxTopk];
    __shared__ int s_j[kWarps][kMaxTopk];
    const int lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = a.H / 8;
    for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
        const int nd = permuted_destinations(a.topk_idx, a.offsets, a.eslot, t, a.k, a.E, a.R, a.max_rows,
                                             s_row[warp], s_j[warp], a.status);
        if (lane < nd) {
            const size_t row = static_cast<size_t>(s_row[warp][lane]);
            if (a.perm_src != nullptr) a.perm_src[row] = t;
            if (a.perm_w != nullptr) a.perm_w[row] = a.topk_w[static_cast<size_t>(t) * a.k + s_j[warp][lane]];
        }
        copy_row(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H),
                 reinterpret_cast<uint4*>(a.perm_x), s_row[warp], nd, nvec);
        __syncwarp();
    }
}

// the fused dispatch + permute through the shared bulk-copy scatter (ep_scatter.cuh)
struct PermScatter {
    PermDispatchArgs a;
    char* dst;
    uint32_t row_bytes;
    int32_t* status;
    __device__ int items() const { return a.T; }
    __device__ const void* source(int t) const { return a.x + static_cast<size_t>(t) * a.H; }
    __device__ int destinations(int t, long long* rows, int* aux) const {
        return permuted_destinations(a.topk_idx, a.offsets, a.eslot, t, a.k, a.E, a.R, a.max_rows, rows, aux,
                                     a.status);
    }
    __device__ void side_work(int t, int nd, const long long* rows, const int* aux) const {
        const int lane = lane_id();
        if (lane < nd) {
            const size_t row = static_cast<size_t>(rows[lane]);
            if (a.perm_src != nullptr) a.perm_src[row] = t;
            if (a.perm_w != nullptr) a.perm_w[row] = a.topk_w[static_cast<size_t>(t) * a.k + aux[lane]];
        }
    }
    __device__ void prologue() const {}
};

struct PermuteRecvArgs {
    const uint16_t* recv_x;
    const int32_t* recv_src;
    const int32_t* recv_tidx;
    const float* recv_tw;
    const int32_t* tokens_per_rank;
    const int32_t* offsets;
    const int32_t* eslot;
    int T, H, k, E, R, max_tokens, max_rows;
    uint16_t* perm_x;
    int32_t* perm_src;
    float* perm_w;
    int32_t* status;
};

// Receive phase of a split dispatch: warp per received row. The CTA first turns the
// per-rank received counts into a prefix so that warps walk only rows that exist.
__global__ void __launch_bounds__(kThreads) permute_received_kernel(PermuteRecvArgs a) {
    __shared__ long long s_row[kWarps][kMaxTopk];
    __shared__ int s_j[kWarps][kMaxTopk];
    __shared__ int s_base[257];
    const int lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = a.H / 8;
    const int epr = a.E / a.R;
    if (warp == 0) {  // exclusive prefix of the received counts, 32 ranks per step
        int carry = 0;
        for (int r0 = 0; r0 < a.R; r0 += 32) {
            const int r = r0 + lane;
            int c = 0;
            if (r < a.R) {
                c = a.tokens_per_rank[r];
                c = c < 0 ? 0 : (c < a.max_tokens ? c : a.max_tokens);
            }
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            if (r < a.R) s_base[r] = carry + incl - c;
            carry += __shfl_sync(kFullMask, incl, 31);
        }
        if (lane == 0) s_base[a.R] = carry;
    }
    __syncthreads();
    const int total = s_base[a.R];
    for (int q = blockIdx.x * kWarps + warp; q < total; q += gridDim.x * kWarps) {
        int lo = 0, hi = a.R;  // last r with s_base[r] <= q
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_base[mid] <= q) lo = mid;
            else hi = mid;
        }
        const int r = lo;
        const int s = q - s_base[r];
        const size_t in_row = static_cast<size_t>(r) * a.max_tokens + s;
        const int t = a.recv_src[in_row];
        bool ok = false, over = false;
        long long rowi = 0;
        if (lane < a.k && t >= 0 && t < a.T) {
            const int l = a.recv_tidx[in_row * a.k + lane];
            const int32_t sl = a.eslot[static_cast<size_t>(t) * a.k + lane];
            if (l >= 0 && l < epr && sl >= 0) {
                const int e = r * epr + l;
                const int p = a.offsets[e] - a.offsets[r * epr] + sl;
                if (p >= 0 && p < a.max_rows) {
                    ok = true;
                    rowi = static_cast<long long>(r) * a.max_rows + p;
                } else {
                    over = true;
                }
            }
        }
        const uint32_t m = __ballot_sync(kFullMask, ok);
        if (ok) {
            const int pos = __popc(m & lanemask_lt());
            s_row[warp][pos] = rowi;
            s_j[warp][pos] = lane;
        }
        if (__any_sync(kFullMask, over) && lane == 0) raise_flag(a.status, EP_FLAG_CAPACITY);
        __syncwarp();
        const int nd = __popc(m);
        if (lane < nd) {
            const size_t row = static_cast<size_t>(s_row[warp][lane]);
            if (a.perm_src != nullptr) a.perm_src[row] = t;
            if (a.perm_w != nullptr) a.perm_w[row] = a.recv_tw[in_row * a.k + s_j[warp][lane]];
        }
        copy_row(reinterpret_cast<const uint4*>(a.recv_x + in_row * a.H), reinterpret_cast<uint4*>(a.perm_x),
                 s_row[warp], nd, nvec);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Combine from expert-major slabs
// ---------------------------------------------------------------------------

struct CombinePermArgs {
    const uint16_t* y;
    const int64_t* topk_idx;
    const float* topk_w;  // nullable: unweighted
    const int32_t* offsets;
    const int32_t* eslot;
    int T, H, k, E, R, max_rows;
    uint16_t* out;
    int32_t* status;
};

// Items of (token, 32 output vectors), contiguous per CTA; per item the lanes j < k
// resolve the token's expert-major rows, then up to 8 source vectors are loaded at
// once and accumulated strictly in slot order: acc = acc + w_j * y (one fp32 multiply
// and one fp32 add per term, never fused), or acc = acc + y when unweighted.
__global__ void __launch_bounds__(kThreads, 4) combine_permuted_kernel(CombinePermArgs a) {
    __shared__ long long s_src[kWarps][kMaxTopk];
    __shared__ float s_w[kWarps][kMaxTopk];
    const int lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = a.H / 8;
    const int ngroups = (nvec + 31) / 32;
    const long long items = static_cast<long long>(a.T) * ngroups;
    const long long i0 = static_cast<long long>(blockIdx.x) * items / gridDim.x;
    const long long i1 = static_cast<long long>(blockIdx.x + 1) * items / gridDim.x;
    const uint4* ys = reinterpret_cast<const uint4*>(a.y);
    uint4* os = reinterpret_cast<uint4*>(a.out);
    const int epr = a.E / a.R;
    for (long long it = i0 + warp; it < i1; it += kWarps) {
        const int t = static_cast<int>(it / ngroups);
        const int v = static_cast<int>(it - static_cast<long long>(t) * ngroups) * 32 + lane;
        bool ok = false, over = false;
        long long rowi = 0;
        float wj = 1.0f;
        if (lane < a.k) {
            const int32_t sl = a.eslot[static_cast<size_t>(t) * a.k + lane];
            const int64_t e = a.topk_idx[static_cast<size_t>(t) * a.k + lane];
            if (sl >= 0 && e >= 0 && e < a.E) {
                const int r = static_cast<int>(e) / epr;
                const int p = a.offsets[e] - a.offsets[r * epr] + sl;
                if (p >= 0 && p < a.max_rows) {
                    ok = true;
                    rowi = (static_cast<long long>(r) * a.max_rows + p) * nvec;
                    if (a.topk_w != nullptr) wj = a.topk_w[static_cast<size_t>(t) * a.k + lane];
                } else {
                    over = true;
                }
            }
        }
        const uint32_t m = __ballot_sync(kFullMask, ok);
        if (ok) {
            const int pos = __popc(m & lanemask_lt());
            s_src[warp][pos] = rowi;
            s_w[warp][pos] = wj;
        }
        if (__any_sync(kFullMask, over) && v == lane) raise_flag(a.status, EP_FLAG_CAPACITY);
        __syncwarp();
        const int ns = __popc(m);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int d0 = 0; d0 < ns; d0 += kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (d0 + i < ns && v < nvec) buf[i] = ld_stream_v4(ys + s_src[warp][d0 + i] + v);
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (d0 + i >= ns) continue;
                const uint32_t wd[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
                if (a.topk_w != nullptr) {
                    const float w = s_w[warp][d0 + i];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(bf16_lo(wd[q]), w));
                        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(bf16_hi(wd[q]), w));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fadd_rn(acc[2 * q], bf16_lo(wd[q]));
                        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16_hi(wd[q]));
                    }
                }
            }
        }
        if (v < nvec) {
            uint4 o;
            o.x = pack_bf16x2_rn(acc[0], acc[1]);
            o.y = pack_bf16x2_rn(acc[2], acc[3]);
            o.z = pack_bf16x2_rn(acc[4], acc[5]);
            o.w = pack_bf16x2_rn(acc[6], acc[7]);
            st_v4(os + static_cast<size_t>(t) * nvec + v, o);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Low-latency (decode-sized) dispatch + permute: one launch
// ---------------------------------------------------------------------------
// For a small batch (T <= kLLMaxTokens) every CTA computes the whole expert layout in
// shared memory -- the per-warp expert masks and in-warp ranks of expert_layout_kernel,
// chunk after chunk of 256 tokens with a running count per expert, then the offsets by a
// block scan -- so no CTA waits on another and no workspace is needed. CTA 0 writes the
// offsets and slots; CTA b then moves tokens b, b + gridDim.x, ...: warp 0 resolves the
// token's expert-major rows and writes the metadata, and the 8 warps copy an eighth of
// the row each to every destination. Same results as ep_get_expert_layout followed by
// ep_dispatch_permuted.
constexpr int kLLMaxTokens = 1024;
constexpr int kLLMaxEntries = 8192;  // T * k

struct LLArgs {
    const uint16_t* x;
    const int64_t* topk_idx;
    const float* topk_w;
    int T, H, k, E, R, max_rows;
    int32_t* offsets;  // [E+1] out
    int32_t* eslot;    // [T][k] out
    uint16_t* perm_x;
    int32_t* perm_src;
    float* perm_w;
    int32_t* status;
};

inline size_t ll_smem_bytes(int T, int k, int E) {
    return (static_cast<size_t>(2 * kWarps) * E + ((E + 1 + 3) & ~3) + static_cast<size_t>(T) * k) * sizeof(int32_t);
}

__global__ void __launch_bounds__(kThreads, 1) dispatch_permuted_ll_kernel(LLArgs a) {
    // a decode batch's grid leaves most of every SM free: the next kernel (the expert work,
    // or the low-latency combine launched as a dependent launch) may settle its CTAs now and
    // wait on the device for this grid, so its launch latency is hidden behind this one
    allow_dependents();
    grid_dependency_wait();  // dependent launch: inputs are ready after this
    extern __shared__ uint32_t smem[];
    uint32_t* s_emask = smem;                                              // [kWarps][E]
    int32_t* s_wpref = reinterpret_cast<int32_t*>(smem + kWarps * a.E);  // [kWarps][E]
    int32_t* s_cnt = s_wpref + kWarps * a.E;                             // [E+1]: counts, then offsets
    int32_t* s_slot = s_cnt + ((a.E + 1 + 3) & ~3);                      // [T][k]: expert, then slot
    __shared__ int32_t s_part[kWarps];
    __shared__ long long s_row[kMaxTopk];
    __shared__ int s_nd;
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int k = a.k;
    const int E = a.E;
    const int nvec = a.H / 8;
    const int per_warp = (nvec + kWarps - 1) / kWarps;  // 16-byte vectors of a row per warp
    const int v_lo = warp * per_warp;
    const int v_hi = v_lo + per_warp < nvec ? v_lo + per_warp : nvec;

    // the first token's row (this warp's slice) is requested before the layout work, so
    // that its memory latency overlaps it
    uint4 first[kUnroll];
    if (static_cast<int>(blockIdx.x) < a.T) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(blockIdx.x) * a.H);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v_lo + u * 32 + lane;
            if (v < v_hi) first[u] = ld_stream_v4(src + v);
        }
    }

    // 1. the expert layout of the whole batch, in shared memory
    for (int e = tid; e < E; e += kThreads) s_cnt[e] = 0;
    bool bad = false;
    for (int c0 = 0; c0 < a.T; c0 += kThreads) {
        const int t = c0 + tid;
        for (int e = lane; e < E; e += 32) s_emask[warp * E + e] = 0u;
        __syncthreads();
        if (t < a.T) {
            const long long* row = reinterpret_cast<const long long*>(a.topk_idx) + static_cast<size_t>(t) * k;
            for (int j0 = 0; j0 < k; j0 += kBatch) {
                long long ev[kBatch];  // eight ids in flight
#pragma unroll
                for (int i = 0; i < kBatch; ++i) ev[i] = j0 + i < k ? __ldg(row + j0 + i) : -1ll;
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int j = j0 + i;
                    if (j >= k) break;
                    const long long e = ev[i];
                    int x = -1;
                    if (e >= 0) {
                        if (e >= E) {
                            bad = true;
                        } else {
                            bool rep = false;  // a repeat of an earlier slot of the row counts once
#pragma unroll
                            for (int ii = 0; ii < i; ++ii) rep |= ev[ii] == e;
                            for (int jj = 0; jj < j0; ++jj) rep |= s_slot[t * k + jj] == static_cast<int>(e);
                            if (rep) bad = true;
                            else x = static_cast<int>(e);
                        }
                    }
                    s_slot[t * k + j] = x;
                    if (x >= 0) atomicOr(&s_emask[warp * E + x], 1u << lane);
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kThreads) {
            int run = s_cnt[e];
            for (int w = 0; w < kWarps; ++w) {
                s_wpref[w * E + e] = run;
                run += __popc(s_emask[w * E + e]);
            }
            s_cnt[e] = run;
        }
        __syncthreads();
        if (t < a.T) {
            const uint32_t below = (1u << lane) - 1u;
            for (int j = 0; j < k; ++j) {
                const int x = s_slot[t * k + j];
                s_slot[t * k + j] = x >= 0 ? s_wpref[warp * E + x] + __popc(s_emask[warp * E + x] & below) : -1;
            }
        }
        __syncthreads();
    }
    // exclusive scan of the counts into the offsets (per-thread runs, then warp and block)
    {
        const int per = (E + kThreads - 1) / kThreads;
        const int e0 = tid * per;
        int sum = 0;
        for (int i = 0; i < per; ++i)
            if (e0 + i < E) sum += s_cnt[e0 + i];
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) s_part[warp] = incl;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += s_part[w];
        int run = base + incl - sum;
        for (int i = 0; i < per; ++i) {
            if (e0 + i < E) {
                const int c = s_cnt[e0 + i];
                s_cnt[e0 + i] = run;
                run += c;
            }
        }
        if (tid == kThreads - 1) s_cnt[E] = base + incl;
        __syncthreads();
    }
    if (blockIdx.x == 0) {
        for (int e = tid; e <= E; e += kThreads) a.offsets[e] = s_cnt[e];
        for (int i = tid; i < a.T * k; i += kThreads) a.eslot[i] = s_slot[i];
        if (bad) raise_flag(a.status, EP_FLAG_BAD_EXPERT);
    }

    // 2. the rows
    const int epr = E / a.R;
    for (int t = static_cast<int>(blockIdx.x); t < a.T; t += static_cast<int>(gridDim.x)) {
        if (warp == 0) {
            bool ok = false, over = false;
            long long rowi = 0;
            if (lane < k) {
                const int sl = s_slot[t * k + lane];
                if (sl >= 0) {
                    const int e = static_cast<int>(a.topk_idx[static_cast<size_t>(t) * k + lane]);
                    const int r = e / epr;
                    const int p = s_cnt[e] - s_cnt[r * epr] + sl;
                    if (p < a.max_rows) {
                        ok = true;
                        rowi = static_cast<long long>(r) * a.max_rows + p;
                    } else {
                        over = true;
                    }
                }
            }
            const uint32_t m = __ballot_sync(kFullMask, ok);
            if (ok) {
                const int pos = __popc(m & lanemask_lt());
                s_row[pos] = rowi;
                if (a.perm_src != nullptr) a.perm_src[rowi] = t;
                if (a.perm_w != nullptr) a.perm_w[rowi] = a.topk_w[static_cast<size_t>(t) * k + lane];
            }
            if (__any_sync(kFullMask, over) && lane == 0) raise_flag(a.status, EP_FLAG_CAPACITY);
            if (lane == 0) s_nd = __popc(m);
        }
        __syncthreads();
        const int nd = s_nd;
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H);
        uint4* base = reinterpret_cast<uint4*>(a.perm_x);
        for (int v0 = v_lo; v0 < v_hi; v0 += 32 * kUnroll) {
            uint4 buf[kUnroll];
            const bool prefetched = t == static_cast<int>(blockIdx.x) && v0 == v_lo;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < v_hi) buf[u] = prefetched ? first[u] : ld_stream_v4(src + v);
            }
            for (int d = 0; d < nd; ++d) {
                uint4* dst = base + static_cast<size_t>(s_row[d]) * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < v_hi) st_v4(dst + v, buf[u]);
                }
            }
        }
        __syncthreads();  // s_row / s_nd are rewritten for the next token
    }
}

// ---------------------------------------------------------------------------
// Send phase of a split (hook-mode) combine
// ---------------------------------------------------------------------------

struct CombineSendArgs {
    const uint16_t* y_perm;  // [R][max_rows][H]
    const int32_t* recv_src;
    const int32_t* recv_tidx;
    const float* recv_tw;  // nullable: unweighted
    const int32_t* tokens_per_rank;
    const int32_t* offsets;
    const int32_t* eslot;
    int T, H, k, E, R, max_tokens, max_rows;
    uint16_t* y_rank;  // [R][max_tokens][H]
    int32_t* status;
    float neg_zero;  // -0, passed at run time (see ep::pair_add_product)
};

constexpr int kSendStages = 4;   // units in a warp's shared-memory ring: three in flight, one computed
constexpr int kSendChunk = 128;  // 16-byte vectors of a row per unit: 4 per lane
constexpr int kSendGroups = 2;  // 32-vector groups of a row send_row handles at once
constexpr int kSendBatch = 2;   // sources loaded together
constexpr int kSendRows = 32;   // rows a warp resolves at once (a lane per row)
constexpr int kSendMaxSrc = 8;  // sources per row kept from that resolution

// Copies one rank-level row from its ns compacted sources (expert-major row offsets in
// units of 16-byte vectors, weights), strictly in slot order: acc = 0, then per term one
// fp32 multiply by the weight (when weighted) and one fp32 add, never fused; one rounding
// to bf16 at the end.
__device__ __forceinline__ void send_row(const CombineSendArgs& a, const uint4* ys, uint4* dst, int nvec, int ns,
                                         const int* srcs, const float* ws) {
    const int lane = lane_id();
    for (int v0 = lane; v0 < nvec; v0 += 32 * kSendGroups) {
        float acc[kSendGroups][8];
#pragma unroll
        for (int g = 0; g < kSendGroups; ++g)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] = 0.0f;
        for (int d0 = 0; d0 < ns; d0 += kSendBatch) {
            uint4 buf[kSendBatch][kSendGroups];
#pragma unroll
            for (int b = 0; b < kSendBatch; ++b)
#pragma unroll
                for (int g = 0; g < kSendGroups; ++g)
                    if (d0 + b < ns && v0 + 32 * g < nvec) buf[b][g] = ld_stream_v4(ys + static_cast<size_t>(srcs[d0 + b]) * nvec + v0 + 32 * g);
#pragma unroll
            for (int b = 0; b < kSendBatch; ++b) {
                if (d0 + b >= ns) continue;
                const float w = ws[d0 + b];
#pragma unroll
                for (int g = 0; g < kSendGroups; ++g) {
                    const uint32_t wd[4] = {buf[b][g].x, buf[b][g].y, buf[b][g].z, buf[b][g].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (a.recv_tw != nullptr) {
                            acc[g][2 * h] = __fadd_rn(acc[g][2 * h], __fmul_rn(bf16_lo(wd[h]), w));
                            acc[g][2 * h + 1] = __fadd_rn(acc[g][2 * h + 1], __fmul_rn(bf16_hi(wd[h]), w));
                        } else {
                            acc[g][2 * h] = __fadd_rn(acc[g][2 * h], bf16_lo(wd[h]));
                            acc[g][2 * h + 1] = __fadd_rn(acc[g][2 * h + 1], bf16_hi(wd[h]));
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < kSendGroups; ++g) {
            if (v0 + 32 * g < nvec) {
                uint4 o;
                o.x = pack_bf16x2_rn(acc[g][0], acc[g][1]);
                o.y = pack_bf16x2_rn(acc[g][2], acc[g][3]);
                o.z = pack_bf16x2_rn(acc[g][4], acc[g][5]);
                o.w = pack_bf16x2_rn(acc[g][6], acc[g][7]);
                st_v4(dst + v0 + 32 * g, o);
            }
        }
    }
}

// Warp w of the W warps takes the received rows w, w + W, w + 2W, ... (rows strided over the
// batch, so every SM works on all ranks' rows alike), kSendRows rows at a time. Phase 1, a
// lane per row: the row (r, s) is
// found from the prefix of the per-rank counts in shared memory (binary search), and its
// local experts are resolved to expert-major rows -- received id, expert slot, offsets --
// so the dependent metadata loads of 32 rows overlap instead of running row after row.
// Up to kSendMaxSrc sources per row are kept in shared memory, in slot order; a row with
// more local experts is resolved again by the whole warp (lanes across slots) when its turn
// comes and copied by send_row. Phase 2 streams the other rows of the batch through the
// warp's shared-memory ring (stream_rows), so the loads of the next three units are in
// flight while one is computed and occupy no registers.
// kWeighted: a.recv_tw != nullptr (terms multiplied by their weights)
template <bool kWeighted>
__global__ void __launch_bounds__(kThreads, 2) combine_send_kernel(CombineSendArgs a) {
    grid_dependency_wait();  // dependent launch: the expert outputs are complete after this
    // per batch row: its sources as expert-major row indices r * max_rows + p (below 2^31)
    // with their weights, their number, the rank row r * max_tokens + s (below 2^31), token
    __shared__ int s_bsrc[kWarps][kSendRows][kSendMaxSrc];
    __shared__ float s_bw[kWarps][kSendRows][kSendMaxSrc];
    __shared__ int s_bns[kWarps][kSendRows];
    __shared__ int s_brow[kWarps][kSendRows];
    __shared__ int s_bt[kWarps][kSendRows];
    __shared__ int s_src[kWarps][kMaxTopk];
    __shared__ float s_w[kWarps][kMaxTopk];
    __shared__ int s_base[257];
    extern __shared__ __align__(16) uint4 s_ring[];  // [kWarps][kSendStages][kSendChunk]
    const int lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = a.H / 8;
    const int epr = a.E / a.R;
    if (warp == 0) {  // exclusive prefix of the received counts, 32 ranks per step
        int carry = 0;
        for (int r0 = 0; r0 < a.R; r0 += 32) {
            const int r = r0 + lane;
            int c = 0;
            if (r < a.R) {
                c = a.tokens_per_rank[r];
                c = c < 0 ? 0 : (c < a.max_tokens ? c : a.max_tokens);
            }
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            if (r < a.R) s_base[r] = carry + incl - c;
            carry += __shfl_sync(kFullMask, incl, 31);
        }
        if (lane == 0) s_base[a.R] = carry;
    }
    __syncthreads();
    const int total = s_base[a.R];
    const uint4* ys = reinterpret_cast<const uint4*>(a.y_perm);
    uint4* outs = reinterpret_cast<uint4*>(a.y_rank);
    // phase 2's stream: units (row i of the batch, chunk c of kSendChunk vectors, source j)
    // in order -- all sources of a chunk, then the next chunk, then the next row; a row
    // without sources has one unit per chunk (zeros). The issuing side runs kSendStages - 1
    // units ahead: each lane copies its 4 vectors of the unit into its own slots of the
    // warp's ring (so no barrier between lanes is needed), and the arithmetic side reads
    // them back. Per chunk: acc = +0, then acc += RN(x * w) (or x) in slot order, one
    // rounding to bf16 at the end.
    uint4* ring = s_ring + warp * (kSendStages * kSendChunk);
    const int nchunks = (nvec + kSendChunk - 1) / kSendChunk;
    auto stream_rows = [&](int i0, int i1) {
        // issuing side: unit (pi, pc, pj) of row pi with pns sources, the source's offset psrc
        int pi = i0, pc = 0, pj = 0;
        int pns = s_bns[warp][i0];
        size_t psrc = pns > 0 ? static_cast<size_t>(s_bsrc[warp][i0][0]) * nvec : 0;
        // arithmetic side: unit (ci, cc, cj) of row ci with cns sources, the source's weight cw
        // and the row's output offset cout; the next unit's values are loaded a call ahead
        int ci = i0, cc = 0, cj = 0;
        int cns = pns;
        float cw = pns > 0 ? s_bw[warp][i0][0] : 1.0f;
        size_t cout = static_cast<size_t>(s_brow[warp][i0]) * nvec;
        float acc[32];
        auto produce = [&](int st) {
            if (pi < i1) {
                const int vb = pc * kSendChunk + lane;
                if (pns > 0) {
                    const uint4* src = ys + psrc + vb;
                    uint4* dst = ring + st * kSendChunk + lane;
                    if ((pc + 1) * kSendChunk <= nvec) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) cp_async16(dst + g * 32, src + g * 32);
                    } else {
#pragma unroll
                        for (int g = 0; g < 4; ++g) cp_async16_if(dst + g * 32, src + g * 32, vb + g * 32 < nvec);
                    }
                }
                if (++pj < pns) {
                    psrc = static_cast<size_t>(s_bsrc[warp][pi][pj]) * nvec;
                } else {
                    pj = 0;
                    bool row_changed = false;
                    if (++pc == nchunks) {
                        pc = 0;
                        row_changed = ++pi < i1;
                        if (row_changed) pns = s_bns[warp][pi];
                    }
                    if ((row_changed || pns > 1) && pi < i1 && pns > 0)
                        psrc = static_cast<size_t>(s_bsrc[warp][pi][0]) * nvec;
                }
            }
            cp_async_commit();  // an empty group past the end keeps the waits uniform
        };
        auto consume = [&](int st) {
            const int vb = cc * kSendChunk + lane;
            const bool full = (cc + 1) * kSendChunk <= nvec;  // all 4 of every lane's vectors in range
            if (cj == 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
            }
            auto add_vec = [&](int g, const uint4& x) {
                const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float& a0 = acc[g * 8 + 2 * h];
                    float& a1 = acc[g * 8 + 2 * h + 1];
                    if (kWeighted) pair_add_product(a0, a1, bf16_lo(wd[h]), bf16_hi(wd[h]), cw, a.neg_zero);
                    else pair_add(a0, a1, bf16_lo(wd[h]), bf16_hi(wd[h]));
                }
            };
            if (cns > 0) {
                const uint4* slot = ring + st * kSendChunk + lane;
                if (full) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) add_vec(g, slot[g * 32]);
                } else {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (vb + g * 32 < nvec) add_vec(g, slot[g * 32]);
                }
            }
            if (cj + 1 < cns) {
                ++cj;
                cw = s_bw[warp][ci][cj];
                return;
            }
            // the chunk's last source: its bf16 vectors
            uint4* dst = outs + cout + vb;
            auto put = [&](int g) {
                uint4 o;
                o.x = pack_bf16x2_rn(acc[g * 8 + 0], acc[g * 8 + 1]);
                o.y = pack_bf16x2_rn(acc[g * 8 + 2], acc[g * 8 + 3]);
                o.z = pack_bf16x2_rn(acc[g * 8 + 4], acc[g * 8 + 5]);
                o.w = pack_bf16x2_rn(acc[g * 8 + 6], acc[g * 8 + 7]);
                st_v4(dst + g * 32, o);
            };
            if (full) {
#pragma unroll
                for (int g = 0; g < 4; ++g) put(g);
            } else {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    if (vb + g * 32 < nvec) put(g);
            }
            cj = 0;
            if (++cc == nchunks) {
                cc = 0;
                if (++ci < i1) {
                    cns = s_bns[warp][ci];
                    cout = static_cast<size_t>(s_brow[warp][ci]) * nvec;
                }
            }
            if (ci < i1 && cns > 0) cw = s_bw[warp][ci][0];
        };
#pragma unroll
        for (int u = 0; u < kSendStages - 1; ++u) produce(u);
        int st = 0;
        while (ci < i1) {
            produce(st == 0 ? kSendStages - 1 : st - 1);  // the stage consumed last step
            cp_async_wait<kSendStages - 1>();
            consume(st);
            st = st + 1 == kSendStages ? 0 : st + 1;
        }
        cp_async_wait<0>();  // only empty groups can be left: nothing in flight on return
    };

    // warp gw of W takes the rows gw, gw + W, gw + 2W, ... (every SM then works on all
    // ranks' rows alike), resolved up to kSendRows at a time: batch rows q0 + i * W
    const int nwarps = static_cast<int>(gridDim.x) * kWarps;
    const int gw = static_cast<int>(blockIdx.x) * kWarps + warp;
    for (long long q0 = gw; q0 < total; q0 += static_cast<long long>(kSendRows) * nwarps) {
        const long long left = (total - q0 + nwarps - 1) / nwarps;
        const int nb = left < kSendRows ? static_cast<int>(left) : kSendRows;
        // phase 1: lane i resolves row q0 + i * W
        const int q = static_cast<int>(q0 + static_cast<long long>(lane) * nwarps);
        int n = 0, t = -1;
        bool over = false;
        long long orow = 0;
        if (lane < nb) {
            int lo = 0, hi = a.R;  // last r with s_base[r] <= q
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_base[mid] <= q) lo = mid;
                else hi = mid;
            }
            const int r = lo;
            orow = static_cast<long long>(r) * a.max_tokens + (q - s_base[r]);
            t = a.recv_src[orow];
            if (t >= 0 && t < a.T) {
                const int base = a.offsets[r * epr];
                for (int j0 = 0; j0 < a.k; j0 += 8) {
                    int lv[8], sv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        lv[i] = j0 + i < a.k ? a.recv_tidx[orow * a.k + j0 + i] : -1;
                        sv[i] = j0 + i < a.k ? a.eslot[static_cast<size_t>(t) * a.k + j0 + i] : -1;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (lv[i] < 0 || lv[i] >= epr || sv[i] < 0) continue;
                        const int p = a.offsets[r * epr + lv[i]] - base + sv[i];
                        if (p < 0 || p >= a.max_rows) {
                            over = true;
                            continue;
                        }
                        if (n < kSendMaxSrc) {
                            s_bsrc[warp][lane][n] = r * a.max_rows + p;
                            s_bw[warp][lane][n] = a.recv_tw != nullptr ? a.recv_tw[orow * a.k + j0 + i] : 1.0f;
                        }
                        ++n;
                    }
                }
            }
        }
        s_bns[warp][lane] = n;
        s_brow[warp][lane] = static_cast<int>(orow);
        s_bt[warp][lane] = t;
        if (__any_sync(kFullMask, over) && lane == 0) raise_flag(a.status, EP_FLAG_CAPACITY);
        __syncwarp();
        // phase 2: runs of rows with at most kSendMaxSrc sources stream through the ring; a
        // row with more is resolved again by the whole warp and copied on its own
        for (int i = 0; i < nb;) {
            int j = i;
            while (j < nb && s_bns[warp][j] <= kSendMaxSrc) ++j;
            if (j > i) stream_rows(i, j);
            if (j == nb) break;
            const long long row = s_brow[warp][j];  // the rank row r * max_tokens + s
            // more local experts than phase 1 kept: lanes across slots, compacted by a ballot
            const int r = static_cast<int>(row / a.max_tokens);
            const int tt = s_bt[warp][j];
            bool ok = false;
            int src = 0;
            float wj = 1.0f;
            if (lane < a.k) {
                const int l = a.recv_tidx[row * a.k + lane];
                const int32_t sl = a.eslot[static_cast<size_t>(tt) * a.k + lane];
                if (l >= 0 && l < epr && sl >= 0) {
                    const int p = a.offsets[r * epr + l] - a.offsets[r * epr] + sl;
                    if (p >= 0 && p < a.max_rows) {
                        ok = true;
                        src = r * a.max_rows + p;
                        if (a.recv_tw != nullptr) wj = a.recv_tw[row * a.k + lane];
                    }
                }
            }
            const uint32_t m = __ballot_sync(kFullMask, ok);
            if (ok) {
                const int pos = __popc(m & lanemask_lt());
                s_src[warp][pos] = src;
                s_w[warp][pos] = wj;
            }
            __syncwarp();
            send_row(a, ys, outs + row * nvec, nvec, __popc(m), s_src[warp], s_w[warp]);
            __syncwarp();
            i = j + 1;
        }
        __syncwarp();  // the batch's lists are rewritten next
    }
    allow_dependents();
}

// ---------------------------------------------------------------------------
// Low-latency (decode-sized) combine from expert-major slabs
// ---------------------------------------------------------------------------
// The same result as combine_permuted_kernel, shaped for latency: CTA (t, part) handles
// one token and one slice of at most 256 vectors of its row, a vector per thread. At the
// start every thread helps to load the expert offsets into shared memory while warp 0
// loads the token's expert slots, ids and weights, so both reach the CTA in one memory
// round trip; the rows' positions then come from shared memory, and each thread issues
// the loads of all of the token's source vectors (kBatch at a time) in a second round
// trip before adding them in slot order.
constexpr int kLLCombineVec = kThreads;  // vectors of a row per CTA

__global__ void __launch_bounds__(kThreads) combine_permuted_ll_kernel(CombinePermArgs a, int parts) {
    grid_dependency_wait();  // dependent launch: the expert outputs are complete after this
    __shared__ int32_t s_off[kMaxExpertsPerm + 1];
    __shared__ long long s_src[kMaxTopk];
    __shared__ float s_w[kMaxTopk];
    __shared__ int s_ns;
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int nvec = a.H / 8;
    const int epr = a.E / a.R;
    const uint4* ys = reinterpret_cast<const uint4*>(a.y);
    uint4* os = reinterpret_cast<uint4*>(a.out);
    for (int b = static_cast<int>(blockIdx.x); b < a.T * parts; b += static_cast<int>(gridDim.x)) {
        const int t = b / parts;
        const int v = (b - t * parts) * kLLCombineVec + tid;
        int32_t sl = -1;
        int64_t e = -1;
        float wj = 1.0f;
        if (tid < a.k) {
            sl = a.eslot[static_cast<size_t>(t) * a.k + tid];
            e = a.topk_idx[static_cast<size_t>(t) * a.k + tid];
            if (a.topk_w != nullptr) wj = a.topk_w[static_cast<size_t>(t) * a.k + tid];
        }
        for (int i = tid; i <= a.E; i += kThreads) s_off[i] = a.offsets[i];
        __syncthreads();
        if (tid < 32) {
            bool ok = false, over = false;
            long long src = 0;
            if (lane < a.k && sl >= 0 && e >= 0 && e < a.E) {
                const int r = static_cast<int>(e) / epr;
                const int p = s_off[e] - s_off[r * epr] + sl;
                if (p >= 0 && p < a.max_rows) {
                    ok = true;
                    src = (static_cast<long long>(r) * a.max_rows + p) * nvec;
                } else {
                    over = true;
                }
            }
            const uint32_t m = __ballot_sync(kFullMask, ok);
            if (ok) {
                const int pos = __popc(m & lanemask_lt());
                s_src[pos] = src;
                s_w[pos] = wj;
            }
            if (__any_sync(kFullMask, over) && lane == 0 && b % parts == 0) raise_flag(a.status, EP_FLAG_CAPACITY);
            if (lane == 0) s_ns = __popc(m);
        }
        __syncthreads();
        const int ns = s_ns;
        if (v < nvec) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int d0 = 0; d0 < ns; d0 += kBatch) {
                uint4 buf[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
                    if (d0 + i < ns) buf[i] = ld_stream_v4(ys + s_src[d0 + i] + v);
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    if (d0 + i >= ns) continue;
                    const uint32_t wd[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
                    const float w = s_w[d0 + i];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (a.topk_w != nullptr) {
                            acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(bf16_lo(wd[q]), w));
                            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(bf16_hi(wd[q]), w));
                        } else {
                            acc[2 * q] = __fadd_rn(acc[2 * q], bf16_lo(wd[q]));
                            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16_hi(wd[q]));
                        }
                    }
                }
            }
            uint4 o;
            o.x = pack_bf16x2_rn(acc[0], acc[1]);
            o.y = pack_bf16x2_rn(acc[2], acc[3]);
            o.z = pack_bf16x2_rn(acc[4], acc[5]);
            o.w = pack_bf16x2_rn(acc[6], acc[7]);
            st_v4(os + static_cast<size_t>(t) * nvec + v, o);
        }
        __syncthreads();  // s_off / s_src / s_ns are rewritten for the next token
    }
}

std::atomic<int> g_send_smem_set[kMaxDevices];
std::atomic<int> g_send_smem_set_w[kMaxDevices];
std::atomic<int> g_send_per_sm[kMaxDevices];
std::atomic<int> g_send_per_sm_w[kMaxDevices];

std::atomic<int> g_ll_attr_set[kMaxDevices];
std::atomic<int> g_attr_set[kMaxDevices];
std::atomic<int> g_combine_per_sm[kMaxDevices];

int token_grid(long long work) {
    const long long want = (work + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

extern "C" size_t ep_expert_layout_workspace_size(int32_t T, int32_t E) {
    if (T < 0 || E <= 0) return 0;
    return 256 + align256(static_cast<size_t>(num_tiles_for(T)) * E * sizeof(unsigned long long));
}

extern "C" ep_status_t ep_get_expert_layout(const int64_t* topk_idx, int32_t T, int32_t k, int32_t E,
                                            int32_t* expert_offsets, int32_t* expert_slot, void* workspace,
                                            size_t workspace_bytes, int32_t* status, void* stream) {
    if (T < 0 || T >= (1 << 30) || k < 1 || k > kMaxTopk || E < 1 || E > kMaxExpertsPerm) return EP_ERR_INVALID;
    if (expert_offsets == nullptr || workspace == nullptr) return EP_ERR_INVALID;
    if (T > 0 && (topk_idx == nullptr || expert_slot == nullptr)) return EP_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EP_ERR_INVALID;
    if (workspace_bytes < ep_expert_layout_workspace_size(T, E)) return EP_ERR_INVALID;
    if (!aligned16_or_null(topk_idx) || !aligned16(expert_offsets) || !aligned16_or_null(expert_slot))
        return EP_ERR_INVALID;
    ExpertLayoutArgs a{};
    a.topk_idx = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.num_tiles = num_tiles_for(T);
    a.offsets = expert_offsets;
    a.eslot = expert_slot;
    a.hdr = static_cast<ep_layout_ws_header_t*>(workspace);
    a.words = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + 256);
    a.status = status;
    const size_t smem = (static_cast<size_t>(E) * (2 * kWarps + 2) + static_cast<size_t>(k) * kThreads) * sizeof(int32_t);
    const ep_status_t attr = ensure_dynamic_smem(
        g_attr_set, expert_layout_kernel,
        (kMaxExpertsPerm * (2 * kWarps + 2) + kMaxTopk * kThreads) * static_cast<int>(sizeof(int32_t)));
    if (attr != EP_OK) return attr;
    expert_layout_kernel<<<a.num_tiles, kThreads, smem, as_stream(stream)>>>(a);
    return check_launch();
}

static bool perm_common_ok(int T, int H, int k, int E, int R, int max_rows) {
    return T >= 0 && H > 0 && H % 8 == 0 && k >= 1 && k <= kMaxTopk && R >= 1 && R <= 256 && E >= R && E % R == 0 &&
           E <= 8192 && max_rows >= 0 && static_cast<long long>(R) * max_rows <= 0x7fffffffLL;
}

extern "C" ep_status_t ep_dispatch_permuted(const void* x, const int64_t* topk_idx, const float* topk_w,
                                            const int32_t* expert_offsets, const int32_t* expert_slot, int32_t T,
                                            int32_t H, int32_t k, int32_t E, int32_t R, int32_t max_rows,
                                            void* perm_x, int32_t* perm_src, float* perm_w, int32_t* status,
                                            void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || perm_x == nullptr) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (x == nullptr || topk_idx == nullptr || expert_offsets == nullptr || expert_slot == nullptr ||
        (perm_w != nullptr && topk_w == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16(x) || !aligned16(perm_x) || !aligned16(topk_idx) || !aligned16_or_null(topk_w) ||
        !aligned16(expert_offsets) || !aligned16(expert_slot) || !aligned16_or_null(perm_src) ||
        !aligned16_or_null(perm_w))
        return EP_ERR_INVALID;
    PermDispatchArgs a{static_cast<const uint16_t*>(x), topk_idx, topk_w, expert_offsets, expert_slot, T, H, k, E, R,
                       max_rows, static_cast<uint16_t*>(perm_x), perm_src, perm_w, status};
    const PermScatter sp{a, static_cast<char*>(perm_x), static_cast<uint32_t>(H) * 2u, status};
    const ep_status_t st = launch_scatter_rows(sp, T, as_stream(stream));
    if (st != EP_ERR_INVALID) return st;  // rows too large for the shared-memory buffers: registers
    dispatch_permuted_kernel<<<token_grid(T), kThreads, 0, as_stream(stream)>>>(a);
    return check_launch();
}

extern "C" ep_status_t ep_permute_received(const void* recv_x, const int32_t* recv_src_idx,
                                           const int32_t* recv_topk_idx, const float* recv_topk_w,
                                           const int32_t* tokens_per_rank, const int32_t* expert_offsets,
                                           const int32_t* expert_slot, int32_t T, int32_t H, int32_t k, int32_t E,
                                           int32_t R, int32_t max_tokens, int32_t max_rows, void* perm_x,
                                           int32_t* perm_src, float* perm_w, int32_t* status, void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || max_tokens < 0 || perm_x == nullptr) return EP_ERR_INVALID;
    if (T == 0 || max_tokens == 0) return EP_OK;
    if (recv_x == nullptr || recv_src_idx == nullptr || recv_topk_idx == nullptr || tokens_per_rank == nullptr ||
        expert_offsets == nullptr || expert_slot == nullptr || (perm_w != nullptr && recv_topk_w == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16(recv_x) || !aligned16(perm_x) || !aligned16(recv_src_idx) || !aligned16(recv_topk_idx) ||
        !aligned16_or_null(recv_topk_w) || !aligned16(tokens_per_rank) || !aligned16(expert_offsets) ||
        !aligned16(expert_slot) || !aligned16_or_null(perm_src) || !aligned16_or_null(perm_w))
        return EP_ERR_INVALID;
    PermuteRecvArgs a{static_cast<const uint16_t*>(recv_x), recv_src_idx, recv_topk_idx, recv_topk_w, tokens_per_rank,
                      expert_offsets, expert_slot, T, H, k, E, R, max_tokens, max_rows,
                      static_cast<uint16_t*>(perm_x), perm_src, perm_w, status};
    // rows received never exceed T per rank nor max_tokens
    const long long bound = static_cast<long long>(R) * (T < max_tokens ? T : max_tokens);
    permute_received_kernel<<<token_grid(bound), kThreads, 0, as_stream(stream)>>>(a);
    return check_launch();
}

extern "C" ep_status_t ep_combine_permuted(const void* y, const int64_t* topk_idx, const float* topk_w,
                                           const int32_t* expert_offsets, const int32_t* expert_slot, int32_t T,
                                           int32_t H, int32_t k, int32_t E, int32_t R, int32_t max_rows, void* out,
                                           int32_t* status, void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || out == nullptr) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (topk_idx == nullptr || expert_offsets == nullptr || expert_slot == nullptr || (max_rows > 0 && y == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(y) || !aligned16(out) || !aligned16(topk_idx) || !aligned16_or_null(topk_w) ||
        !aligned16(expert_offsets) || !aligned16(expert_slot))
        return EP_ERR_INVALID;
    CombinePermArgs a{static_cast<const uint16_t*>(y), topk_idx, topk_w, expert_offsets, expert_slot, T, H, k, E, R,
                      max_rows, static_cast<uint16_t*>(out), status};
    int per_sm = 1;
    const ep_status_t occ = blocks_per_sm(g_combine_per_sm, combine_permuted_kernel, kThreads, 0, &per_sm);
    if (occ != EP_OK) return occ;
    const long long items = static_cast<long long>(T) * ((H / 8 + 31) / 32);
    const long long want = (items + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * per_sm;
    combine_permuted_kernel<<<static_cast<int>(want < cap ? want : cap), kThreads, 0, as_stream(stream)>>>(a);
    return check_launch();
}

extern "C" ep_status_t ep_dispatch_permuted_ll(const void* x, const int64_t* topk_idx, const float* topk_w,
                                               int32_t T, int32_t H, int32_t k, int32_t E, int32_t R,
                                               int32_t max_rows, int32_t* expert_offsets, int32_t* expert_slot,
                                               void* perm_x, int32_t* perm_src, float* perm_w, int32_t* status,
                                               void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || T > kLLMaxTokens || T * k > kLLMaxEntries ||
        E > kMaxExpertsPerm || expert_offsets == nullptr)
        return EP_ERR_INVALID;
    if (T > 0 && (x == nullptr || topk_idx == nullptr || expert_slot == nullptr || perm_x == nullptr ||
                  (perm_w != nullptr && topk_w == nullptr)))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(x) || !aligned16_or_null(perm_x) || !aligned16_or_null(topk_idx) ||
        !aligned16_or_null(topk_w) || !aligned16(expert_offsets) || !aligned16_or_null(expert_slot) ||
        !aligned16_or_null(perm_src) || !aligned16_or_null(perm_w))
        return EP_ERR_INVALID;
    const ep_status_t attr = ensure_dynamic_smem(
        g_ll_attr_set, dispatch_permuted_ll_kernel,
        static_cast<int>(ll_smem_bytes(kLLMaxTokens, kLLMaxEntries / kLLMaxTokens, kMaxExpertsPerm)));
    if (attr != EP_OK) return attr;
    LLArgs a{static_cast<const uint16_t*>(x), topk_idx, topk_w, T, H, k, E, R, max_rows, expert_offsets, expert_slot,
             static_cast<uint16_t*>(perm_x), perm_src, perm_w, status};
    const int sms = sm_count();
    const int grid = T < 1 ? 1 : (T < sms ? T : sms);
    return launch_dependent(dispatch_permuted_ll_kernel, dim3(grid), dim3(kThreads), ll_smem_bytes(T, k, E),
                            as_stream(stream), a);
}

extern "C" ep_status_t ep_combine_send(const void* y_perm, const int32_t* recv_src_idx, const int32_t* recv_topk_idx,
                                       const float* recv_topk_w, const int32_t* tokens_per_rank,
                                       const int32_t* expert_offsets, const int32_t* expert_slot, int32_t T, int32_t H,
                                       int32_t k, int32_t E, int32_t R, int32_t max_tokens, int32_t max_rows,
                                       void* y_rank, int32_t* status, void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || max_tokens < 0 ||
        static_cast<long long>(R) * max_tokens > 0x7fffffffLL || y_rank == nullptr)
        return EP_ERR_INVALID;
    if (T == 0 || max_tokens == 0) return EP_OK;
    if (recv_src_idx == nullptr || recv_topk_idx == nullptr || tokens_per_rank == nullptr ||
        expert_offsets == nullptr || expert_slot == nullptr || (max_rows > 0 && y_perm == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(y_perm) || !aligned16(y_rank) || !aligned16(recv_src_idx) || !aligned16(recv_topk_idx) ||
        !aligned16_or_null(recv_topk_w) || !aligned16(tokens_per_rank) || !aligned16(expert_offsets) ||
        !aligned16(expert_slot))
        return EP_ERR_INVALID;
    CombineSendArgs a{static_cast<const uint16_t*>(y_perm), recv_src_idx, recv_topk_idx, recv_topk_w, tokens_per_rank,
                      expert_offsets, expert_slot, T, H, k, E, R, max_tokens, max_rows,
                      static_cast<uint16_t*>(y_rank), status, -0.0f};
    constexpr int kRingBytes = kWarps * kSendStages * kSendChunk * 16;
    auto kernel = recv_topk_w != nullptr ? combine_send_kernel<true> : combine_send_kernel<false>;
    ep_status_t occ = ensure_dynamic_smem(recv_topk_w != nullptr ? g_send_smem_set_w : g_send_smem_set, kernel,
                                          kRingBytes);
    if (occ != EP_OK) return occ;
    int per_sm = 1;
    occ = blocks_per_sm(recv_topk_w != nullptr ? g_send_per_sm_w : g_send_per_sm, kernel, kThreads, kRingBytes,
                        &per_sm);
    if (occ != EP_OK) return occ;
    // rows received never exceed T per rank nor max_tokens
    const long long rows = static_cast<long long>(R) * (T < max_tokens ? T : max_tokens);
    const long long want = (rows + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
    return launch_dependent(kernel, dim3(grid), dim3(kThreads), kRingBytes, as_stream(stream), a);
}

extern "C" ep_status_t ep_combine_permuted_ll(const void* y, const int64_t* topk_idx, const float* topk_w,
                                              const int32_t* expert_offsets, const int32_t* expert_slot, int32_t T,
                                              int32_t H, int32_t k, int32_t E, int32_t R, int32_t max_rows,
                                              void* out, int32_t* status, void* stream) {
    if (!perm_common_ok(T, H, k, E, R, max_rows) || T > kLLMaxTokens || E > kMaxExpertsPerm || out == nullptr)
        return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (topk_idx == nullptr || expert_offsets == nullptr || expert_slot == nullptr || (max_rows > 0 && y == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(y) || !aligned16(out) || !aligned16(topk_idx) || !aligned16_or_null(topk_w) ||
        !aligned16(expert_offsets) || !aligned16(expert_slot))
        return EP_ERR_INVALID;
    CombinePermArgs a{static_cast<const uint16_t*>(y), topk_idx, topk_w, expert_offsets, expert_slot, T, H, k, E, R,
                      max_rows, static_cast<uint16_t*>(out), status};
    const int nvec = H / 8;
    const int parts = (nvec + kLLCombineVec - 1) / kLLCombineVec;
    const long long ctas = static_cast<long long>(T) * parts;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    const int grid = static_cast<int>(ctas < cap ? ctas : cap);
    return launch_dependent(combine_permuted_ll_kernel, dim3(grid), dim3(kThreads), 0, as_stream(stream), a, parts);
}
