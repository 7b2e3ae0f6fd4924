// ep_nodes.cu -- node-level dense / sparse dispatch with a token-indexed receive
// layout ("[PR #634] Hybrid ep nixl restripe", section "Fix": one copy of the
// hidden rows and one of the staged prob slices per (chunk, destination) on the
// dense path, one per run of consecutive routed tokens on the sparse path;
// NUM_OF_TOKENS_PER_CHUNK = 256 in "Baseline problem"; the receive side keeps
// token-major strides, "Receive-side and DOCA path are unchanged").
//
// On one GPU a "copy per chunk" and a "copy per run" both land rows at the same
// token-indexed positions, so both paths run as one warp-per-token scatter that
// reads each hidden row once and writes it to every destination node (all
// nodes when dense, the routed ones when sparse), plus the token's staged prob
// slice for that node. The run count per (node, chunk) -- the number of copies
// the chunked formulation makes -- is computed by the first warps of the grid
// with ballots over 32 tokens at a time (a run starts where a bit is set and
// the bit before it, carried across groups, is clear).
#include "ep_common.cuh"
#include "ep_scatter.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;  // 16-byte vectors in flight per lane
constexpr int kMaxNodes = 256;

struct NodeArgs {
    const uint16_t* x;
    const float* staging;
    const uint8_t* in_node;
    int T, H, N, P, max_tokens, chunk, nchunks;
    bool dense;
    uint16_t* recv_x;
    float* recv_prob;
    int32_t* num_runs;
};

__global__ void __launch_bounds__(kThreads) node_dispatch_kernel(NodeArgs a) {
    __shared__ int s_node[kWarps][kMaxNodes];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int gw = blockIdx.x * kWarps + warp;
    const int nw = gridDim.x * kWarps;

    // run counts, one warp per (node, chunk)
    if (a.num_runs != nullptr) {
        for (int q = gw; q < a.N * a.nchunks; q += nw) {
            const int n = q / a.nchunks;
            const int c = q - n * a.nchunks;
            const int t0 = c * a.chunk;
            const int t1 = t0 + a.chunk < a.T ? t0 + a.chunk : a.T;
            int runs = 0;
            if (a.dense) {
                runs = t1 > t0 ? 1 : 0;
            } else {
                uint32_t carry = 0;  // bit of the token just before this group
                for (int g = t0; g < t1; g += 32) {
                    const int t = g + lane;
                    const bool in = t < t1 && a.in_node[static_cast<size_t>(t) * a.N + n] != 0;
                    const uint32_t m = __ballot_sync(ep::kFullMask, in);
                    runs += __popc(m & ~((m << 1) | carry));
                    carry = m >> 31;
                }
            }
            if (lane == 0) a.num_runs[q] = runs;
        }
    }

    const int nvec = a.H / 8;
    const int pvec = a.P / 4;
    const uint4* xs = reinterpret_cast<const uint4*>(a.x);
    uint4* rx = reinterpret_cast<uint4*>(a.recv_x);
    for (int t = gw; t < a.T; t += nw) {
        // destination nodes of token t (ascending)
        int nd = 0;
        for (int n0 = 0; n0 < a.N; n0 += 32) {
            const int n = n0 + lane;
            const bool go = n < a.N && (a.dense || a.in_node[static_cast<size_t>(t) * a.N + n] != 0);
            const uint32_t m = __ballot_sync(ep::kFullMask, go);
            if (go) s_node[warp][nd + __popc(m & ep::lanemask_lt())] = n;
            nd += __popc(m);
        }
        __syncwarp();
        const uint4* src = xs + static_cast<size_t>(t) * nvec;
        for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
            uint4 buf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) buf[u] = ep::ld_stream_v4(src + v);
            }
            for (int d = 0; d < nd; ++d) {
                uint4* dst = rx + (static_cast<size_t>(s_node[warp][d]) * a.max_tokens + t) * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < nvec) ep::st_v4(dst + v, buf[u]);
                }
            }
        }
        if (a.recv_prob != nullptr) {
            for (int d = 0; d < nd; ++d) {
                const size_t row = static_cast<size_t>(s_node[warp][d]) * a.max_tokens + t;
                const uint4* ps = reinterpret_cast<const uint4*>(a.staging + row * a.P);
                uint4* pd = reinterpret_cast<uint4*>(a.recv_prob + row * a.P);
                for (int v = lane; v < pvec; v += 32) ep::st_v4(pd + v, ep::ld_stream_v4(ps + v));
            }
        }
        __syncwarp();
    }
}

// Run count of (node n, chunk c) for q = n * nchunks + c, one warp: ballots over 32
// tokens at a time; a run starts where a bit is set and the bit before it (carried
// across groups) is clear.
__device__ __forceinline__ void count_runs(const NodeArgs& a, int q) {
    const int lane = ep::lane_id();
    const int n = q / a.nchunks;
    const int c = q - n * a.nchunks;
    const int t0 = c * a.chunk;
    const int t1 = t0 + a.chunk < a.T ? t0 + a.chunk : a.T;
    int runs = 0;
    if (a.dense) {
        runs = t1 > t0 ? 1 : 0;
    } else {
        uint32_t carry = 0;
        for (int g = t0; g < t1; g += 32) {
            const int t = g + lane;
            const bool in = t < t1 && a.in_node[static_cast<size_t>(t) * a.N + n] != 0;
            const uint32_t m = __ballot_sync(ep::kFullMask, in);
            runs += __popc(m & ~((m << 1) | carry));
            carry = m >> 31;
        }
    }
    if (lane == 0) a.num_runs[q] = runs;
}

// Node dispatch through the shared bulk-copy scatter (ep_scatter.cuh): token t goes to
// row t of every destination node; the side work copies the token's staged prob slice
// to each destination, and the prologue counts the runs.
struct NodeScatter {
    NodeArgs a;
    char* dst;
    uint32_t row_bytes;
    int32_t* status;
    __device__ int items() const { return a.T; }
    __device__ const void* source(int t) const { return a.x + static_cast<size_t>(t) * a.H; }
    __device__ int destinations(int t, long long* rows, int* aux) const {
        const int lane = ep::lane_id();
        int nd = 0;
        for (int n0 = 0; n0 < a.N; n0 += 32) {
            const int n = n0 + lane;
            const bool go = n < a.N && (a.dense || a.in_node[static_cast<size_t>(t) * a.N + n] != 0);
            const uint32_t m = __ballot_sync(ep::kFullMask, go);
            if (go) {
                const int pos = nd + __popc(m & ep::lanemask_lt());
                rows[pos] = static_cast<long long>(n) * a.max_tokens + t;
                aux[pos] = n;
            }
            nd += __popc(m);
        }
        __syncwarp();
        return nd;
    }
    __device__ void side_work(int t, int nd, const long long* rows, const int* aux) const {
        if (a.recv_prob == nullptr) return;
        const int lane = ep::lane_id();
        const int pvec = a.P / 4;
        for (int d = 0; d < nd; ++d) {
            const size_t row = static_cast<size_t>(rows[d]);
            const uint4* ps = reinterpret_cast<const uint4*>(a.staging + row * a.P);
            uint4* pd = reinterpret_cast<uint4*>(a.recv_prob + row * a.P);
            for (int v = lane; v < pvec; v += 32) ep::st_v4(pd + v, ep::ld_stream_v4(ps + v));
        }
        (void)t;
        (void)aux;
    }
    __device__ void prologue() const {
        if (a.num_runs == nullptr) return;
        for (int q = static_cast<int>(blockIdx.x); q < a.N * a.nchunks; q += static_cast<int>(gridDim.x)) count_runs(a, q);
    }
};

}  // namespace

extern "C" ep_status_t ep_dispatch_nodes(const void* x, const float* prob_staging, const uint8_t* is_token_in_node,
                                         int32_t T, int32_t H, int32_t num_nodes, int32_t P, int32_t max_tokens,
                                         int32_t chunk_tokens, ep_node_mode_t mode, void* recv_x_node,
                                         float* recv_prob_node, int32_t* num_runs, void* stream) {
    using namespace ep;
    const bool dense = mode == EP_NODES_DENSE;
    if (!dense && mode != EP_NODES_SPARSE) return EP_ERR_INVALID;
    if (T < 0 || H <= 0 || H % 8 != 0 || num_nodes < 1 || num_nodes > kMaxNodes || max_tokens < T ||
        chunk_tokens < 1)
        return EP_ERR_INVALID;
    const bool with_prob = prob_staging != nullptr || recv_prob_node != nullptr;
    if (with_prob && (prob_staging == nullptr || recv_prob_node == nullptr || P < 4 || P % 4 != 0))
        return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (x == nullptr || recv_x_node == nullptr || (!dense && is_token_in_node == nullptr)) return EP_ERR_INVALID;
    if (!aligned16(x) || !aligned16(recv_x_node) || !aligned16_or_null(prob_staging) ||
        !aligned16_or_null(recv_prob_node) || !aligned16_or_null(is_token_in_node) || !aligned16_or_null(num_runs))
        return EP_ERR_INVALID;
    NodeArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.staging = prob_staging;
    a.in_node = is_token_in_node;
    a.T = T;
    a.H = H;
    a.N = num_nodes;
    a.P = with_prob ? P : 0;
    a.max_tokens = max_tokens;
    a.chunk = chunk_tokens;
    a.nchunks = (T + chunk_tokens - 1) / chunk_tokens;
    a.dense = dense;
    a.recv_x = static_cast<uint16_t*>(recv_x_node);
    a.recv_prob = with_prob ? recv_prob_node : nullptr;
    a.num_runs = num_runs;
    const NodeScatter sp{a, static_cast<char*>(recv_x_node), static_cast<uint32_t>(H) * 2u, nullptr};
    const ep_status_t st = launch_scatter_rows(sp, T, as_stream(stream));
    if (st != EP_ERR_INVALID) return st;  // rows too large for the shared-memory buffers: registers
    const long long work = static_cast<long long>(T) > static_cast<long long>(num_nodes) * a.nchunks
                               ? T
                               : static_cast<long long>(num_nodes) * a.nchunks;
    const long long want = (work + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    node_dispatch_kernel<<<grid, kThreads, 0, as_stream(stream)>>>(a);
    return check_launch();
}
