// ep_restripe.cu -- prob restripe [T][nodes][P] -> [nodes][max_tokens][P]
// ("[PR #634] Hybrid ep nixl restripe", sections "Baseline problem" and "Fix").
//
// The page's kernel gives one CTA to each (token, destination) and lets its threads copy
// the P floats with vector loads. Here the copy is a transpose of the two outer
// dimensions done by the tensor-memory accelerator: the source is described by a 3-D
// tensor map whose dimensions are taken in the order (p, t, n) -- strides 4, N*P*4 and
// P*4 bytes -- so one box load of (P, m tokens, nb nodes) lands in shared memory already
// laid out [n][t][p], exactly the order of a box of the destination map (p, t, n) with
// strides 4, P*4 and max_tokens*P*4 bytes. A tile therefore costs one tensor load and one
// tensor store, issued by a single thread; the SM does no per-byte work.
//
// A persistent grid (one CTA per SM) walks the tiles; each CTA keeps up to 16 tiles of
// ~16 KB in flight in a ring of shared-memory stages: a stage is refilled once the store
// that read it has finished reading. The destination map's token dimension is T, so the
// store of a ragged last tile skips rows t >= T (rows [T, max_tokens) are never written).
// Every barrier wait is bounded in time. The kernel is a pure copy bound by HBM
// bandwidth: 2 * T * nodes * P * 4 bytes.
//
// Shapes the tensor maps cannot take (P > 256 floats) use restripe_warp_kernel: a warp per
// (token, node) slice, four slices in flight per warp, 16-byte vectors.
#include <algorithm>

#include "ep_common.cuh"
#include "ep_tma.cuh"

namespace {

using namespace ep;

constexpr int kMaxStages = 16;
constexpr uint32_t kTileTarget = 16 * 1024;  // bytes per tile
constexpr uint32_t kSmemBudget = 192 * 1024;

struct RestripeTiles {
    int tiles_n;          // node blocks per token block
    int n_tiles;          // token blocks * node blocks
    int m, nb;            // box: m tokens x nb nodes (x P floats)
    uint32_t tile_bytes;  // P * m * nb * 4
    uint32_t stride;      // stage stride in shared memory (tile_bytes rounded up to 128)
    int stages;
};

__global__ void __launch_bounds__(32) restripe_tma_kernel(const __grid_constant__ CUtensorMap src,
                                                          const __grid_constant__ CUtensorMap dst, RestripeTiles g) {
    extern __shared__ __align__(128) unsigned char s_tiles[];
    __shared__ __align__(8) uint64_t s_bar[kMaxStages];
    grid_dependency_wait();  // dependent launch: the prob tensor is complete after this
    if (threadIdx.x != 0) return;
    const int first = static_cast<int>(blockIdx.x);
    const int step = static_cast<int>(gridDim.x);
    const int n_my = first < g.n_tiles ? (g.n_tiles - 1 - first) / step + 1 : 0;
    prefetch_tensor_map(src);
    prefetch_tensor_map(dst);
    for (int st = 0; st < g.stages; ++st) mbar_init(&s_bar[st], 1);
    mbar_init_fence();

    // tile j of this CTA: token block q / tiles_n, node block q % tiles_n
    auto origin = [&](int j, int& t0, int& n0) {
        const int q = first + j * step;
        const int tb = q / g.tiles_n;
        t0 = tb * g.m;
        n0 = (q - tb * g.tiles_n) * g.nb;
    };
    auto load = [&](int j) {
        int t0, n0;
        origin(j, t0, n0);
        const int st = j % g.stages;
        mbar_arrive_expect_tx(&s_bar[st], g.tile_bytes);
        tma_load_3d(s_tiles + static_cast<size_t>(st) * g.stride, src, 0, t0, n0, &s_bar[st]);
    };

    int issued = 0;
    for (; issued < g.stages && issued < n_my; ++issued) load(issued);
    int j = 0;
    bool ok = true;
    for (; j < n_my; ++j) {
        const int st = j % g.stages;
        ok = mbar_wait_bounded(&s_bar[st], static_cast<uint32_t>((j / g.stages) & 1));
        if (!ok) break;
        int t0, n0;
        origin(j, t0, n0);
        tma_store_3d(dst, 0, t0, n0, s_tiles + static_cast<size_t>(st) * g.stride);
        bulk_commit();
        if (j >= 1 && issued < n_my) {
            // the stage of tile j - 1 takes tile issued = j - 1 + stages once its store
            // has finished reading it (every bulk group but the newest)
            bulk_wait_read<1>();
            load(issued);
            ++issued;
        }
    }
    allow_dependents();
    if (!ok) {
        // a load never completed (the hardware gave up): wait, bounded, for the loads still
        // in flight before the CTA releases its shared memory; the copy stays incomplete
        for (int q = j; q < issued; ++q)
            (void)mbar_wait_bounded(&s_bar[q % g.stages], static_cast<uint32_t>((q / g.stages) & 1));
    }
    bulk_wait_all();
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlices = 4;  // slices a warp has in flight

// Fallback: blockIdx.y = node n; warps walk the tokens, kSlices slices at a time.
__global__ void __launch_bounds__(kThreads)
    restripe_warp_kernel(const float* __restrict__ prob, int T, int N, int P, int max_tokens, float* __restrict__ out) {
    grid_dependency_wait();
    const int lane = lane_id();
    const int n = static_cast<int>(blockIdx.y);
    const int nvec = P / 4;
    const int warps = static_cast<int>(gridDim.x) * kWarps;
    for (int t0 = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(threadIdx.x >> 5); t0 < T;
         t0 += warps * kSlices) {
        for (int v = lane; v < nvec; v += 32) {
            uint4 buf[kSlices];
#pragma unroll
            for (int i = 0; i < kSlices; ++i) {
                const int t = t0 + i * warps;
                if (t < T)
                    buf[i] = ld_stream_v4(reinterpret_cast<const uint4*>(prob + (static_cast<size_t>(t) * N + n) * P) + v);
            }
#pragma unroll
            for (int i = 0; i < kSlices; ++i) {
                const int t = t0 + i * warps;
                if (t < T) st_v4(reinterpret_cast<uint4*>(out + (static_cast<size_t>(n) * max_tokens + t) * P) + v, buf[i]);
            }
        }
    }
}

std::atomic<int> g_tma_smem_set[kMaxDevices];

}  // namespace

extern "C" ep_status_t ep_restripe_prob(const float* prob, int32_t T, int32_t num_nodes, int32_t P,
                                        int32_t max_tokens, float* out, void* stream) {
    using namespace ep;
    if (T < 0 || num_nodes < 1 || num_nodes > 65535 || P < 4 || P % 4 != 0 || max_tokens < T) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (prob == nullptr || out == nullptr || !aligned16(prob) || !aligned16(out)) return EP_ERR_INVALID;
    const cudaStream_t s = as_stream(stream);
    const uint32_t slice = static_cast<uint32_t>(P) * 4u;
    if (P <= 256) {
        RestripeTiles g{};
        g.nb = num_nodes <= 256 && slice * num_nodes <= kTileTarget ? num_nodes
                                                                    : static_cast<int>(std::max(1u, kTileTarget / slice));
        if (g.nb > 256) g.nb = 256;
        g.m = static_cast<int>(std::max(1u, kTileTarget / (slice * static_cast<uint32_t>(g.nb))));
        if (g.m > 256) g.m = 256;
        if (g.m > T) g.m = T;
        g.tile_bytes = slice * static_cast<uint32_t>(g.m) * static_cast<uint32_t>(g.nb);
        g.stride = (g.tile_bytes + 127u) & ~127u;
        g.stages = static_cast<int>(std::min<uint32_t>(kMaxStages, kSmemBudget / g.stride));
        g.tiles_n = (num_nodes + g.nb - 1) / g.nb;
        const long long n_tiles = static_cast<long long>((T + g.m - 1) / g.m) * g.tiles_n;
        if (g.stages >= 2 && n_tiles < (1ll << 31)) {
            g.n_tiles = static_cast<int>(n_tiles);
            // source walked as (p, t, n); destination as (p, t, n) with t limited to T
            const uint64_t sdims[3] = {static_cast<uint64_t>(P), static_cast<uint64_t>(T), static_cast<uint64_t>(num_nodes)};
            const uint64_t sstr[2] = {static_cast<uint64_t>(num_nodes) * slice, slice};
            const uint64_t dstr[2] = {slice, static_cast<uint64_t>(max_tokens) * slice};
            const uint32_t box[3] = {static_cast<uint32_t>(P), static_cast<uint32_t>(g.m), static_cast<uint32_t>(g.nb)};
            CUtensorMap src_map, dst_map;
            ep_status_t st = encode_tensor_map(&src_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, prob, sdims, sstr, box);
            if (st != EP_OK) return st;
            st = encode_tensor_map(&dst_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, out, sdims, dstr, box);
            if (st != EP_OK) return st;
            const size_t smem = static_cast<size_t>(g.stages) * g.stride;
            st = ensure_dynamic_smem(g_tma_smem_set, restripe_tma_kernel, static_cast<int>(kSmemBudget));
            if (st != EP_OK) return st;
            const long long grid = std::min<long long>(n_tiles, sm_count());
            return launch_dependent(restripe_tma_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), smem, s, src_map,
                                    dst_map, g);
        }
    }
    const long long want = (static_cast<long long>(T) + kWarps * kSlices - 1) / (kWarps * kSlices);
    const long long cap = std::max<long long>(1, static_cast<long long>(sm_count()) * 8 / num_nodes);
    const dim3 grid(static_cast<unsigned>(std::min(want, cap)), static_cast<unsigned>(num_nodes));
    return launch_dependent(restripe_warp_kernel, grid, dim3(kThreads), 0, s, prob, T, num_nodes, P, max_tokens, out);
}
