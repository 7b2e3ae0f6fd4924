// ep_restripe.cu -- prob restripe [T][nodes][P] -> [nodes][max_tokens][P]
// ("[PR #634] Hybrid ep nixl restripe", sections "Baseline problem" and "Fix").
//
// The page's kernel gives one CTA to each (token, destination) and lets its
// threads copy the P floats with vector loads. Here one warp moves one
// (token, destination) slice of P floats in 16-byte vectors (P = 128 is
// exactly one 512-byte warp transaction). Slices are numbered destination-
// major, so consecutive warps write consecutive rows of one destination slab
// (fully coalesced stores) while their reads stride by nodes * P floats. The
// kernel is a pure copy bound by HBM bandwidth: 2 * T * nodes * P * 4 bytes.
#include "ep_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads)
    restripe_kernel(const float* __restrict__ prob, int T, int N, int P, int max_tokens, float* __restrict__ out) {
    const int lane = ep::lane_id();
    const int nvec = P / 4;
    const long long slices = static_cast<long long>(T) * N;
    for (long long q = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); q < slices;
         q += static_cast<long long>(gridDim.x) * kWarps) {
        const int n = static_cast<int>(q / T);
        const int t = static_cast<int>(q - static_cast<long long>(n) * T);
        const uint4* src = reinterpret_cast<const uint4*>(prob + (static_cast<size_t>(t) * N + n) * P);
        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(n) * max_tokens + t) * P);
        for (int v = lane; v < nvec; v += 32) ep::st_v4(dst + v, ep::ld_stream_v4(src + v));
    }
}

}  // namespace

extern "C" ep_status_t ep_restripe_prob(const float* prob, int32_t T, int32_t num_nodes, int32_t P,
                                        int32_t max_tokens, float* out, void* stream) {
    using namespace ep;
    if (T < 0 || num_nodes < 1 || P < 4 || P % 4 != 0 || max_tokens < T) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (prob == nullptr || out == nullptr || !aligned16(prob) || !aligned16(out)) return EP_ERR_INVALID;
    const long long slices = static_cast<long long>(T) * num_nodes;
    long long want = (slices + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    restripe_kernel<<<grid, kThreads, 0, as_stream(stream)>>>(prob, T, num_nodes, P, max_tokens, out);
    return check_launch();
}
