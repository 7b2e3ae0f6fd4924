// ep_host.cu -- library-wide host entry points and launch-sizing helpers.
#include <atomic>

#include "ep_common.cuh"

namespace ep {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
thread_local int g_last_cuda_error = 0;
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

ep_status_t cuda_fail(cudaError_t err) {
    g_last_cuda_error = static_cast<int>(err);
    return EP_ERR_CUDA;
}

ep_status_t check_launch() {
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? EP_OK : cuda_fail(err);
}

}  // namespace ep

extern "C" {

int32_t ep_abi_version(void) { return EP_ABI_VERSION; }

const char* ep_status_str(ep_status_t s) {
    switch (s) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID: return "EP_ERR_INVALID: an argument was rejected; nothing was launched";
        case EP_ERR_CUDA: return "EP_ERR_CUDA: a CUDA launch or runtime call failed";
        case EP_ERR_SCRATCH:
            return "EP_ERR_SCRATCH: the sizes need more layout workspace than the fixed scratch of "
                   "ep_get_layout_noalloc holds; call ep_get_layout with a workspace instead";
        default: return "unknown ep_status_t";
    }
}

// cudaError_t of the most recent EP_ERR_CUDA returned on this host thread (0 if none).
int32_t ep_last_cuda_error(void) { return ep::g_last_cuda_error; }

}  // extern "C"
