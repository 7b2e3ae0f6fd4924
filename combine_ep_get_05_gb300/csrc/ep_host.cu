// ep_host.cu -- library-wide host entry points and launch-sizing helpers.
#include <atomic>

#include "ep_common.cuh"
#include "ep_tma.cuh"

namespace ep {

namespace {
std::atomic<int> g_sm_count[kMaxDevices];
thread_local int g_last_cuda_error = 0;
}  // namespace

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 152;
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

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::atomic<EncodeTiledFn> g_encode_tiled{nullptr};
}  // namespace

ep_status_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, uint32_t elem_bytes, uint32_t rank,
                              const void* base, const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
    if (rank < 1 || rank > 5 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return EP_ERR_INVALID;
    if ((static_cast<uint64_t>(box[0]) * elem_bytes) % 16 != 0) return EP_ERR_INVALID;
    for (uint32_t i = 0; i < rank; ++i) {
        if (box[i] < 1 || box[i] > 256 || dims[i] < 1 || dims[i] > (1ull << 32)) return EP_ERR_INVALID;
        if (i + 1 < rank && (strides[i] % 16 != 0 || strides[i] >= (1ull << 40))) return EP_ERR_INVALID;
    }
    EncodeTiledFn fn = g_encode_tiled.load(std::memory_order_acquire);
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        const cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err != cudaSuccess) return cuda_fail(err);
        if (q != cudaDriverEntryPointSuccess || p == nullptr) return cuda_fail(cudaErrorSymbolNotFound);
        fn = reinterpret_cast<EncodeTiledFn>(p);
        g_encode_tiled.store(fn, std::memory_order_release);
    }
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides[i];
    }
    const CUresult r = fn(map, type, rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? EP_OK : cuda_fail(cudaErrorInvalidValue);
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
