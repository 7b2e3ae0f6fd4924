// ep_common.cuh -- helpers shared by the library's translation units (device
// PTX wrappers, argument checks, per-device launch sizing). Internal header.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------- host side

constexpr int kMaxDevices = 64;  // device ordinals the per-device caches below cover

// SM count of the current device (cached per device ordinal).
int sm_count();

// Record a CUDA error for ep_last_cuda_error() and map it to EP_ERR_CUDA.
ep_status_t cuda_fail(cudaError_t err);

// EP_OK after a launch, or EP_ERR_CUDA if the launch was rejected.
ep_status_t check_launch();

// Ordinal of the current device, or -1 if there is none or it is >= kMaxDevices.
inline int current_device() {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices ? dev : -1;
}

// Per-device launch caches. Each is an array of kMaxDevices atomics owned by the caller
// (static storage, so zero = "not known yet"). Host threads may make their first calls
// on a device at the same time: both compute the same value and store it; the atomics
// keep those accesses free of data races.

// Lets `kernel` use `bytes` of dynamic shared memory, once per device.
template <typename Kernel>
ep_status_t ensure_dynamic_smem(std::atomic<int>* done, Kernel* kernel, int bytes) {
    const int dev = current_device();
    if (dev >= 0 && done[dev].load(std::memory_order_acquire) != 0) return EP_OK;
    const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err != cudaSuccess) return cuda_fail(err);
    if (dev >= 0) done[dev].store(1, std::memory_order_release);
    return EP_OK;
}

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of dynamic shared
// memory on the current device (at least 1), computed once per device.
template <typename Kernel>
ep_status_t blocks_per_sm(std::atomic<int>* cache, Kernel* kernel, int threads, size_t smem, int* out) {
    const int dev = current_device();
    int n = dev >= 0 ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        const cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
        if (err != cudaSuccess) return cuda_fail(err);
        if (n < 1) n = 1;
        if (dev >= 0) cache[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return EP_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned16_or_null(const void* p) { return p == nullptr || aligned16(p); }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch kernel<<<grid, block, smem, stream>>>(args...) as a programmatic dependent launch:
// it may be scheduled before the previous kernel of the stream has ended, once every CTA
// of that kernel has called allow_dependents() (or ended), so its CTAs are resident and
// set up when the data arrives. The kernel must call grid_dependency_wait() before it
// reads global memory: that wait returns once the previous kernel has completed and its
// writes are visible. Returns EP_OK or EP_ERR_CUDA.
template <typename... KArgs, typename... Args>
ep_status_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return err == cudaSuccess ? check_launch() : cuda_fail(err);
}

// ---------------------------------------------------------------- device side

__device__ __forceinline__ int lane_id() { return static_cast<int>(threadIdx.x & 31u); }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ void raise_flag(int32_t* status, int32_t bits) {
    if (status != nullptr) atomicOr(status, bits);
}

// 16-byte read of data that no thread writes during the kernel; not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// gpu-scope relaxed 64-bit load/store (single-copy atomic, coherent at L2)
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Returns the old value; release covers the writes that a preceding __syncthreads
// ordered before it, acquire makes the other CTAs' released writes visible.
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Programmatic dependent launch, device side: wait until the previous kernel of the
// stream has completed and its writes are visible (returns at once for an ordinary
// launch); and allow the next kernel, if launched with launch_dependent, to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// hint: bring the line holding p into L2 (no register result, never faults on a valid address)
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- bulk async copies (TMA)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// make barrier initialisation visible to the async (bulk copy) proxy
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// wait for the barrier phase with the given parity; gives up after ~1 s and returns false
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_addr(bar);
    const unsigned long long start = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 255u) == 255u && globaltimer_ns() - start > 1000000000ull) return false;
    }
    return false;
}
// global -> shared bulk copy completing on an mbarrier (bytes % 16 == 0, both 16-byte aligned)
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
// shared -> global bulk copy in the issuing thread's current bulk group
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src_smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all committed bulk stores of this thread have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all committed bulk stores of this thread but the newest `N` have finished reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// all committed bulk stores of this thread are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// make this thread's ordinary shared-memory writes visible to later bulk copies (async proxy)
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// bf16 pair (one 32-bit word, element 0 in the low half) -> two fp32, exact
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// two fp32 -> bf16 pair, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// two fp32 -> two OCP E4M3 codes, round to nearest even, saturating to +-448
// (lo in bits 0..7, hi in bits 8..15)
__device__ __forceinline__ uint32_t pack_e4m3x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// four fp32 -> four OCP E4M3 codes (a in byte 0 ... d in byte 3), each rounded to nearest
// even and saturated to +-448
__device__ __forceinline__ uint32_t pack_e4m3x4_rn_sat(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n"
        " .reg .b16 lo, hi;\n"
        " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        " mov.b32 %0, {lo, hi};\n"
        "}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// two OCP E4M3 codes (byte 0 -> low half, byte 1 -> high half) -> two fp16, exactly
// (every E4M3 value is an fp16 value); then fp16 -> fp32, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t r;
    const uint16_t c = static_cast<uint16_t>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}
// four OCP E4M3 codes (byte i of w) -> four fp32 values, exactly: each 16-bit half of w
// becomes an fp16 pair (every E4M3 value is an fp16 value) and each fp16 an fp32; the
// halves are named as 16-bit registers so no masking or shifting is needed
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float& a, float& b, float& c, float& d) {
    asm("{\n"
        " .reg .b16 c0, c1, f0, f1, f2, f3;\n"
        " .reg .b32 h01, h23;\n"
        " mov.b32 {c0, c1}, %4;\n"
        " cvt.rn.f16x2.e4m3x2 h01, c0;\n"
        " cvt.rn.f16x2.e4m3x2 h23, c1;\n"
        " mov.b32 {f0, f1}, h01;\n"
        " mov.b32 {f2, f3}, h23;\n"
        " cvt.f32.f16 %0, f0;\n"
        " cvt.f32.f16 %1, f1;\n"
        " cvt.f32.f16 %2, f2;\n"
        " cvt.f32.f16 %3, f3;\n"
        "}"
        : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
        : "r"(w));
}
__device__ __forceinline__ float f16_to_f32(uint32_t h) {
    float f;
    const uint16_t b = static_cast<uint16_t>(h);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(b));
    return f;
}


// ---------------------------------------------------------------- per-thread async copies
// global -> shared copies performed by the issuing thread in the background; a thread's
// copies are grouped by commit and waited on by group count (a hardware wait, no spin)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
// issued only where `p` holds (a predicate, not a branch)
__device__ __forceinline__ void cp_async16_if(void* smem, const void* gmem, bool p) {
    asm volatile(
        "{\n"
        " .reg .pred q;\n"
        " setp.ne.b32 q, %2, 0;\n"
        " @q cp.async.cg.shared.global [%0], [%1], 16;\n"
        "}" ::"r"(smem_addr(smem)),
        "l"(gmem), "r"(static_cast<int>(p))
        : "memory");
}
__device__ __forceinline__ void cp_async4_if(void* smem, const void* gmem, bool p) {
    asm volatile(
        "{\n"
        " .reg .pred q;\n"
        " setp.ne.b32 q, %2, 0;\n"
        " @q cp.async.ca.shared.global [%0], [%1], 4;\n"
        "}" ::"r"(smem_addr(smem)),
        "l"(gmem), "r"(static_cast<int>(p))
        : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// until at most N of the thread's newest groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- paired fp32 arithmetic
// Two channels per instruction with the roundings of the scalar definition. The product is
// a paired fused multiply-add with a zero: RN(f * s + -0) = RN(f * s) for every f and s,
// zeros and their signs included, so with nz = -0 it is the rounded product; the zero
// comes in at run time because a plain paired multiply, or one with a constant zero, is
// contracted with a following paired add into one fused multiply-add (one rounding) by the
// code generator.

// a0, a1 = RN(a0 + RN(f0 * s)), RN(a1 + RN(f1 * s)); nz = -0
__device__ __forceinline__ void pair_add_product(float& a0, float& a1, float f0, float f1, float s, float nz) {
    asm("{\n"
        " .reg .b64 f, w, z, p, a;\n"
        " mov.b64 f, {%2, %3};\n"
        " mov.b64 w, {%4, %4};\n"
        " mov.b64 z, {%5, %5};\n"
        " fma.rn.f32x2 p, f, w, z;\n"
        " mov.b64 a, {%0, %1};\n"
        " add.rn.f32x2 a, a, p;\n"
        " mov.b64 {%0, %1}, a;\n"
        "}"
        : "+f"(a0), "+f"(a1)
        : "f"(f0), "f"(f1), "f"(s), "f"(nz));
}
// a0, a1 = RN(f0 * s + z), RN(f1 * s + z), one rounding each
__device__ __forceinline__ void pair_fma(float& a0, float& a1, float f0, float f1, float s, float z) {
    asm("{\n"
        " .reg .b64 f, w, y, a;\n"
        " mov.b64 f, {%2, %3};\n"
        " mov.b64 w, {%4, %4};\n"
        " mov.b64 y, {%5, %5};\n"
        " fma.rn.f32x2 a, f, w, y;\n"
        " mov.b64 {%0, %1}, a;\n"
        "}"
        : "=f"(a0), "=f"(a1)
        : "f"(f0), "f"(f1), "f"(s), "f"(z));
}
// a0, a1 = RN(a0 + f0), RN(a1 + f1)
__device__ __forceinline__ void pair_add(float& a0, float& a1, float f0, float f1) {
    asm("{\n"
        " .reg .b64 f, a;\n"
        " mov.b64 f, {%2, %3};\n"
        " mov.b64 a, {%0, %1};\n"
        " add.rn.f32x2 a, a, f;\n"
        " mov.b64 {%0, %1}, a;\n"
        "}"
        : "+f"(a0), "+f"(a1)
        : "f"(f0), "f"(f1));
}

}  // namespace ep
