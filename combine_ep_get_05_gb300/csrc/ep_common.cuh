// ep_common.cuh -- helpers shared by the library's translation units (device
// PTX wrappers, argument checks, per-device launch sizing). Internal header.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------- host side

// SM count of the current device (cached per device ordinal).
int sm_count();

// Record a CUDA error for ep_last_cuda_error() and map it to EP_ERR_CUDA.
ep_status_t cuda_fail(cudaError_t err);

// EP_OK after a launch, or EP_ERR_CUDA if the launch was rejected.
ep_status_t check_launch();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned16_or_null(const void* p) { return p == nullptr || aligned16(p); }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

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

// hint: bring the line holding p into L2 (no register result, never faults on a valid address)
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

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

}  // namespace ep
