// ep_tma.cuh -- tiled tensor copies (TMA, cp.async.bulk.tensor) over this GPU's own
// memory: the host side encodes a tensor map, the device side moves boxes between global
// and shared memory. Internal header.
//
// A tensor map names a strided array by its dimensions (innermost first) and the byte
// stride of every outer dimension; the strides need not grow, so one map may walk an
// array in another order than it is stored (the restripe uses that to transpose). A box
// load writes the box into shared memory with dimension 0 fastest; coordinates past a
// dimension's end read zeros, and a box store skips elements past the end. Rules the
// host checks before encoding: the base address and every stride are multiples of 16
// bytes, dimension 0 of a box spans a multiple of 16 bytes, every box dimension is at
// most 256 elements; the device side only ever uses x = 0 (aligned) and non-negative
// coordinates.
#pragma once

#include <cuda.h>

#include "ep_common.cuh"

namespace ep {

// Encodes a tiled tensor map of `rank` dimensions (dims[0] innermost, element size
// elem_bytes, strides[i] = byte stride of dimension i + 1). Returns EP_OK, EP_ERR_INVALID
// when the shape breaks a rule above, or EP_ERR_CUDA when the driver refuses it.
ep_status_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType type, uint32_t elem_bytes, uint32_t rank,
                              const void* base, const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

// ---------------------------------------------------------------- device side

__device__ __forceinline__ uint64_t tmap_addr(const CUtensorMap& m) { return reinterpret_cast<uint64_t>(&m); }

// 3-D box global -> shared, completing on an mbarrier (tx bytes = the whole box)
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap& map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_addr(dst_smem)),
        "l"(tmap_addr(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// 3-D box shared -> global in the issuing thread's current bulk group
__device__ __forceinline__ void tma_store_3d(const CUtensorMap& map, int x, int y, int z, const void* src_smem) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(tmap_addr(map)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_addr(src_smem))
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap& m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap_addr(m)) : "memory");
}

}  // namespace ep
