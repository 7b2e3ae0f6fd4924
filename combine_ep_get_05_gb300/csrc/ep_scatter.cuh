// ep_scatter.cuh -- "read a row once, write it to several destination rows" with bulk
// asynchronous copies (TMA), shared by the rank-level dispatch, the fused
// dispatch + permute and the node-level dispatch. Internal header.
//
// One warp per CTA and kScatterStages row buffers in shared memory. Lane 0 streams the
// CTA's source rows (items blockIdx.x, +gridDim.x, ...) into the buffers with bulk
// global->shared copies that complete on an mbarrier, kScatterStages-1 rows ahead of
// use, and sends each row to every destination with one bulk shared->global copy; a
// buffer is refilled only after the bulk stores that read it have finished reading it.
// The other lanes resolve destinations and write metadata meanwhile. No row data passes
// through registers, so the load/store unit queue stays free; the grid has one CTA per
// 1.5 rows, so the block scheduler balances rows with different numbers of
// destinations. Every barrier wait is bounded: on timeout the kernel waits (bounded) for
// its own loads still in flight, raises EP_FLAG_TIMEOUT and stops. It runs as a dependent launch (its CTAs may start while the previous kernel
// finishes, and wait for it before reading anything) and lets the next kernel be
// scheduled once every CTA is past its last row.
//
// A Spec is a trivially copyable struct with these device members, called by all 32
// lanes of the warp:
//   int items() const;                              number of source rows
//   const void* source(int i) const;                row i (row_bytes, 16-byte aligned)
//   int destinations(int i, long long* rows, int* aux) const;
//       fills rows[0..nd) with destination row indices (units of row_bytes from dst),
//       aux with per-destination data for side_work, ends with __syncwarp, returns nd
//   void side_work(int i, int nd, const long long* rows, const int* aux) const;
//   void prologue() const;                          once per CTA, before the rows
// and members `char* dst`, `uint32_t row_bytes`, `int32_t* status`.
#pragma once

#include "ep_common.cuh"

namespace ep {

constexpr int kScatterStages = 3;
constexpr int kScatterMaxDest = 256;
constexpr size_t kScatterMaxSmem = 200 * 1024;

template <class Spec>
__global__ void __launch_bounds__(32) scatter_rows_tma_kernel(Spec spec) {
    extern __shared__ __align__(128) unsigned char s_rows[];
    __shared__ __align__(8) uint64_t s_bar[kScatterStages];
    __shared__ long long s_dst[kScatterMaxDest];
    __shared__ int s_aux[kScatterMaxDest];
    grid_dependency_wait();  // launched as a dependent launch: inputs are ready after this
    const int lane = lane_id();
    const uint32_t rowb = spec.row_bytes;
    const int n_items = spec.items();
    const int first = static_cast<int>(blockIdx.x);
    const int step = static_cast<int>(gridDim.x);
    const int n_my = first < n_items ? (n_items - 1 - first) / step + 1 : 0;
    spec.prologue();

    int issued = 0;  // loads issued by lane 0: items 0 .. issued-1 of this CTA
    if (lane == 0) {
        for (int st = 0; st < kScatterStages; ++st) mbar_init(&s_bar[st], 1);
        mbar_init_fence();
        for (; issued < kScatterStages - 1 && issued < n_my; ++issued) {
            mbar_arrive_expect_tx(&s_bar[issued], rowb);
            bulk_load(s_rows + static_cast<size_t>(issued) * rowb, spec.source(first + issued * step), rowb,
                      &s_bar[issued]);
        }
    }
    __syncwarp();
    int j = 0;
    bool ok = true;
    for (; j < n_my && ok; ++j) {
        const int i = first + j * step;
        const int st = j % kScatterStages;
        const int nd = spec.destinations(i, s_dst, s_aux);
        spec.side_work(i, nd, s_dst, s_aux);
        if (lane == 0) {
            if (issued < n_my && issued == j + kScatterStages - 1) {
                bulk_wait_read_all();  // the buffer of item j-1 is free once its stores have read it
                const int sn = issued % kScatterStages;
                mbar_arrive_expect_tx(&s_bar[sn], rowb);
                bulk_load(s_rows + static_cast<size_t>(sn) * rowb, spec.source(first + issued * step), rowb,
                          &s_bar[sn]);
                ++issued;
            }
            ok = mbar_wait_bounded(&s_bar[st], static_cast<uint32_t>((j / kScatterStages) & 1));
            if (ok) {
                const unsigned char* buf = s_rows + static_cast<size_t>(st) * rowb;
                for (int d = 0; d < nd; ++d) bulk_store(spec.dst + static_cast<size_t>(s_dst[d]) * rowb, buf, rowb);
                bulk_commit();
            }
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        __syncwarp();
    }
    allow_dependents();  // the next kernel may be scheduled once every CTA is past its rows
    if (lane == 0) {
        bulk_wait_read_all();  // the buffers may be released once the stores have read them
        if (!ok) {
            // item j-1 timed out: wait (bounded) for every load still in flight before leaving
            for (int q = j - 1; q < issued; ++q)
                (void)mbar_wait_bounded(&s_bar[q % kScatterStages], static_cast<uint32_t>((q / kScatterStages) & 1));
            raise_flag(spec.status, EP_FLAG_TIMEOUT);
        }
    }
}

// Launch the scatter for `items` rows of `row_bytes`. Returns EP_OK / EP_ERR_CUDA, or
// EP_ERR_INVALID when kScatterStages rows do not fit in shared memory (the caller then
// uses its register kernel).
template <class Spec>
ep_status_t launch_scatter_rows(const Spec& spec, int items, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(kScatterStages) * spec.row_bytes;
    if (smem > kScatterMaxSmem || spec.row_bytes % 16 != 0) return EP_ERR_INVALID;
    static std::atomic<int> attr_set[kMaxDevices];  // per device, for each Spec instantiation
    const ep_status_t attr = ensure_dynamic_smem(attr_set, scatter_rows_tma_kernel<Spec>,
                                                 static_cast<int>(kScatterMaxSmem));
    if (attr != EP_OK) return attr;
    // one CTA per 1.5 rows: a third of the CTAs take a second row, whose load overlaps the
    // first row's stores, and the block scheduler still balances rows with different
    // numbers of destinations (measured best for 4096 x 7168 and 16384 x 4096 bf16 batches)
    const long long rows = items > 0 ? items : 1;
    const long long grid = (2 * rows + 2) / 3;
    return launch_dependent(scatter_rows_tma_kernel<Spec>, dim3(static_cast<unsigned>(grid)), dim3(32), smem, stream,
                            spec);
}

}  // namespace ep
