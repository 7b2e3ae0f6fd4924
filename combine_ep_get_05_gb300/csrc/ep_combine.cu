// ep_combine.cu -- combine: gather every rank's expert output for a token and
// reduce it back in token order ("[PR #347] Feature/sm free normal kernel",
// 2.1 Feature; BF16 combine of 3.2.1).
//
//   out[t][h] = bf16_rn( ((0 + y[r0][s0][h]) + y[r1][s1][h]) + ... ),  r0 < r1 < ...
//
// Work is split into items of (token, group of 32 output vectors): one warp
// item covers 32 lanes x 8 channels = 256 channels of one token. Each CTA takes a
// contiguous range of items, so every SM gets the same amount of work whatever
// T is, and consecutive warps of a CTA share a token (its slot row stays in L1).
// Per item the warp reads the token's slot row (lanes across ranks) and
// compacts the contributing rows in ascending rank order with a ballot, issues
// the loads of up to 8 source rows at once, and adds them into fp32
// accumulators strictly in that order (one IEEE addition per term, no
// reassociation); then it stores one bf16 vector rounded to nearest even. The
// kernel is capped at 64 registers so four 256-thread CTAs fit on an SM, which
// keeps enough loads in flight to saturate HBM: it reads one row per (token,
// rank) pair and writes T rows.
#include "ep_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSrc = 256;  // = largest R: every rank may contribute
constexpr int kBatch = 8;  // source rows loaded together
constexpr int kMinBlocks = 4;  // CTAs per SM the register budget is sized for
constexpr int kBatchFp8 = 4;  // FP8 source rows loaded together (16 codes = half the bytes of 8 bf16)

__device__ __forceinline__ void add8(float* acc, const uint4& v) {
    acc[0] = __fadd_rn(acc[0], ep::bf16_lo(v.x));
    acc[1] = __fadd_rn(acc[1], ep::bf16_hi(v.x));
    acc[2] = __fadd_rn(acc[2], ep::bf16_lo(v.y));
    acc[3] = __fadd_rn(acc[3], ep::bf16_hi(v.y));
    acc[4] = __fadd_rn(acc[4], ep::bf16_lo(v.z));
    acc[5] = __fadd_rn(acc[5], ep::bf16_hi(v.z));
    acc[6] = __fadd_rn(acc[6], ep::bf16_lo(v.w));
    acc[7] = __fadd_rn(acc[7], ep::bf16_hi(v.w));
}

__global__ void __launch_bounds__(kThreads, kMinBlocks)
    combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ slot, int T, int H, int R,
                   int max_tokens, uint16_t* __restrict__ out, int32_t* status) {
    ep::grid_dependency_wait();  // dependent launch: the slabs are complete after this
    __shared__ long long s_src[kWarps][kMaxSrc];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = H / 8;
    const int ngroups = (nvec + 31) / 32;
    const long long items = static_cast<long long>(T) * ngroups;
    const long long i0 = static_cast<long long>(blockIdx.x) * items / gridDim.x;
    const long long i1 = static_cast<long long>(blockIdx.x + 1) * items / gridDim.x;
    const uint4* ys = reinterpret_cast<const uint4*>(y);
    uint4* os = reinterpret_cast<uint4*>(out);

    for (long long it = i0 + warp; it < i1; it += kWarps) {
        const int t = static_cast<int>(it / ngroups);
        const int v = static_cast<int>(it - static_cast<long long>(t) * ngroups) * 32 + lane;
        int ns = 0;
        bool over_any = false;
        for (int r0 = 0; r0 < R; r0 += 32) {
            const int r = r0 + lane;
            const int s = r < R ? slot[static_cast<size_t>(t) * R + r] : -1;
            const bool over = s >= max_tokens;
            over_any |= over;
            const bool ok = s >= 0 && !over;
            const uint32_t m = __ballot_sync(ep::kFullMask, ok);
            if (ok) s_src[warp][ns + __popc(m & ep::lanemask_lt())] = (static_cast<long long>(r) * max_tokens + s) * nvec;
            ns += __popc(m);
        }
        // one report per token: the item that starts the token's row
        if (over_any && v == lane) ep::raise_flag(status, EP_FLAG_CAPACITY);
        __syncwarp();

        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int d0 = 0; d0 < ns; d0 += kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (d0 + i < ns && v < nvec) buf[i] = ep::ld_stream_v4(ys + s_src[warp][d0 + i] + v);
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (d0 + i < ns) add8(acc, buf[i]);
        }
        if (v < nvec) {
            uint4 o;
            o.x = ep::pack_bf16x2_rn(acc[0], acc[1]);
            o.y = ep::pack_bf16x2_rn(acc[2], acc[3]);
            o.z = ep::pack_bf16x2_rn(acc[4], acc[5]);
            o.w = ep::pack_bf16x2_rn(acc[6], acc[7]);
            ep::st_v4(os + static_cast<size_t>(t) * nvec + v, o);
        }
        __syncwarp();
    }
}

// Combine of FP8 rows (E4M3 codes [R][max_tokens][H], one fp32 scale per 128 channels
// [R][max_tokens][H/128]). Items are (token, 32 lanes x 16 channels); each warp takes a
// contiguous run of its CTA's items, so consecutive items mostly belong to one token and
// the token's compacted source list (ascending rank) is built once and reused. Per item a
// lane loads, for kBatchFp8 sources at a time, 16 codes (one 16-byte vector) and its
// block's scale, converts the codes to fp32 exactly (E4M3 -> fp16 -> fp32 through 16-bit
// register halves) and adds __fmul_rn(code, scale) to its accumulators in source order.
// The first term is taken as fma(code, scale, +0) = RN(code * scale + 0), one instruction
// instead of two. It equals 0 + RN(code * scale) unless a nonzero product rounds to zero
// (the fused form would keep a -0): with |code| >= 2^-9 that needs a scale below 2^-140,
// so such scales (never produced by real data) take the two-instruction form.
// (The arithmetic stays scalar: a packed .f32x2 multiply feeding a packed add is
// contracted into a fused multiply-add by the code generator, one rounding instead of two.)
template <bool kFirst>
__device__ __forceinline__ void fp8_term16(float* acc, const uint4& v, float sc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float f[4];
        ep::e4m3x4_to_f32(w[q], f[0], f[1], f[2], f[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc[4 * q + i] = kFirst ? __fmaf_rn(f[i], sc, 0.0f) : __fadd_rn(acc[4 * q + i], __fmul_rn(f[i], sc));
    }
}

__device__ __forceinline__ bool fused_first_ok(float sc) { return sc == 0.0f || sc >= 0x1p-140f; }

__global__ void __launch_bounds__(kThreads, kMinBlocks)
    combine_fp8_kernel(const uint8_t* __restrict__ y, const float* __restrict__ y_scales,
                       const int32_t* __restrict__ slot, int T, int H, int R, int max_tokens,
                       uint16_t* __restrict__ out, int32_t* status) {
    ep::grid_dependency_wait();  // dependent launch: the slabs are complete after this
    __shared__ long long s_src[kWarps][kMaxSrc];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = H / 16;  // 16-code vectors per row
    const int nblk = H / 128;
    const int ngroups = (nvec + 31) / 32;
    const long long items = static_cast<long long>(T) * ngroups;
    const long long c0 = static_cast<long long>(blockIdx.x) * items / gridDim.x;
    const long long c1 = static_cast<long long>(blockIdx.x + 1) * items / gridDim.x;
    const long long i0 = c0 + (c1 - c0) * warp / kWarps;  // this warp's contiguous run
    const long long i1 = c0 + (c1 - c0) * (warp + 1) / kWarps;
    const uint4* ys = reinterpret_cast<const uint4*>(y);
    uint4* os = reinterpret_cast<uint4*>(out);

    int t_cur = -1, ns = 0;
    // (token, group) of the run's first item; later items advance it without dividing
    int t = static_cast<int>(i0 / ngroups);
    int g = static_cast<int>(i0 - static_cast<long long>(t) * ngroups);
    for (long long it = i0; it < i1; ++it) {
        const int v = g * 32 + lane;
        if (t != t_cur) {  // the token's sources, ascending rank
            t_cur = t;
            ns = 0;
            bool over_any = false;
            __syncwarp();
            for (int r0 = 0; r0 < R; r0 += 32) {
                const int r = r0 + lane;
                const int s = r < R ? slot[static_cast<size_t>(t) * R + r] : -1;
                const bool over = s >= max_tokens;
                over_any |= over;
                const bool ok = s >= 0 && !over;
                const uint32_t m = __ballot_sync(ep::kFullMask, ok);
                if (ok) s_src[warp][ns + __popc(m & ep::lanemask_lt())] = static_cast<long long>(r) * max_tokens + s;
                ns += __popc(m);
            }
            // one report per token: the warp whose run holds the token's first item
            if (__any_sync(ep::kFullMask, over_any) && lane == 0 && v < 32) ep::raise_flag(status, EP_FLAG_CAPACITY);
            __syncwarp();
        }

        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        const int blk = v / 8;  // the lane's 16 channels lie in block v / 8
        if (v < nvec) {
            for (int d0 = 0; d0 < ns; d0 += kBatchFp8) {
                uint4 buf[kBatchFp8];
                float sc[kBatchFp8];
#pragma unroll
                for (int i = 0; i < kBatchFp8; ++i) {
                    if (d0 + i < ns) {
                        const long long row = s_src[warp][d0 + i];
                        buf[i] = ep::ld_stream_v4(ys + row * nvec + v);
                        sc[i] = __ldg(y_scales + row * nblk + blk);
                    }
                }
                if (d0 == 0 && fused_first_ok(sc[0])) fp8_term16<true>(acc, buf[0], sc[0]);
                else fp8_term16<false>(acc, buf[0], sc[0]);
#pragma unroll
                for (int i = 1; i < kBatchFp8; ++i)
                    if (d0 + i < ns) fp8_term16<false>(acc, buf[i], sc[i]);
            }
            uint4 o0, o1;
            o0.x = ep::pack_bf16x2_rn(acc[0], acc[1]);
            o0.y = ep::pack_bf16x2_rn(acc[2], acc[3]);
            o0.z = ep::pack_bf16x2_rn(acc[4], acc[5]);
            o0.w = ep::pack_bf16x2_rn(acc[6], acc[7]);
            o1.x = ep::pack_bf16x2_rn(acc[8], acc[9]);
            o1.y = ep::pack_bf16x2_rn(acc[10], acc[11]);
            o1.z = ep::pack_bf16x2_rn(acc[12], acc[13]);
            o1.w = ep::pack_bf16x2_rn(acc[14], acc[15]);
            uint4* dst = os + (static_cast<size_t>(t) * nvec + v) * 2;
            ep::st_v4(dst, o0);
            ep::st_v4(dst + 1, o1);
        }
        if (++g == ngroups) {
            g = 0;
            ++t;
        }
    }
}

// Combined top-k weights: a warp per token. Lanes read the token's slot row (lanes across
// ranks) and compact the receiving ranks in ascending order with a ballot; lane j then
// loads weight j of up to kBatch of those rows at once and adds them in rank order
// (fp32 from +0).
__global__ void __launch_bounds__(kThreads)
    combine_weights_kernel(const float* __restrict__ w, const int32_t* __restrict__ slot, int T, int k, int R,
                           int max_tokens, float* __restrict__ out, int32_t* status) {
    ep::grid_dependency_wait();
    __shared__ long long s_src[kWarps][kMaxSrc];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    for (int t = static_cast<int>(blockIdx.x) * kWarps + warp; t < T; t += static_cast<int>(gridDim.x) * kWarps) {
        int ns = 0;
        bool over_any = false;
        for (int r0 = 0; r0 < R; r0 += 32) {
            const int r = r0 + lane;
            const int s = r < R ? __ldg(slot + static_cast<size_t>(t) * R + r) : -1;
            const bool over = s >= max_tokens;
            over_any |= over;
            const bool ok = s >= 0 && !over;
            const uint32_t m = __ballot_sync(ep::kFullMask, ok);
            if (ok) s_src[warp][ns + __popc(m & ep::lanemask_lt())] = (static_cast<long long>(r) * max_tokens + s) * k;
            ns += __popc(m);
        }
        if (__any_sync(ep::kFullMask, over_any) && lane == 0) ep::raise_flag(status, EP_FLAG_CAPACITY);
        __syncwarp();
        float acc = 0.0f;
        for (int d0 = 0; d0 < ns; d0 += kBatch) {
            float v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (d0 + i < ns && lane < k) v[i] = __ldg(w + s_src[warp][d0 + i] + lane);
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (d0 + i < ns) acc = __fadd_rn(acc, v[i]);
        }
        if (lane < k) out[static_cast<size_t>(t) * k + lane] = acc;
        __syncwarp();
    }
}

std::atomic<int> g_fp8_blocks_per_sm[ep::kMaxDevices];
std::atomic<int> g_blocks_per_sm[ep::kMaxDevices];

}  // namespace

extern "C" ep_status_t ep_combine(const void* y, const int32_t* slot, int32_t T, int32_t H, int32_t R,
                                  int32_t max_tokens, void* out, int32_t* status, void* stream) {
    using namespace ep;
    if (T < 0 || H <= 0 || H % 8 != 0 || R < 1 || R > 256 || max_tokens < 0) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (slot == nullptr || out == nullptr || (max_tokens > 0 && y == nullptr)) return EP_ERR_INVALID;
    if (!aligned16_or_null(y) || !aligned16(slot) || !aligned16(out)) return EP_ERR_INVALID;
    int per_sm = 1;
    const ep_status_t occ = blocks_per_sm(g_blocks_per_sm, combine_kernel, kThreads, 0, &per_sm);
    if (occ != EP_OK) return occ;
    const long long items = static_cast<long long>(T) * ((H / 8 + 31) / 32);
    const long long want = (items + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    return launch_dependent(combine_kernel, dim3(grid), dim3(kThreads), 0, as_stream(stream),
                            static_cast<const uint16_t*>(y), slot, T, H, R, max_tokens, static_cast<uint16_t*>(out),
                            status);
}

extern "C" ep_status_t ep_combine_fp8(const uint8_t* y, const float* y_scales, const int32_t* slot, int32_t T,
                                      int32_t H, int32_t R, int32_t max_tokens, void* out, int32_t* status,
                                      void* stream) {
    using namespace ep;
    if (T < 0 || H <= 0 || H % 128 != 0 || R < 1 || R > 256 || max_tokens < 0) return EP_ERR_INVALID;
    if (static_cast<long long>(R) * max_tokens > 0x7fffffffLL) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (slot == nullptr || out == nullptr || (max_tokens > 0 && (y == nullptr || y_scales == nullptr)))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(y) || !aligned16_or_null(y_scales) || !aligned16(slot) || !aligned16(out))
        return EP_ERR_INVALID;
    int per_sm = 1;
    const ep_status_t occ = blocks_per_sm(g_fp8_blocks_per_sm, combine_fp8_kernel, kThreads, 0, &per_sm);
    if (occ != EP_OK) return occ;
    const long long items = static_cast<long long>(T) * ((H / 16 + 31) / 32);
    const long long want = (items + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    return launch_dependent(combine_fp8_kernel, dim3(grid), dim3(kThreads), 0, as_stream(stream), y, y_scales, slot,
                            T, H, R, max_tokens, static_cast<uint16_t*>(out), status);
}

extern "C" ep_status_t ep_combine_weights(const float* recv_topk_w, const int32_t* slot, int32_t T, int32_t k,
                                          int32_t R, int32_t max_tokens, float* combined_w, int32_t* status,
                                          void* stream) {
    using namespace ep;
    if (T < 0 || k < 1 || k > 32 || R < 1 || R > 256 || max_tokens < 0) return EP_ERR_INVALID;
    if (static_cast<long long>(R) * max_tokens > 0x7fffffffLL) return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    if (slot == nullptr || combined_w == nullptr || (max_tokens > 0 && recv_topk_w == nullptr))
        return EP_ERR_INVALID;
    if (!aligned16_or_null(recv_topk_w) || !aligned16(slot) || !aligned16(combined_w)) return EP_ERR_INVALID;
    const long long want = (static_cast<long long>(T) + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    return launch_dependent(combine_weights_kernel, dim3(grid), dim3(kThreads), 0, as_stream(stream), recv_topk_w,
                            slot, T, k, R, max_tokens, combined_w, status);
}
