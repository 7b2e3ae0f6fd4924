// ep_dispatch.cu -- rank-level dispatch: every token goes once to every rank it
// routes to, into that rank's slab of the destination-major receive buffers
// ("[PR #347] Feature/sm free normal kernel", 2.1 Feature; workload of 3.1;
// FP8 and BF16 dispatch of 3.2.1), with the optional per-token 1x128 E4M3
// quantisation fused into the copy.
//
// bf16 rows move with bulk asynchronous copies (the shared scatter of ep_scatter.cuh); the
// register kernel described next serves rows too large for its shared-memory buffers
// and, with the quantisation added, the FP8 path.
//
// Register design: a persistent grid of warps, one token per warp at a time. The warp
// reads the token's slot row once (lanes across ranks) and compacts the
// destinations (ascending rank) into shared memory with a ballot; then it
// streams the hidden row through registers in 16-byte vectors, 8 per lane
// (4 KB per warp) in flight, reading each vector once from HBM and storing it
// to every destination slab. Metadata
// (source index, local expert ids, weights) is written by one lane per
// destination. Nothing here is a contraction, so no tensor cores: the kernel
// is bound by HBM bandwidth (read T rows, write one row per (token, rank)).
#include <algorithm>

#include "ep_common.cuh"
#include "ep_scatter.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDest = 256;  // = largest R: a slot row may name every rank
constexpr int kMaxTopk = 32;
constexpr int kUnroll = 8;     // 16-byte vectors in flight per lane (bf16 path)
constexpr int kRegDest = 8;    // destinations whose row offsets a warp keeps in registers
constexpr int kUnrollFp8 = 2;  // warp iterations (4 blocks of 128 each) in flight (FP8 path)
constexpr uint32_t kFp8BulkMaxSmem = 52 * 1024;  // shared memory of the bulk FP8 kernel (4 CTAs per SM)
constexpr int kFp8Stages = 3;  // staging rows of the bulk FP8 kernel
// roles of the bulk FP8 kernel's warps: 0-5 quantise, 6 writes scale rows, 7 lists tokens
constexpr int kQuantWarps = 6;
constexpr int kScaleWarp = 6;
constexpr int kListWarp = 7;

struct DispatchArgs {
    const uint16_t* x;
    const int64_t* topk_idx;
    const float* topk_w;
    const int32_t* slot;
    int T, H, k, E, R, epr, max_tokens;
    void* recv_x;
    float* recv_scales;
    int32_t* recv_src_idx;
    int32_t* recv_topk_idx;
    float* recv_topk_w;
    int32_t* status;
};

// Destinations of token t: compacted (ascending rank) into s_rank / s_row.
// Returns their number; drops slots >= max_tokens (EP_FLAG_CAPACITY).
__device__ __forceinline__ int gather_destinations(const DispatchArgs& a, int t, int* s_rank, long long* s_row) {
    const int lane = ep::lane_id();
    int nd = 0;
    bool over_any = false;
    for (int r0 = 0; r0 < a.R; r0 += 32) {
        const int r = r0 + lane;
        const int s = r < a.R ? a.slot[static_cast<size_t>(t) * a.R + r] : -1;
        const bool over = s >= a.max_tokens;
        over_any |= over;
        const bool ok = s >= 0 && !over;
        const uint32_t m = __ballot_sync(ep::kFullMask, ok);
        if (ok) {
            const int pos = nd + __popc(m & ep::lanemask_lt());
            s_rank[pos] = r;
            s_row[pos] = static_cast<long long>(r) * a.max_tokens + s;
        }
        nd += __popc(m);
    }
    if (over_any) ep::raise_flag(a.status, EP_FLAG_CAPACITY);
    __syncwarp();
    return nd;
}

__device__ __forceinline__ void write_metadata(const DispatchArgs& a, int t, int nd, const int* s_rank,
                                               const long long* s_row) {
    const int lane = ep::lane_id();
    if (lane == 0) {
        bool bad = false;
        for (int j = 0; j < a.k; ++j) bad |= a.topk_idx[static_cast<size_t>(t) * a.k + j] >= a.E;
        if (bad) ep::raise_flag(a.status, EP_FLAG_BAD_EXPERT);
    }
    const int64_t* ids = a.topk_idx + static_cast<size_t>(t) * a.k;
    for (int d = lane; d < nd; d += 32) {
        const int r = s_rank[d];
        const size_t row = static_cast<size_t>(s_row[d]);
        if (a.recv_src_idx != nullptr) a.recv_src_idx[row] = t;
        for (int j = 0; j < a.k; ++j) {
            const int64_t e = ids[j];
            const bool on = e >= 0 && e < a.E && static_cast<int>(e) / a.epr == r;
            if (a.recv_topk_idx != nullptr)
                a.recv_topk_idx[row * a.k + j] = on ? static_cast<int32_t>(e) - r * a.epr : -1;
            if (a.recv_topk_w != nullptr)
                a.recv_topk_w[row * a.k + j] = on ? a.topk_w[static_cast<size_t>(t) * a.k + j] : 0.0f;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) dispatch_bf16_kernel(DispatchArgs a) {
    ep::grid_dependency_wait();  // dependent launch: inputs are ready after this
    __shared__ int s_rank[kWarps][kMaxDest];
    __shared__ long long s_row[kWarps][kMaxDest];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nvec = a.H / 8;  // 16-byte vectors per row
    uint4* recv = static_cast<uint4*>(a.recv_x);

    for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
        const int nd = gather_destinations(a, t, s_rank[warp], s_row[warp]);
        write_metadata(a, t, nd, s_rank[warp], s_row[warp]);
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H);
        // the first kRegDest destination rows stay in registers for the whole row
        uint32_t row_of[kRegDest];  // R * max_tokens < 2^31 is checked on the host
#pragma unroll
        for (int d = 0; d < kRegDest; ++d) row_of[d] = d < nd ? static_cast<uint32_t>(s_row[warp][d]) : 0u;
        for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
            uint4 buf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) buf[u] = ep::ld_stream_v4(src + v);
            }
#pragma unroll
            for (int d = 0; d < kRegDest; ++d) {
                if (d < nd) {
                    uint4* dst = recv + static_cast<size_t>(row_of[d]) * nvec;
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int v = v0 + u * 32 + lane;
                        if (v < nvec) ep::st_v4(dst + v, buf[u]);
                    }
                }
            }
            for (int d = kRegDest; d < nd; ++d) {
                uint4* dst = recv + static_cast<size_t>(s_row[warp][d]) * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < nvec) ep::st_v4(dst + v, buf[u]);
                }
            }
        }
        __syncwarp();
    }
}

// x / scale correctly rounded to fp32, for a normal scale. The quotient is the product by
// the correctly rounded reciprocal, corrected once by its residual (Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34,
// 1990): with rcp = RN(1/scale) and q0 = RN(x * rcp) within an ulp of x / scale, the
// residual x - q0 * scale is exact in one fused multiply-add and q0 + rcp * residual,
// rounded once, is RN(x / scale). Quotients that fall below the fp32 normal range only
// ever round to an E4M3 zero, whose sign is the sign of x; the correction turns a zero x
// into +0, so x's sign bit is put back (for every other x it is already there).
__device__ __forceinline__ float quotient(float x, float scale, float rcp) {
    const float q0 = __fmul_rn(x, rcp);
    const float e = __fmaf_rn(-q0, scale, x);
    const float q1 = __fmaf_rn(e, rcp, q0);
    return __uint_as_float(__float_as_uint(q1) | (__float_as_uint(x) & 0x80000000u));
}

// amax / 448 correctly rounded: the same correction with RN(1/448), valid while the
// quotient is a normal fp32 (amax >= 2^-116); smaller amax take the IEEE division
__device__ __forceinline__ float scale_of(float amax) {
    constexpr float kInv448 = 1.0f / 448.0f;  // correctly rounded at compile time
    if (amax < 0x1p-116f) return __fdiv_rn(amax, 448.0f);
    const float q0 = __fmul_rn(amax, kInv448);
    return __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), kInv448, q0);
}

// bf16 dispatch through the shared bulk-copy scatter (ep_scatter.cuh): source row t is
// x[t], its destinations are the compacted slot row, the side work is the metadata.
struct DispatchScatter {
    DispatchArgs a;
    char* dst;
    uint32_t row_bytes;
    int32_t* status;
    __device__ int items() const { return a.T; }
    __device__ const void* source(int t) const { return a.x + static_cast<size_t>(t) * a.H; }
    __device__ int destinations(int t, long long* rows, int* aux) const {
        return gather_destinations(a, t, aux, rows);
    }
    __device__ void side_work(int t, int nd, const long long* rows, const int* aux) const {
        write_metadata(a, t, nd, aux, rows);
    }
    __device__ void prologue() const {}
};

// One 128-element block is held by 8 lanes, 16 bf16 (two 16-byte vectors) per
// lane. Returns the lane's 16 E4M3 codes as one 16-byte vector (element i in
// byte i) and the block's scale (the same in all 8 lanes).
__device__ __forceinline__ void quantize16(const uint4& a, const uint4& b, uint4& q, float& scale) {
    float f[16];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = ep::bf16_lo(w[i]);
        f[2 * i + 1] = ep::bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    // max over the 8 lanes of this block (xor offsets < 8 stay in the group)
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(ep::kFullMask, amax, off));
    scale = scale_of(amax);
    if (amax == 0.0f) {
        // all elements are +-0: keep the sign of each zero
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = (__float_as_uint(f[4 * i]) >> 31) << 7 | (__float_as_uint(f[4 * i + 1]) >> 31) << 15 |
                   (__float_as_uint(f[4 * i + 2]) >> 31) << 23 | (__float_as_uint(f[4 * i + 3]) >> 31) << 31;
        q = make_uint4(c[0], c[1], c[2], c[3]);
    } else if (scale >= 1.17549435e-38f) {  // 1/scale is finite: the corrected product
        const float rcp = __frcp_rn(scale);
        q.x = ep::pack_e4m3x4_rn_sat(quotient(f[0], scale, rcp), quotient(f[1], scale, rcp),
                                     quotient(f[2], scale, rcp), quotient(f[3], scale, rcp));
        q.y = ep::pack_e4m3x4_rn_sat(quotient(f[4], scale, rcp), quotient(f[5], scale, rcp),
                                     quotient(f[6], scale, rcp), quotient(f[7], scale, rcp));
        q.z = ep::pack_e4m3x4_rn_sat(quotient(f[8], scale, rcp), quotient(f[9], scale, rcp),
                                     quotient(f[10], scale, rcp), quotient(f[11], scale, rcp));
        q.w = ep::pack_e4m3x4_rn_sat(quotient(f[12], scale, rcp), quotient(f[13], scale, rcp),
                                     quotient(f[14], scale, rcp), quotient(f[15], scale, rcp));
    } else {
        q.x = ep::pack_e4m3x4_rn_sat(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale), __fdiv_rn(f[2], scale),
                                     __fdiv_rn(f[3], scale));
        q.y = ep::pack_e4m3x4_rn_sat(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale), __fdiv_rn(f[6], scale),
                                     __fdiv_rn(f[7], scale));
        q.z = ep::pack_e4m3x4_rn_sat(__fdiv_rn(f[8], scale), __fdiv_rn(f[9], scale), __fdiv_rn(f[10], scale),
                                     __fdiv_rn(f[11], scale));
        q.w = ep::pack_e4m3x4_rn_sat(__fdiv_rn(f[12], scale), __fdiv_rn(f[13], scale), __fdiv_rn(f[14], scale),
                                     __fdiv_rn(f[15], scale));
    }
}

// FP8 dispatch: a warp iteration covers 4 blocks (512 elements); lane l owns elements
// 16*(l % 8) .. +15 of block l / 8, so every code store is one 16-byte vector per lane
// (512 bytes per warp instruction). The block scales of a token (up to kScaleRow blocks,
// H <= 32768) are gathered in shared memory and each destination's scale row is written
// once per token, 16 bytes per lane when the row is 16-byte aligned -- instead of one
// single-lane 16-byte store per destination and iteration, which made half of all store
// instructions.
constexpr int kScaleRow = 256;

__global__ void __launch_bounds__(kThreads) dispatch_fp8_kernel(DispatchArgs a, int interleave) {
    ep::grid_dependency_wait();  // dependent launch: inputs are ready after this
    __shared__ int s_rank[kWarps][kMaxDest];
    __shared__ long long s_row[kWarps][kMaxDest];
    __shared__ __align__(16) float s_sc[kWarps][kScaleRow];
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int nblk = a.H / 128;
    const int grp = lane >> 3;  // block of the iteration this lane works on (0..3)
    const int pos = lane & 7;   // 16-element slice within the block
    const bool row_scales = nblk <= kScaleRow;
    uint8_t* recv = static_cast<uint8_t*>(a.recv_x);

    // one wave: token c + G*w goes to warp w of CTA c, so every SM gets the same number of
    // tokens; several waves: consecutive tokens per CTA and the hardware balances CTAs
    for (int t = interleave ? static_cast<int>(blockIdx.x + gridDim.x * warp) : static_cast<int>(blockIdx.x) * kWarps + warp;
         t < a.T; t += gridDim.x * kWarps) {
        const int nd = gather_destinations(a, t, s_rank[warp], s_row[warp]);
        write_metadata(a, t, nd, s_rank[warp], s_row[warp]);
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H);
        for (int b0 = 0; b0 < nblk; b0 += 4 * kUnrollFp8) {
            uint4 lo[kUnrollFp8], hi[kUnrollFp8];
#pragma unroll
            for (int u = 0; u < kUnrollFp8; ++u) {
                const int b = b0 + 4 * u + grp;
                if (b < nblk) {
                    lo[u] = ep::ld_stream_v4(src + b * 16 + 2 * pos);
                    hi[u] = ep::ld_stream_v4(src + b * 16 + 2 * pos + 1);
                } else {
                    lo[u] = make_uint4(0, 0, 0, 0);
                    hi[u] = lo[u];
                }
            }
            uint4 q[kUnrollFp8];
            float sc[kUnrollFp8];
#pragma unroll
            for (int u = 0; u < kUnrollFp8; ++u) {
                quantize16(lo[u], hi[u], q[u], sc[u]);
                const int b = b0 + 4 * u + grp;
                if (row_scales && pos == 0 && b < nblk) s_sc[warp][b] = sc[u];
            }
            for (int d = 0; d < nd; ++d) {
                const size_t row = static_cast<size_t>(s_row[warp][d]);
                uint8_t* dst = recv + row * a.H;
#pragma unroll
                for (int u = 0; u < kUnrollFp8; ++u) {
                    const int b = b0 + 4 * u + grp;
                    if (b < nblk) {
                        ep::st_v4(dst + b * 128 + pos * 16, q[u]);
                        if (!row_scales && pos == 0) a.recv_scales[row * nblk + b] = sc[u];
                    }
                }
            }
        }
        if (row_scales) {  // the token's scale row to every destination
            __syncwarp();
            const bool vec = (nblk & 3) == 0;
            for (int d = 0; d < nd; ++d) {
                float* dsc = a.recv_scales + static_cast<size_t>(s_row[warp][d]) * nblk;
                if (vec) {
                    for (int i = lane; i < nblk / 4; i += 32)
                        ep::st_v4(dsc + 4 * i, *reinterpret_cast<const uint4*>(&s_sc[warp][4 * i]));
                } else {
                    for (int i = lane; i < nblk; i += 32) dsc[i] = s_sc[warp][i];
                }
            }
        }
        __syncwarp();
    }
}

// FP8 dispatch through shared memory and bulk copies: a CTA of 8 warps takes one token at a
// time (tokens blockIdx.x, +gridDim.x, ...). Every thread copies its 16-byte pieces of the
// tokens' bf16 rows into two shared-memory row buffers by asynchronous copies, two tokens
// ahead (these go through the load path, so they do not queue behind the CTA's bulk
// stores). The warps have roles: warps 0-5 quantise the row from shared memory -- 8 lanes
// per 128-element block, the quantiser of the register kernel -- into a staging code row (H
// bytes) and scale row (H/128 floats); meanwhile warp 7 resolves the next token's
// destinations and writes its metadata rows (from the slot row, ids and weights it loaded
// into registers a token earlier) and warp 6 writes the previous token's scale rows with
// 16-byte stores. After the CTA barrier thread 0 sends the code row to every destination
// with one bulk shared->global copy. The staging rows form a ring of three and the
// destination lists one of three (tokens i - 1, i, i + 1), so the stores of two tokens drain
// while the next is quantised. No code passes through a store from registers. All waits
// are hardware waits on the CTA's own copies (no spinning). Used when H % 512 == 0 (scale
// rows of whole 16-byte vectors) and the buffers fit.
struct Fp8Smem {
    uint32_t row_bytes, code_bytes, scale_bytes;
    uint32_t row_stride;    // row buffer b at b * row_stride
    uint32_t stage_base;    // staging buffer s at stage_base + s * stage_stride: codes, then scales
    uint32_t stage_stride;
    uint32_t scale_off;     // scales within a staging buffer
    uint32_t total;
};

inline Fp8Smem fp8_smem_layout(int H) {
    auto up = [](uint32_t n) { return (n + 127u) & ~127u; };
    Fp8Smem m{};
    m.row_bytes = static_cast<uint32_t>(H) * 2u;
    m.code_bytes = static_cast<uint32_t>(H);
    m.scale_bytes = static_cast<uint32_t>(H / 128) * 4u;
    m.row_stride = up(m.row_bytes);
    m.stage_base = 2u * m.row_stride;
    m.scale_off = up(m.code_bytes);
    m.stage_stride = m.scale_off + up(m.scale_bytes);
    m.total = m.stage_base + kFp8Stages * m.stage_stride;
    return m;
}

__global__ void __launch_bounds__(kThreads, 4) dispatch_fp8_bulk_kernel(DispatchArgs a, Fp8Smem m) {
    extern __shared__ __align__(128) unsigned char smem[];
    // destination lists of three tokens (i - 1: its scale rows; i: quantised, its code rows;
    // i + 1: being listed): row index r * max_tokens + slot (below 2^31) and rank
    __shared__ int s_row[3][kMaxDest];
    __shared__ uint8_t s_rank[3][kMaxDest];
    __shared__ int s_nd[3];
    ep::grid_dependency_wait();  // dependent launch: inputs are ready after this
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nblk = a.H / 128;
    const int grp = lane >> 3;
    const int pos = lane & 7;
    const int first = static_cast<int>(blockIdx.x);
    const int step = static_cast<int>(gridDim.x);
    const int n_my = first < a.T ? (a.T - 1 - first) / step + 1 : 0;
    uint8_t* recv = static_cast<uint8_t*>(a.recv_x);
    // row loads: every thread copies its 16-byte pieces of the token's bf16 row into row
    // buffer q & 1, one commit group per token (empty past the last), two tokens ahead
    const int nvec = a.H / 8;
    auto load_row = [&](int q) {
        if (q < n_my) {
            const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(first + q * step) * a.H);
            uint4* dst = reinterpret_cast<uint4*>(smem + (q & 1) * m.row_stride);
            for (int v = tid; v < nvec; v += kThreads) ep::cp_async16(dst + v, src + v);
        }
        ep::cp_async_commit();
    };
    auto stage_of = [&](int q) { return smem + m.stage_base + (q % kFp8Stages) * m.stage_stride; };

    // the listing warp holds a token's slot row (lane r + 32c), top-k ids and weights (lane j)
    // in registers, loaded a token before it lists that token
    int sv[kMaxDest / 32];
    long long idv = -1;
    float wv = 0.0f;
    auto fetch_meta = [&](int t) {
#pragma unroll
        for (int c = 0; c < kMaxDest / 32; ++c) {
            const int r = c * 32 + lane;
            sv[c] = (c * 32 < a.R && r < a.R) ? a.slot[static_cast<size_t>(t) * a.R + r] : -1;
        }
        idv = lane < a.k ? a.topk_idx[static_cast<size_t>(t) * a.k + lane] : -1;
        wv = (lane < a.k && a.recv_topk_w != nullptr) ? a.topk_w[static_cast<size_t>(t) * a.k + lane] : 0.0f;
    };
    // list token t's destinations (ascending rank; slots >= max_tokens dropped) into list
    // set `ls` and write its metadata rows (lane j: slot j of every destination)
    auto list_token = [&](int t, int ls) {
        int nd = 0;
        bool over_any = false;
#pragma unroll
        for (int c = 0; c < kMaxDest / 32; ++c) {
            if (c * 32 >= a.R) break;
            const int r = c * 32 + lane;
            const int sl = sv[c];
            const bool over = sl >= a.max_tokens;
            over_any |= over;
            const bool ok = r < a.R && sl >= 0 && !over;
            const uint32_t msk = __ballot_sync(ep::kFullMask, ok);
            if (ok) {
                const int p = nd + __popc(msk & ep::lanemask_lt());
                s_rank[ls][p] = static_cast<uint8_t>(r);
                s_row[ls][p] = r * a.max_tokens + sl;
            }
            nd += __popc(msk);
        }
        if (__any_sync(ep::kFullMask, over_any) && lane == 0) ep::raise_flag(a.status, EP_FLAG_CAPACITY);
        if (__any_sync(ep::kFullMask, idv >= a.E) && lane == 0) ep::raise_flag(a.status, EP_FLAG_BAD_EXPERT);
        __syncwarp();
        for (int d = 0; d < nd; ++d) {
            const int r = s_rank[ls][d];
            const size_t row = static_cast<size_t>(s_row[ls][d]);
            if (lane == 0 && a.recv_src_idx != nullptr) a.recv_src_idx[row] = t;
            if (lane < a.k) {
                const bool on = idv >= 0 && idv < a.E && static_cast<int>(idv) / a.epr == r;
                if (a.recv_topk_idx != nullptr)
                    a.recv_topk_idx[row * a.k + lane] = on ? static_cast<int32_t>(idv) - r * a.epr : -1;
                if (a.recv_topk_w != nullptr) a.recv_topk_w[row * a.k + lane] = on ? wv : 0.0f;
            }
        }
        if (lane == 0) s_nd[ls] = nd;
    };
    // token q's scale rows: 16 bytes per lane, one store instruction per destination
    auto store_scales = [&](int q) {
        const int ls = q % 3;
        const float* scales = reinterpret_cast<const float*>(stage_of(q) + m.scale_off);
        for (int d = 0; d < s_nd[ls]; ++d) {
            float* dsc = a.recv_scales + static_cast<size_t>(s_row[ls][d]) * nblk;
            for (int v = lane; v < nblk / 4; v += 32)
                ep::st_v4(dsc + 4 * v, *reinterpret_cast<const uint4*>(scales + 4 * v));
        }
    };

    load_row(0);
    load_row(1);
    if (warp == kListWarp && n_my > 0) {
        fetch_meta(first);
        list_token(first, 0);
        if (n_my > 1) fetch_meta(first + step);
    }
    for (int i = 0; i < n_my; ++i) {
        const int t = first + i * step;
        const int ls = i % 3;
        ep::cp_async_wait<1>();  // this thread's pieces of token i's row have landed
        __syncthreads();     // ... everyone's, token i listed, its staging buffer free
        const int nd = s_nd[ls];
        uint8_t* codes = stage_of(i);
        if (warp < kQuantWarps) {
            if (nd > 0) {
                // a warp's 4 blocks are all in range or all out of it (nblk % 4 == 0), so the
                // quantiser's shuffles always run on whole warps
                const uint16_t* row = reinterpret_cast<const uint16_t*>(smem + (i & 1) * m.row_stride);
                float* scales = reinterpret_cast<float*>(codes + m.scale_off);
                for (int blk = warp * 4 + grp; blk < nblk; blk += kQuantWarps * 4) {
                    const uint4* src = reinterpret_cast<const uint4*>(row + blk * 128 + pos * 16);
                    uint4 q;
                    float sc;
                    quantize16(src[0], src[1], q, sc);
                    *reinterpret_cast<uint4*>(codes + blk * 128 + pos * 16) = q;
                    if (pos == 0) scales[blk] = sc;
                }
                ep::fence_proxy_async_smem();
            }
        } else if (warp == kScaleWarp) {
            if (i > 0) store_scales(i - 1);
        } else if (i + 1 < n_my) {  // the listing warp: the next token
            list_token(t + step, (i + 1) % 3);
            if (i + 2 < n_my) fetch_meta(t + 2 * step);
        }
        __syncthreads();  // token i quantised, token i + 1 listed
        load_row(i + 2);  // row buffer i & 1 is free
        if (tid == 0) {
            for (int d = 0; d < nd; ++d)
                ep::bulk_store(recv + static_cast<size_t>(s_row[ls][d]) * a.H, codes, m.code_bytes);
            ep::bulk_commit();
            // token i + 1 goes into the staging buffer of token i + 1 - kFp8Stages: all but
            // the newest kFp8Stages - 1 bulk groups (one per token) must have read theirs
            ep::bulk_wait_read<kFp8Stages - 1>();
        }
    }
    if (warp == kScaleWarp && n_my > 0) store_scales(n_my - 1);
    ep::allow_dependents();
    if (tid == 0) ep::bulk_wait_all();
}

std::atomic<int> g_fp8_bulk_smem_set[ep::kMaxDevices];

std::atomic<int> g_fp8_per_sm[ep::kMaxDevices];

int grid_for(int T, int blocks_per_sm) {
    const int want = (T + kWarps - 1) / kWarps;
    const int cap = ep::sm_count() * blocks_per_sm;
    return want < 1 ? 1 : (want < cap ? want : cap);
}

}  // namespace

extern "C" ep_status_t ep_dispatch(const void* x, ep_dtype_t out_dtype, const int64_t* topk_idx,
                                   const float* topk_w, const int32_t* slot, int32_t T, int32_t H, int32_t k,
                                   int32_t E, int32_t R, int32_t max_tokens, void* recv_x, float* recv_scales,
                                   int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_w,
                                   int32_t* status, void* stream) {
    using namespace ep;
    const bool fp8 = out_dtype == EP_DTYPE_E4M3;
    if (out_dtype != EP_DTYPE_BF16 && !fp8) return EP_ERR_INVALID;
    if (T < 0 || H <= 0 || H % 8 != 0 || (fp8 && H % 128 != 0) || k < 1 || k > kMaxTopk || R < 1 ||
        R > 256 || E < R || E % R != 0 || max_tokens < 0)
        return EP_ERR_INVALID;
    if (static_cast<long long>(R) * max_tokens > 0x7fffffffLL) return EP_ERR_INVALID;
    if (recv_x == nullptr || (fp8 && recv_scales == nullptr) || (!fp8 && recv_scales != nullptr))
        return EP_ERR_INVALID;
    if (T > 0 && (x == nullptr || topk_idx == nullptr || slot == nullptr)) return EP_ERR_INVALID;
    if (recv_topk_w != nullptr && T > 0 && topk_w == nullptr) return EP_ERR_INVALID;
    if (!aligned16_or_null(x) || !aligned16_or_null(topk_idx) || !aligned16_or_null(topk_w) ||
        !aligned16_or_null(slot) || !aligned16(recv_x) || !aligned16_or_null(recv_scales) ||
        !aligned16_or_null(recv_src_idx) || !aligned16_or_null(recv_topk_idx) || !aligned16_or_null(recv_topk_w))
        return EP_ERR_INVALID;
    if (T == 0) return EP_OK;
    DispatchArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.slot = slot;
    a.T = T;
    a.H = H;
    a.k = k;
    a.E = E;
    a.R = R;
    a.epr = E / R;
    a.max_tokens = max_tokens;
    a.recv_x = recv_x;
    a.recv_scales = recv_scales;
    a.recv_src_idx = recv_src_idx;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_w = recv_topk_w;
    a.status = status;
    if (fp8) {
        const Fp8Smem m = fp8_smem_layout(H);
        if (H % 512 == 0 && m.total <= kFp8BulkMaxSmem) {
            const ep_status_t attr =
                ensure_dynamic_smem(g_fp8_bulk_smem_set, dispatch_fp8_bulk_kernel, static_cast<int>(kFp8BulkMaxSmem));
            if (attr != EP_OK) return attr;
            const long long grid = std::min<long long>(T, static_cast<long long>(sm_count()) * 4);
            return launch_dependent(dispatch_fp8_bulk_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads),
                                    static_cast<size_t>(m.total), as_stream(stream), a, m);
        }
        int per_sm = 1;
        const ep_status_t occ = blocks_per_sm(g_fp8_per_sm, dispatch_fp8_kernel, kThreads, 0, &per_sm);
        if (occ != EP_OK) return occ;
        const long long resident = static_cast<long long>(sm_count()) * per_sm;
        const bool one_wave = static_cast<long long>(T) <= resident * kWarps;
        const int grid = one_wave ? static_cast<int>(resident) : grid_for(T, 8);
        return launch_dependent(dispatch_fp8_kernel, dim3(grid), dim3(kThreads), 0, as_stream(stream), a,
                                one_wave ? 1 : 0);
    }
    const DispatchScatter sp{a, static_cast<char*>(recv_x), static_cast<uint32_t>(H) * 2u, status};
    const ep_status_t st = launch_scatter_rows(sp, T, as_stream(stream));
    if (st != EP_ERR_INVALID) return st;  // rows too large for the shared-memory buffers: registers
    return launch_dependent(dispatch_bf16_kernel, dim3(grid_for(T, 8)), dim3(kThreads), 0, as_stream(stream), a);
}
