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
constexpr int kUnitSrc = 8;  // FP8 combine: sources per unit of its two-stage shared-memory ring
static_assert(kUnitSrc == 8, "the FP8 combine's unit is written out for 8 sources (32 lanes = 8 x 4 scales)");
constexpr int kFp8CombineBlocks = 3;  // FP8 combine CTAs per SM (shared memory: ~67 KB per CTA)

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
// [R][max_tokens][H/128]). Items are (token, 32 lanes x 16 channels), taken by the warps in
// runs of two strided over the batch (combine_fp8_kernel below). A warp walks its items in
// units of up to kUnitSrc sources of one item and keeps two units in a shared-memory ring:
// while it computes one, the next one's codes (16 per lane, one 16-byte vector) and block
// scales are on their way by per-lane asynchronous copies, so the loads in flight occupy no
// registers. Per source a lane converts its 16 codes to fp32 exactly (E4M3 -> fp16 -> fp32
// through 16-bit register halves) and adds RN(code * scale) to its accumulators in source
// order, two channels per instruction with both roundings kept (ep::pair_add_product, with
// the -0 it needs passed in as a kernel argument).
// The first term is taken as fma(code, scale, +0) = RN(code * scale + 0), one instruction
// instead of two. It equals 0 + RN(code * scale) unless a nonzero product rounds to zero
// (the fused form would keep a -0): with |code| >= 2^-9 that needs a scale below 2^-140,
// so such scales (never produced by real data) take the two-instruction form.
// zero: +0 for the first term's fused form, -0 for every later product
template <bool kFirst>
__device__ __forceinline__ void fp8_term16(float* acc, const uint4& v, float sc, float zero) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float f[4];
        ep::e4m3x4_to_f32(w[q], f[0], f[1], f[2], f[3]);
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            if (kFirst) ep::pair_fma(acc[4 * q + i], acc[4 * q + i + 1], f[i], f[i + 1], sc, zero);
            else ep::pair_add_product(acc[4 * q + i], acc[4 * q + i + 1], f[i], f[i + 1], sc, zero);
        }
    }
}

__device__ __forceinline__ bool fused_first_ok(float sc) { return sc == 0.0f || sc >= 0x1p-140f; }

// Per-lane asynchronous copies, issued only where `p` holds (a predicate, not a branch).
// one unit of the FP8 combine: up to kUnitSrc sources of item (t, lane vector v)
struct Fp8Unit {
    int t, v, n;
    bool first, last;  // first unit of its item (accumulators start), last (the row is written)
};

// Shared memory of one warp: two stages of kUnitSrc sources (32 lanes x 16 codes, and the
// 4 block scales of the item), then the item's source list (R rounded up to kUnitSrc).
struct Fp8CombineSmem {
    static constexpr int kStageCodes = kUnitSrc * 32;  // uint4 per stage
    static constexpr int kStageScales = kUnitSrc * 4;   // floats per stage
    static __host__ __device__ int list_len(int R) { return (R + kUnitSrc - 1) / kUnitSrc * kUnitSrc; }
    static __host__ __device__ size_t warp_bytes(int R) {
        return 2 * (kStageCodes * 16 + kStageScales * 4) + static_cast<size_t>(list_len(R)) * 4;
    }
};

// Warps take items in runs of two neighbours strided across the whole batch (warp w of
// the grid: items 2w, 2w + 1, then 2w + 2W, 2w + 2W + 1, ... for W warps), so every warp
// sees a sample of many tokens and the warps' work stays even although tokens differ in
// their number of sources, while the two items of a run mostly share a token and its
// source list. A list is built from the token's slot row, whose first 64 entries were
// loaded one item ahead.
__global__ void __launch_bounds__(kThreads, kFp8CombineBlocks)
    combine_fp8_kernel(const uint8_t* __restrict__ y, const float* __restrict__ y_scales,
                       const int32_t* __restrict__ slot, int T, int H, int R, int max_tokens,
                       uint16_t* __restrict__ out, int32_t* status, float pz, float nz) {
    ep::grid_dependency_wait();  // dependent launch: the slabs are complete after this
    extern __shared__ __align__(16) unsigned char s_dyn[];
    using L = Fp8CombineSmem;
    const int lane = ep::lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    unsigned char* wbase = s_dyn + static_cast<size_t>(warp) * L::warp_bytes(R);
    uint4* s_code = reinterpret_cast<uint4*>(wbase);                              // [2][kUnitSrc][32]
    float* s_scale = reinterpret_cast<float*>(wbase + 2 * L::kStageCodes * 16);  // [2][kUnitSrc][4]
    int* list = reinterpret_cast<int*>(wbase + 2 * (L::kStageCodes * 16 + L::kStageScales * 4));
    const int nvec = H / 16;  // 16-code vectors per row
    const int nblk = H / 128;
    const int ngroups = (nvec + 31) / 32;
    const long long items = static_cast<long long>(T) * ngroups;
    const long long W2 = static_cast<long long>(gridDim.x) * kWarps * 2;  // the run stride
    long long pit = (static_cast<long long>(blockIdx.x) * kWarps + warp) * 2;  // the issuing side's item
    if (pit >= items) return;
    // the step from a run's second item to the next run's first, as (tokens, groups)
    const int jt = static_cast<int>((W2 - 1) / ngroups);
    const int jg = static_cast<int>((W2 - 1) - static_cast<long long>(jt) * ngroups);
    // the item after (t, g), which is item `it` of a run: its token, group, index
    auto step = [&](long long it, int t, int g, int& t2, int& g2) -> long long {
        const bool second = (it & 1) != 0;
        t2 = t + (second ? jt : 0);
        g2 = g + (second ? jg : 1);
        if (g2 >= ngroups) {
            g2 -= ngroups;
            ++t2;
        }
        return it + (second ? W2 - 1 : 1);
    };
    const uint4* ys = reinterpret_cast<const uint4*>(y);
    uint4* os = reinterpret_cast<uint4*>(out);

    // slot entries of ranks lane and lane + 32 of the next item's token, loaded ahead
    int pre0 = -1, pre1 = -1;
    auto fetch = [&](int t) {
        const size_t row = static_cast<size_t>(t) * R;
        pre0 = lane < R ? __ldg(slot + row + lane) : -1;
        pre1 = lane + 32 < R ? __ldg(slot + row + lane + 32) : -1;
    };
    // the token's sources in ascending rank order, from the entries fetched for it; one
    // report of a dropped slot per token, from the warp that lists it for its group 0
    auto build = [&](int t, bool report) {
        int ns = 0;
        bool over_any = false;
        __syncwarp();
        for (int r0 = 0; r0 < R; r0 += 32) {
            const int r = r0 + lane;
            const int s = r0 == 0 ? pre0 : r0 == 32 ? pre1 : (r < R ? __ldg(slot + static_cast<size_t>(t) * R + r) : -1);
            const bool over = s >= max_tokens;
            over_any |= over;
            const bool ok = s >= 0 && !over;
            const uint32_t m = __ballot_sync(ep::kFullMask, ok);
            if (ok) list[ns + __popc(m & ep::lanemask_lt())] = r * max_tokens + s;
            ns += __popc(m);
        }
        if (__any_sync(ep::kFullMask, over_any) && lane == 0 && report) ep::raise_flag(status, EP_FLAG_CAPACITY);
        __syncwarp();
        return ns;
    };

    // issuing side: item pit = (pt, pg), next source pc (a multiple of kUnitSrc) of pns;
    // (nt, ng) is the item after it, whose token's slot entries are loaded ahead
    int pt = static_cast<int>(pit / ngroups);
    int pg = static_cast<int>(pit - static_cast<long long>(pt) * ngroups);
    int pc = 0;
    fetch(pt);
    int pns = build(pt, pg == 0);
    int nt, ng;
    long long nit = step(pit, pt, pg, nt, ng);
    if (nit < items && nt != pt) fetch(nt);
    auto produce = [&](int st, Fp8Unit& u) {
        const int v = pg * 32 + lane;
        const int n = min(kUnitSrc, pns - pc);
        u.t = pt;
        u.v = v;
        u.n = n;
        u.first = pc == 0;
        u.last = pc + n >= pns;
        // lane 4j + b copies the scale of the item's block b of source j
        const int sj = lane >> 2, sb = pg * 4 + (lane & 3);
        const unsigned srow = static_cast<unsigned>(list[pc + sj]);  // stale past n: never used
        ep::cp_async4_if(s_scale + st * L::kStageScales + lane, y_scales + static_cast<size_t>(srow) * nblk + sb,
                     sj < n && sb < nblk);
        if (v < nvec) {
            int rows[kUnitSrc];
#pragma unroll
            for (int i = 0; i < kUnitSrc; i += 4) {
                const int4 r4 = *reinterpret_cast<const int4*>(list + pc + i);
                rows[i] = r4.x;
                rows[i + 1] = r4.y;
                rows[i + 2] = r4.z;
                rows[i + 3] = r4.w;
            }
            const uint4* src = ys + v;
            uint4* dst = s_code + st * L::kStageCodes + lane;
#pragma unroll
            for (int i = 0; i < kUnitSrc; ++i) {
                // entries past n are stale list words: their addresses are formed, never used
                ep::cp_async16_if(dst + i * 32, src + static_cast<size_t>(static_cast<unsigned>(rows[i])) * nvec, i < n);
            }
        }
        ep::cp_async_commit();
        pc += n;
        if (u.last) {
            pc = 0;
            const int prev_t = pt;
            pit = nit;
            pt = nt;
            pg = ng;
            if (pit < items) {
                if (pt != prev_t) pns = build(pt, pg == 0);
                nit = step(pit, pt, pg, nt, ng);
                if (nit < items && nt != pt) fetch(nt);
            }
        }
    };

    float acc[16];
    auto consume = [&](int st, const Fp8Unit& u) {
        if (u.v >= nvec) return;
        const uint4* cs = s_code + st * L::kStageCodes + lane;
        const float* ss = s_scale + st * L::kStageScales + (lane >> 3);
        if (u.first) {
            const float sc0 = u.n > 0 ? ss[0] : 0.0f;
            if (u.n > 0 && fused_first_ok(sc0)) {
                fp8_term16<true>(acc, cs[0], sc0, pz);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
                if (u.n > 0) fp8_term16<false>(acc, cs[0], sc0, nz);
            }
        } else {
            fp8_term16<false>(acc, cs[0], ss[0], nz);  // a later unit holds at least one source
        }
        // sources 1 .. n-1 in order; one exit for all counts keeps the branches cheap
        if (u.n <= 1) goto done;
        fp8_term16<false>(acc, cs[1 * 32], ss[1 * 4], nz);
        if (u.n <= 2) goto done;
        fp8_term16<false>(acc, cs[2 * 32], ss[2 * 4], nz);
        if (u.n <= 3) goto done;
        fp8_term16<false>(acc, cs[3 * 32], ss[3 * 4], nz);
        if (u.n <= 4) goto done;
        fp8_term16<false>(acc, cs[4 * 32], ss[4 * 4], nz);
        if (u.n <= 5) goto done;
        fp8_term16<false>(acc, cs[5 * 32], ss[5 * 4], nz);
        if (u.n <= 6) goto done;
        fp8_term16<false>(acc, cs[6 * 32], ss[6 * 4], nz);
        if (u.n <= 7) goto done;
        fp8_term16<false>(acc, cs[7 * 32], ss[7 * 4], nz);
    done:
        if (u.last) {
            uint4 o0, o1;
            o0.x = ep::pack_bf16x2_rn(acc[0], acc[1]);
            o0.y = ep::pack_bf16x2_rn(acc[2], acc[3]);
            o0.z = ep::pack_bf16x2_rn(acc[4], acc[5]);
            o0.w = ep::pack_bf16x2_rn(acc[6], acc[7]);
            o1.x = ep::pack_bf16x2_rn(acc[8], acc[9]);
            o1.y = ep::pack_bf16x2_rn(acc[10], acc[11]);
            o1.z = ep::pack_bf16x2_rn(acc[12], acc[13]);
            o1.w = ep::pack_bf16x2_rn(acc[14], acc[15]);
            uint4* dst = os + (static_cast<size_t>(u.t) * nvec + u.v) * 2;
            ep::st_v4(dst, o0);
            ep::st_v4(dst + 1, o1);
        }
    };

    // two-stage ring: unit k + 1 is in flight while unit k is computed. The scales of a
    // stage are copied by one lane per block and read by eight, so a stage is refilled only
    // after a warp barrier that follows its reads, and read only after one that follows the
    // copies' completion.
    Fp8Unit cur, nxt;
    int st = 0;
    produce(0, cur);
    for (;;) {
        const bool more = pit < items;
        if (more) produce(st ^ 1, nxt);
        else ep::cp_async_commit();  // an empty group keeps the wait below uniform
        ep::cp_async_wait<1>();
        __syncwarp();
        consume(st, cur);
        if (!more) break;
        __syncwarp();
        cur = nxt;
        st ^= 1;
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

std::atomic<int> g_fp8_smem_set[ep::kMaxDevices];
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
    const size_t smem = static_cast<size_t>(kWarps) * Fp8CombineSmem::warp_bytes(R);
    ep_status_t st = ensure_dynamic_smem(g_fp8_smem_set, combine_fp8_kernel,
                                         static_cast<int>(kWarps * Fp8CombineSmem::warp_bytes(256)));
    if (st != EP_OK) return st;
    const long long items = static_cast<long long>(T) * ((H / 16 + 31) / 32);
    const long long want = (items + kWarps - 1) / kWarps;
    const long long cap = static_cast<long long>(sm_count()) * kFp8CombineBlocks;
    const int grid = static_cast<int>(want < cap ? want : cap);
    return launch_dependent(combine_fp8_kernel, dim3(grid), dim3(kThreads), smem, as_stream(stream), y, y_scales, slot,
                            T, H, R, max_tokens, static_cast<uint16_t*>(out), status, 0.0f, -0.0f);
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
