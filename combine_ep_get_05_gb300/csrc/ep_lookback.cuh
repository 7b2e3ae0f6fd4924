// ep_lookback.cuh -- the decoupled look-back shared by the two layout scans (the rank
// slots of ep_layout.cu and the expert slots of ep_permute.cu). Internal header.
//
// Tile i of a scan publishes, per column (a rank or an expert), one 64-bit word
// {epoch: 32 bits, state: 2 bits, value: 30 bits}; state 1 = the tile's own count,
// state 2 = the inclusive prefix over tiles 0..i. The epoch tags the call, so words
// left in the workspace by earlier calls never pass for current ones. A tile finds
// its exclusive prefix by reading its predecessors' words, newest first, a batch at a
// time, adding counts until it meets an inclusive prefix; a word not yet published is
// polled, and the poll gives up after kWaitLimitNs (or kWaitLimitIters polls).
#pragma once

#include "ep_common.cuh"

namespace ep {

constexpr uint32_t kStateAggregate = 1u;
constexpr uint32_t kStatePrefix = 2u;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr uint32_t kWaitLimitIters = 1u << 24;               // hard cap on polls

__device__ __forceinline__ unsigned long long pack_word(uint32_t epoch, uint32_t state, uint32_t v) {
    return (static_cast<unsigned long long>(epoch) << 32) | (static_cast<unsigned long long>(state) << 30) |
           static_cast<unsigned long long>(v & 0x3fffffffu);
}
__device__ __forceinline__ uint32_t word_epoch(unsigned long long w) { return static_cast<uint32_t>(w >> 32); }
__device__ __forceinline__ uint32_t word_state(unsigned long long w) { return static_cast<uint32_t>(w >> 30) & 3u; }
__device__ __forceinline__ uint32_t word_value(unsigned long long w) { return static_cast<uint32_t>(w) & 0x3fffffffu; }

// Polls a tile word until it carries this call's epoch and a published state; returns
// it, or 0 (no valid word has epoch 0) once the wait has run out. Kept out of line: it
// runs only when a word is not ready yet.
static __device__ __noinline__ unsigned long long wait_word(const unsigned long long* p, uint32_t epoch) {
    const unsigned long long start = globaltimer_ns();
    for (uint32_t polls = 1; polls < kWaitLimitIters; ++polls) {
        if (polls > 16) __nanosleep(256);
        const unsigned long long w = ld_relaxed_u64(p);
        if (word_epoch(w) == epoch && word_state(w) != 0u) return w;
        if (globaltimer_ns() - start > kWaitLimitNs) break;
    }
    return 0ull;
}

// Exclusive prefix of column `col` for tile `tile`: the sum of the counts of tiles
// 0 .. tile-1, from the words words[i * stride + col] (kBatch predecessors requested at
// once). Sets timed_out (and returns a partial sum) when a wait gives up.
template <int kBatch>
__device__ __forceinline__ uint32_t lookback_exclusive(const unsigned long long* words, size_t stride, int tile,
                                                       int col, uint32_t epoch, bool& timed_out) {
    uint32_t excl = 0;
    int j = tile - 1;
    while (j >= 0 && !timed_out) {
        const int nb = j + 1 < kBatch ? j + 1 : kBatch;
        unsigned long long wv[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (i < nb) wv[i] = ld_relaxed_u64(words + static_cast<size_t>(j - i) * stride + col);
        bool found_prefix = false;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (i >= nb || found_prefix || timed_out) continue;
            unsigned long long w = wv[i];
            if (word_epoch(w) != epoch || word_state(w) == 0u) {
                w = wait_word(words + static_cast<size_t>(j - i) * stride + col, epoch);
                if (w == 0ull) {
                    timed_out = true;
                    continue;
                }
            }
            excl += word_value(w);
            if (word_state(w) == kStatePrefix) found_prefix = true;
        }
        if (found_prefix) break;
        j -= nb;
    }
    return excl;
}

}  // namespace ep
