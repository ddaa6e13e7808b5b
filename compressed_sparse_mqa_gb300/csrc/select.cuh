// select.cuh -- block-wide pieces of the indexer's exact top-k select: a radix
// pass over order-preserving u32 keys held in registers, block scans, and the
// ascending-index emission of flagged rows.  Item `it` of thread t is row
// it * NT + t (coalesced loads, index order = (item, warp, lane)).
#pragma once

#include <stdint.h>

#include "ds4a_common.cuh"

namespace ds4a {
namespace sel {

constexpr int kMaxBins = 2048;   // 11-bit digits

// Exclusive scan of one value per thread across the block (NT threads).
template <int NT>
DS4A_DEVINL uint32_t block_excl_scan(uint32_t v, uint32_t *scratch /* NT/32 */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w)
        if (w < warp) before += scratch[w];
    return before + incl - v;
}

// One radix pass: among keys with (key & mask) == prefix, histogram the `bits`-bit
// digit at `shift` and find the digit holding the kk-th largest key.  Writes
// res[0] = digit, res[1] = keys in larger digits, res[2] = keys in the digit.
template <int NT, int ITEMS>
DS4A_DEVINL void radix_pass(const uint32_t (&key)[ITEMS], int n, uint32_t prefix, uint32_t mask, int shift,
                            int bits, uint32_t kk, uint32_t *hist, uint32_t *scratch, uint32_t *res) {
    const int tid = threadIdx.x;
    const int nb = 1 << bits;
    for (int b = tid; b < nb; b += NT) hist[b] = 0;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it)
        if (it * NT + tid < n && (key[it] & mask) == prefix) atomicAdd(&hist[(key[it] >> shift) & (nb - 1)], 1u);
    __syncthreads();
    const int per = nb / NT;   // bins per thread, largest first
    uint32_t lsum = 0;
    for (int e = 0; e < per; ++e) lsum += hist[nb - 1 - per * tid - e];
    const uint32_t before = block_excl_scan<NT>(lsum, scratch);
    if (before < kk && before + lsum >= kk) {
        uint32_t acc = before;
        for (int e = 0; e < per; ++e) {
            const uint32_t c = hist[nb - 1 - per * tid - e];
            if (acc + c >= kk) {
                res[0] = static_cast<uint32_t>(nb - 1 - per * tid - e);
                res[1] = acc;
                res[2] = c;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

// Exact k-th largest of n > k keys: up to three passes (11, 11, 10 bits),
// stopping once the boundary digit holds exactly the rows still needed.
// On return *prefix/*mask describe the boundary, *kk is the number of boundary
// rows still to keep, and the result is `true` when every boundary row is kept.
template <int NT, int ITEMS>
DS4A_DEVINL bool find_threshold(const uint32_t (&key)[ITEMS], int n, int k, uint32_t *hist, uint32_t *scratch,
                                uint32_t *res, uint32_t &prefix, uint32_t &mask, uint32_t &kk) {
    prefix = 0u;
    mask = 0u;
    kk = static_cast<uint32_t>(k);
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 3; ++p) {
        radix_pass<NT, ITEMS>(key, n, prefix, mask, shifts[p], widths[p], kk, hist, scratch, res);
        kk -= res[1];
        prefix |= res[0] << shifts[p];
        mask |= ((1u << widths[p]) - 1u) << shifts[p];
        if (res[2] == kk) return true;
    }
    return false;
}

// Write the rows whose flag bit is set, in ascending row order, to out[].
template <int NT, int ITEMS>
DS4A_DEVINL void emit(uint32_t flags, int32_t *out, uint32_t *cnt /* ITEMS*NT/32 <= NT */, uint32_t *scratch) {
    static_assert(ITEMS * (NT / 32) <= NT, "one count per thread");
    constexpr int kW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const unsigned b = __ballot_sync(0xffffffffu, (flags >> it) & 1u);
        if (lane == 0) cnt[it * kW + warp] = __popc(b);
    }
    __syncthreads();
    const uint32_t v = cnt[tid < ITEMS * kW ? tid : 0];
    const uint32_t ex = block_excl_scan<NT>(tid < ITEMS * kW ? v : 0u, scratch);
    if (tid < ITEMS * kW) cnt[tid] = ex;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const unsigned b = __ballot_sync(0xffffffffu, (flags >> it) & 1u);
        if ((flags >> it) & 1u) out[cnt[it * kW + warp] + __popc(b & lt)] = it * NT + threadIdx.x;
    }
}

// Flags of the exact top-k given the boundary: rows above it, and boundary rows
// in ascending index order up to kk of them (all of them when `all_eq`).
template <int NT, int ITEMS>
DS4A_DEVINL uint32_t topk_flags(const uint32_t (&key)[ITEMS], int n, uint32_t prefix, uint32_t mask, uint32_t kk,
                                bool all_eq, uint32_t *cnt, uint32_t *scratch) {
    constexpr int kW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        if (it * NT + tid < n) {
            const uint32_t km = key[it] & mask;
            gt |= static_cast<uint32_t>(km > prefix) << it;
            eq |= static_cast<uint32_t>(km == prefix) << it;
        }
    }
    if (all_eq) return gt | eq;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const unsigned b = __ballot_sync(0xffffffffu, (eq >> it) & 1u);
        if (lane == 0) cnt[it * kW + warp] = __popc(b);
    }
    __syncthreads();
    const uint32_t v = cnt[tid < ITEMS * kW ? tid : 0];
    const uint32_t ex = block_excl_scan<NT>(tid < ITEMS * kW ? v : 0u, scratch);
    if (tid < ITEMS * kW) cnt[tid] = ex;
    __syncthreads();
    uint32_t take = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const unsigned b = __ballot_sync(0xffffffffu, (eq >> it) & 1u);
        if (((eq >> it) & 1u) && cnt[it * kW + warp] + __popc(b & lt) < kk) take |= 1u << it;
    }
    __syncthreads();   // cnt is reused by emit
    return gt | take;
}

// Flags of the exact top-k, written out in ascending row order, for keys in the
// item-major layout: a warp's ballot of one item is the bit word of 32 consecutive
// rows, so the "above the boundary" and "on the boundary" rows become two bitmasks
// in shared memory; thread t then takes rows t*ITEMS .. t*ITEMS + ITEMS-1 of them
// (row order = thread order), ranks its boundary rows and its kept rows with one
// block scan each, and writes its kept rows.  gt_bits, eq_bits: ITEMS*NT/32 words.
template <int NT, int ITEMS>
DS4A_DEVINL void emit_topk_bits(const uint32_t (&key)[ITEMS], int n, uint32_t prefix, uint32_t mask, uint32_t kk,
                                bool all_eq, uint32_t *gt_bits, uint32_t *eq_bits, uint32_t *scratch,
                                int32_t *out) {
    static_assert(ITEMS <= 32 && 32 % ITEMS == 0, "a thread's rows lie in one bit word");
    constexpr int kW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const bool valid = it * NT + tid < n;
        const uint32_t km = key[it] & mask;
        const unsigned g = __ballot_sync(0xffffffffu, valid && km > prefix);
        const unsigned e = __ballot_sync(0xffffffffu, valid && km == prefix);
        if (lane == 0) {
            gt_bits[it * kW + warp] = g;
            eq_bits[it * kW + warp] = e;
        }
    }
    __syncthreads();
    const int w = tid * ITEMS / 32, sh = tid * ITEMS % 32;
    const uint32_t seg = ITEMS == 32 ? 0xFFFFFFFFu : ((1u << (ITEMS & 31)) - 1u);
    const uint32_t g = (gt_bits[w] >> sh) & seg;
    uint32_t e = (eq_bits[w] >> sh) & seg;
    if (!all_eq) {
        const uint32_t before = block_excl_scan<NT>(static_cast<uint32_t>(__popc(e)), scratch);
        // keep the first kk - before boundary rows of this thread (lowest rows first)
        const int keep = before >= kk ? 0 : static_cast<int>(min(static_cast<uint32_t>(__popc(e)), kk - before));
        uint32_t t = e, kept = 0;
        for (int j = 0; j < keep; ++j) {
            const uint32_t low = t & (0u - t);
            kept |= low;
            t ^= low;
        }
        e = kept;
    }
    uint32_t sel_bits = g | e;
    uint32_t pos = block_excl_scan<NT>(static_cast<uint32_t>(__popc(sel_bits)), scratch);
    while (sel_bits) {
        const int b = __ffs(sel_bits) - 1;
        out[pos++] = tid * ITEMS + b;
        sel_bits &= sel_bits - 1u;
    }
}

// Rows whose bit is set in `bits` (row r is bit r%32 of word r/32), in ascending
// order, to out[]: thread t takes rows t*ITEMS .. t*ITEMS + ITEMS-1 and one block
// scan places them.
template <int NT, int ITEMS>
DS4A_DEVINL void emit_bits(const uint32_t *bits, uint32_t *scratch, int32_t *out) {
    static_assert(ITEMS <= 32 && 32 % ITEMS == 0, "a thread's rows lie in one bit word");
    const int tid = threadIdx.x;
    const uint32_t seg = ITEMS == 32 ? 0xFFFFFFFFu : ((1u << (ITEMS & 31)) - 1u);
    uint32_t m = (bits[tid * ITEMS / 32] >> (tid * ITEMS % 32)) & seg;
    uint32_t pos = block_excl_scan<NT>(static_cast<uint32_t>(__popc(m)), scratch);
    while (m) {
        out[pos++] = tid * ITEMS + __ffs(m) - 1;
        m &= m - 1u;
    }
}

}  // namespace sel
}  // namespace ds4a
