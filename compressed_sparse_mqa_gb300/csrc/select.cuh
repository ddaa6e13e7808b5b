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

// ---- top-k from approximate scores with an exact band ---------------------------------------
// The approximate score s~ of a row differs from its exact score s by at most eps.
// Two 11-bit radix passes over the approximate keys bracket the k-th largest s~ in
// [T_lo, T_hi]; rows with s~ > T_hi + 2 eps + 4 ulp are kept for certain, rows with
// s~ < T_lo - 2 eps - 4 ulp dropped for certain, and only the rows in between (a
// handful) are rescored exactly (TwoSum over the exact fp16 products, rounded once
// to binary32) and ranked (higher score, then lower index).  The result is the
// exact top-k of the binary32-rounded exact scores.  If the band is ever larger
// than its buffer (many equal keys, say), every row is rescored exactly and an
// exact radix select runs instead.

constexpr int kBandCap = 1024;

template <int NT, int MAXROWS>
struct BandSmem {
    uint32_t hist[kMaxBins];
    uint32_t cnt[NT];
    uint32_t scan[NT / 32];
    int band_idx[kBandCap];
    uint32_t band_key[kBandCap];
    uint32_t sel_bits[MAXROWS / 32];
    uint32_t res[3], band_n, n_in;
    float eps;
};

DS4A_DEVINL float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// TwoSum-exact score key of one row, computed by a group of 16 threads (all 32 lanes
// of every warp call this; `valid` masks the rows).  kCoherent: the row is read
// through L2 (a row this kernel has just written), else through the read-only path.
template <bool kCoherent = false>
DS4A_DEVINL uint32_t exact_key16(const uint16_t *q, const uint16_t *krow, int d_idx, bool valid) {
    const int gl = threadIdx.x & 15;
    float s = 0.f, c = 0.f;
    for (int ch = gl; ch < d_idx / 8; ch += 16) {
        if (valid) {
            const uint4 qa = *reinterpret_cast<const uint4 *>(q + ch * 8);
            const uint4 ka = kCoherent ? __ldcg(reinterpret_cast<const uint4 *>(krow + ch * 8))
                                       : __ldg(reinterpret_cast<const uint4 *>(krow + ch * 8));
            const uint16_t *hq = reinterpret_cast<const uint16_t *>(&qa);
            const uint16_t *hk = reinterpret_cast<const uint16_t *>(&ka);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float err;
                two_sum(s, h2f(hq[e]) * h2f(hk[e]), s, err);
                c += err;
            }
        }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float err;
        two_sum(s, s2, s, err);
        c = (c + c2) + err;
    }
    return float_key(s + c);
}

// key[] holds the approximate keys (item `it` of thread t is row it * NT + t), n > k.
// q: the query (d_idx fp16), k_idx: [>= n, d_idx] fp16 key rows; spill: n u32 of
// scratch for the exact keys of the fallback.  Writes the kept rows, ascending, to out.
template <int NT, int ITEMS, int MAXROWS>
__device__ void band_select(uint32_t (&key)[ITEMS], int n, int k, float eps, const uint16_t *q,
                            const uint16_t *k_idx, int d_idx, BandSmem<NT, MAXROWS> &sm, uint32_t *spill,
                            int32_t *out) {
    static_assert(ITEMS * NT <= MAXROWS, "row bitmask covers every row");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // bracket the k-th largest approximate score: bits 31..21, then 20..10
    uint32_t kk = static_cast<uint32_t>(k);
    radix_pass<NT, ITEMS>(key, n, 0u, 0u, 21, 11, kk, sm.hist, sm.scan, sm.res);
    uint32_t prefix = sm.res[0] << 21, mask = 0xFFE00000u;
    kk -= sm.res[1];
    radix_pass<NT, ITEMS>(key, n, prefix, mask, 10, 11, kk, sm.hist, sm.scan, sm.res);
    prefix |= sm.res[0] << 10;
    const uint32_t lo_key = prefix, hi_key = prefix | 0x3FFu;
    const float t_lo = key_to_float(lo_key), t_hi = key_to_float(hi_key);
    const float big = fmaxf(fabsf(t_lo), fabsf(t_hi));
    const float ulp = ldexpf(1.f, ilogbf(big > 0.f ? big : 1.f) - 23);
    const float margin = 2.f * eps + 4.f * ulp;
    const float in_thr = t_hi + margin, out_thr = t_lo - margin;
    // the same two tests on the order-preserving keys: s > in_thr <=> key > key(in_thr) and
    // s >= out_thr <=> key >= key(out_thr), a zero threshold taken as +0 and -0 respectively
    // (-0 and +0 are equal scores but distinct keys)
    const uint32_t in_key = float_key(in_thr == 0.f ? 0.f : in_thr);
    const uint32_t out_key = float_key(out_thr == 0.f ? -0.f : out_thr);

    // classify: certainly in, certainly out, or band (rescored exactly)
    if (tid == 0) {
        sm.band_n = 0;
        sm.n_in = 0;
    }
    for (int w = tid; w < ITEMS * NT / 32; w += NT) sm.sel_bits[w] = 0;
    __syncthreads();
    uint32_t flags = 0, my_in = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * NT + tid;
        if (j < n) {
            if (key[it] > in_key) {
                flags |= 1u << it;
                ++my_in;
            } else if (key[it] >= out_key) {
                const uint32_t b = atomicAdd(&sm.band_n, 1u);
                if (b < kBandCap) sm.band_idx[b] = j;
            }
        }
    }
    my_in = __reduce_add_sync(0xffffffffu, my_in);
    if (lane == 0 && my_in) atomicAdd(&sm.n_in, my_in);
    __syncthreads();
    const uint32_t band_n = sm.band_n, n_in = sm.n_in;
    const bool fits = band_n <= kBandCap && n_in <= static_cast<uint32_t>(k) &&
                      n_in + band_n >= static_cast<uint32_t>(k);
    if (fits) {
        // exact keys of the band rows: 16 threads per row
        for (uint32_t b0 = 0; b0 < band_n; b0 += NT / 16) {
            const uint32_t b = b0 + tid / 16;
            const bool valid = b < band_n;
            const int j = valid ? sm.band_idx[b] : 0;
            const uint32_t kx = exact_key16(q, k_idx + static_cast<size_t>(j) * d_idx, d_idx, valid);
            if (valid && (tid & 15) == 0) sm.band_key[b] = kx;
        }
        __syncthreads();
        // keep the (k - n_in) best band rows: higher exact key, then lower index
        const uint32_t need = static_cast<uint32_t>(k) - n_in;
        for (uint32_t b = tid; b < band_n; b += NT) {
            const uint32_t kb = sm.band_key[b];
            const int jb = sm.band_idx[b];
            uint32_t rank = 0;
            for (uint32_t o = 0; o < band_n; ++o) {
                const uint32_t ko = sm.band_key[o];
                rank += (ko > kb) || (ko == kb && sm.band_idx[o] < jb);
            }
            if (rank < need) atomicOr(&sm.sel_bits[jb >> 5], 1u << (jb & 31));
        }
        // the certainly kept rows join the band's kept rows in the row bitmask
        // (a warp's ballot of one item is the word of its 32 consecutive rows)
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const unsigned b = __ballot_sync(0xffffffffu, (flags >> it) & 1u);
            if (lane == 0 && b) atomicOr(&sm.sel_bits[it * (NT / 32) + warp], b);
        }
        __syncthreads();
        emit_bits<NT, ITEMS>(sm.sel_bits, sm.scan, out);
        return;
    }

    // fallback: exact keys for every visible row, then an exact radix select
    for (int b0 = 0; b0 < ITEMS * NT; b0 += NT / 16) {
        const int j = b0 + tid / 16;
        const uint32_t kx = exact_key16(q, k_idx + static_cast<size_t>(j < n ? j : 0) * d_idx, d_idx, j < n);
        if (j < n && (tid & 15) == 0) spill[j] = kx;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * NT + tid;
        key[it] = j < n ? spill[j] : 0u;
    }
    const bool all_eq = find_threshold<NT, ITEMS>(key, n, k, sm.hist, sm.scan, sm.res, prefix, mask, kk);
    emit_topk_bits<NT, ITEMS>(key, n, prefix, mask, kk, all_eq, sm.cnt, sm.sel_bits, sm.scan, out);
}

}  // namespace sel
}  // namespace ds4a
