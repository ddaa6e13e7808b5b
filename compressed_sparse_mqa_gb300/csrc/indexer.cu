// indexer.cu -- the learned indexer: score every visible compressed row for a
// query and keep the k highest (top-512 on the model's ratio-4 layers).
//
// "DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": even layers
// from 2 use a learned indexer that selects the top-512 compressed rows.
//
// Scores.  score_j = q . kidx_j.  Each fp16 x fp16 product is exact in binary32;
// the products are summed with Knuth's TwoSum (an error-free transformation),
// so the running pair (s, c) carries the exact sum to within ~2^-46 relative and
// fl(s + c) is the binary32 rounding of the exact score.  The ranking decision
// is therefore taken on the correctly rounded binary32 score.
//
// Select.  Scores map to order-preserving u32 keys held in registers (8, 16 or
// 32 per thread; larger row counts re-read them from memory).  A radix select
// over 11-bit digits with one shared histogram per pass (plain shared atomics)
// finds the k-th largest key, stopping early once the boundary digit holds
// exactly the rows still needed.  Rows above the boundary, then
// boundary rows in ascending index order, are written in ascending index order
// using warp ballots and one scan over (item, warp) counts.
//
// Decode (one query): CTAs of 64 rows each load their key rows before waiting on
// the previous kernel (the keys are cache state, not produced by it), score
// them into the workspace, and the last CTA to finish (atomic ticket, no
// waiting) selects and resets the ticket.  Many queries: the tensor-core path
// (indexer_tc.cu) when the shapes allow it, else one CTA per query scores its
// visible rows into shared memory and selects.
#include <type_traits>

#include "compress_dev.cuh"
#include "ds4a_common.cuh"
#include "ds4a_internal.h"
#include "select.cuh"

namespace ds4a {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 16;                        // threads per scored row
constexpr int kRowsPerPass = kThreads / kGroup;   // 32
constexpr int kRowsPerCta = 2 * kRowsPerPass;     // decode slice: 64 rows
constexpr int kStagedRows = 1024;                 // decode: rows per CTA scored before the dependency wait
constexpr int kMaxDIdx = 256;
constexpr int kMaxItems = 32;                     // register select: n <= 512 * 32
constexpr size_t kWsHeader = 256;                 // ticket lives here
constexpr int kSmemKeyCap = 16384;                // prefill: keys staged in shared memory

struct SelectSmem {
    uint32_t hist[sel::kMaxBins];
    uint32_t cnt[kMaxItems * kWarps];
    uint32_t eq_bits[kMaxItems * kWarps];
    uint32_t scan[kWarps];
    uint32_t res[3];
    uint32_t bin;
    uint32_t above;
    uint32_t count_bin;
};

// ---- scoring ---------------------------------------------------------------------------

struct RowLoads {
    uint4 v[2][2];   // [row pass][chunk]
};

DS4A_DEVINL void load_rows(const uint16_t *__restrict__ kidx, int d_idx, long long base, long long j1,
                           RowLoads &L) {
    const int tid = threadIdx.x, gl = tid % kGroup;
    const int n_chunks = d_idx / 8;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const long long j = base + p * kRowsPerPass + tid / kGroup;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int ch = gl + cc * kGroup;
            L.v[p][cc] = (j < j1 && ch < n_chunks)
                             ? __ldg(reinterpret_cast<const uint4 *>(kidx + j * d_idx + ch * 8))
                             : make_uint4(0, 0, 0, 0);
        }
    }
}

DS4A_DEVINL void load_query(const uint16_t *__restrict__ q, int d_idx, float (&qf)[2][8]) {
    const int gl = threadIdx.x % kGroup;
    const int n_chunks = d_idx / 8;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int ch = gl + cc * kGroup;
        if (ch < n_chunks) {
            uint4 raw = *reinterpret_cast<const uint4 *>(q + ch * 8);
            const uint16_t *h = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[cc][e] = h2f(h[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[cc][e] = 0.f;
        }
    }
}

// Scores of the (up to) 64 rows base .. base+63 held in L; keys[j - base] for j < j1.
// Every lane of every warp reaches the shuffles (the loop bounds are block-uniform).
DS4A_DEVINL void score_loaded(const float (&qf)[2][8], const RowLoads &L, long long base, long long j1,
                              uint32_t *keys) {
    const int tid = threadIdx.x, gl = tid % kGroup;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float s = 0.f, c = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const uint16_t *h = reinterpret_cast<const uint16_t *>(&L.v[p][cc]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float err;
                two_sum(s, qf[cc][e] * h2f(h[e]), s, err);
                c += err;
            }
        }
#pragma unroll
        for (int o = kGroup / 2; o > 0; o >>= 1) {
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
            float err;
            two_sum(s, s2, s, err);
            c = (c + c2) + err;
        }
        const long long j = base + p * kRowsPerPass + tid / kGroup;
        if (j < j1 && gl == 0) keys[j - base] = float_key(s + c);
    }
}

// Approximate scores (fp32 FMA, error far below sel::band_select's eps) of the rows held in
// L, as order-preserving keys, and the largest sum_c |q_c k_c| among them (bmax).
DS4A_DEVINL void score_loaded_approx(const float (&qf)[2][8], const RowLoads &L, long long base, long long j1,
                                     uint32_t *keys, float &bmax) {
    const int tid = threadIdx.x, gl = tid % kGroup;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float s = 0.f, m = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const uint16_t *h = reinterpret_cast<const uint16_t *>(&L.v[p][cc]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float kv = h2f(h[e]);
                s = fmaf(qf[cc][e], kv, s);
                m = fmaf(fabsf(qf[cc][e]), fabsf(kv), m);
            }
        }
#pragma unroll
        for (int o = kGroup / 2; o > 0; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            m += __shfl_xor_sync(0xffffffffu, m, o);
        }
        const long long j = base + p * kRowsPerPass + tid / kGroup;
        if (j < j1) {
            bmax = fmaxf(bmax, m);
            if (gl == 0) keys[j - base] = float_key(s);
        }
    }
}

// ---- select ------------------------------------------------------------------------------

// Block-wide exclusive scan of one value per thread (kThreads threads).
DS4A_DEVINL uint32_t block_excl_scan(uint32_t v, uint32_t *scratch, uint32_t &total) {
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
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = scratch[w];
        if (w < warp) before += t;
        all += t;
    }
    total = all;
    return before + incl - v;
}

// Histogram increment (b = 256 adds nothing).  Plain shared atomics: cheaper
// here than aggregating equal digits across the warp first.
DS4A_DEVINL void hist_add(uint32_t *hist, uint32_t b) {
    if (b < 256u) atomicAdd(&hist[b], 1u);
}

// Warp 0: the digit (scanning from the largest) that holds the kk-th largest key.
DS4A_DEVINL void find_bin(SelectSmem &sm, uint32_t kk) {
    if ((threadIdx.x >> 5) != 0) return;
    const int lane = threadIdx.x & 31;
    uint32_t cnt[8], lsum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) { cnt[e] = sm.hist[255 - 8 * lane - e]; lsum += cnt[e]; }
    uint32_t incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= kk);
    if (lane == __ffs(hit) - 1) {
        uint32_t before = incl - lsum;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (before + cnt[e] >= kk) {
                sm.bin = 255 - 8 * lane - e;
                sm.above = before;
                sm.count_bin = cnt[e];
                break;
            }
            before += cnt[e];
        }
    }
}

template <bool GLOBAL>
DS4A_DEVINL uint32_t ld_key(const uint32_t *src, int i) {
    if constexpr (GLOBAL) return __ldcg(src + i);
    else return src[i];
}

// Keys in registers: item `it` of thread t is index it * kThreads + t.  n > k.
template <int ITEMS, bool GLOBAL>
__device__ void select_regs(const uint32_t *src, int n, int k, int32_t *out, SelectSmem &sm) {
    const int tid = threadIdx.x;
    uint32_t key[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int i = it * kThreads + tid;
        key[it] = i < n ? ld_key<GLOBAL>(src, i) : 0u;
    }
    uint32_t prefix, mask, kk;
    const bool all_eq = sel::find_threshold<kThreads, ITEMS>(key, n, k, sm.hist, sm.scan, sm.res, prefix, mask, kk);
    sel::emit_topk_bits<kThreads, ITEMS>(key, n, prefix, mask, kk, all_eq, sm.cnt, sm.eq_bits, sm.scan, out);
}

// Any n > k: keys re-read from memory each pass; thread t emits the contiguous range [t*C, t*C + C).
template <bool GLOBAL>
__device__ void select_generic(const uint32_t *src, int n, int k, int32_t *out, SelectSmem &sm) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, mask = 0, kk = static_cast<uint32_t>(k);
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) sm.hist[tid] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            uint32_t b = 256u;
            if (i < n) {
                const uint32_t key = ld_key<GLOBAL>(src, i);
                if ((key & mask) == prefix) b = (key >> shift) & 255u;
            }
            hist_add(sm.hist, b);
        }
        __syncthreads();
        find_bin(sm, kk);
        __syncthreads();
        kk -= sm.above;
        prefix |= sm.bin << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    const int C = (n + kThreads - 1) / kThreads;
    const int lo = tid * C, hi = min(n, lo + C);
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = ld_key<GLOBAL>(src, i);
        n_gt += key > prefix;
        n_eq += key == prefix;
    }
    uint32_t tot;
    const uint32_t eq_before = block_excl_scan(n_eq, sm.scan, tot);
    const uint32_t take = eq_before >= kk ? 0u : min(n_eq, kk - eq_before);
    uint32_t p = block_excl_scan(n_gt + take, sm.scan, tot), taken = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = ld_key<GLOBAL>(src, i);
        if (key > prefix) out[p++] = i;
        else if (key == prefix && taken < take) { out[p++] = i; ++taken; }
    }
}

// Keep the k largest of src[0..n) (ties to the lower index): ascending indices in
// out[0..min(k,n)), -1 after; out_n (if given) = min(k, n).
template <bool GLOBAL>
__device__ void select_topk(const uint32_t *src, int n, int k, int32_t *out, int32_t *out_n, SelectSmem &sm) {
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
    } else if (n <= kThreads * 8) {
        select_regs<8, GLOBAL>(src, n, k, out, sm);
    } else if (n <= kThreads * 16) {
        select_regs<16, GLOBAL>(src, n, k, out, sm);
    } else if (n <= kThreads * kMaxItems) {
        select_regs<kMaxItems, GLOBAL>(src, n, k, out, sm);
    } else {
        select_generic<GLOBAL>(src, n, k, out, sm);
    }
    if (out_n && threadIdx.x == 0) *out_n = n < k ? n : k;
}

// select_topk with the register-select size fixed at compile time (kItems 8, 16 or 32
// keys a thread, for n <= 512 kItems), or the run-time choice (kItems 0): a decode
// launch whose row count the host knows carries only the select it needs.
template <int kItems>
__device__ void select_topk_sized(const uint32_t *src, int n, int k, int32_t *out, int32_t *out_n, SelectSmem &sm) {
    if constexpr (kItems == 0) {
        select_topk<true>(src, n, k, out, out_n, sm);
    } else {
        if (n <= k) {
            for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        } else {
            select_regs<kItems, true>(src, n, k, out, sm);
        }
        if (out_n && threadIdx.x == 0) *out_n = n < k ? n : k;
    }
}

// ---- kernels -----------------------------------------------------------------------------

struct IndexerArgs {
    const uint16_t *q_idx;
    const uint16_t *k_idx;
    int32_t *out_idx;
    int32_t *out_n;
    unsigned char *ws;
    long long n_rows;
    long long q_pos0;
    int n_q;
    int d_idx;
    int ratio;
    int k;
};

// Approximate keys of n > k rows (the workspace) -> the exact top-k through sel::band_select.
template <int ITEMS, typename Band>
__device__ void band_select_regs(const IndexerArgs &a, uint32_t *keys, int n, float eps, Band &band) {
    uint32_t key[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int i = it * kThreads + threadIdx.x;
        key[it] = i < n ? __ldcg(keys + i) : 0u;
    }
    sel::band_select<kThreads, ITEMS>(key, n, a.k, eps, a.q_idx, a.k_idx, a.d_idx, band, keys, a.out_idx);
}

DS4A_DEVINL long long visible_rows(const IndexerArgs &a, int i) {
    const long long v = (a.q_pos0 + i + 1) / a.ratio;
    return v < a.n_rows ? v : a.n_rows;
}

// The compressor's update for the one new token of a decode step (n_new = 1): its
// score reads only the caller's inputs and is taken before the wait; the running
// state and the pooled row of a completed block are written after it.
DS4A_DEVINL void compress_one_token(const cmp::CompressArgs &c, float *s_w, float *s_red) {
    const long long b = c.pos / c.ratio;
    const bool resume = c.pos % c.ratio != 0;   // the token continues an open block
    cmp::segment_scores<kThreads>(c, c.pos, c.pos + 1, s_w);
    pdl_wait();
    pdl_trigger();
    cmp::pool_segment<kThreads>(c, b, c.pos, c.pos + 1, resume, s_w, s_red);
}

// one cache line of global memory into L2 (no data returned, no alignment needed)
DS4A_DEVINL void prefetch_l2_line(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// Rows [lo, hi) of a slice scored into keys[j - kbase], kDeep 64-row batches per
// round: the loads of a round are all issued before any of them is scored, so a
// CTA that covers many rows (a batched step) keeps kDeep x 16 KB of key rows in
// flight.  A single decode query spreads its rows at 64 per CTA and takes kDeep = 1:
// the deeper round measured 0.8 us slower there.  kApprox: fp32 FMA scores (about a
// quarter of the TwoSum arithmetic) for sel::band_select, which rescores the rows
// near the k-th exactly; bmax collects the largest sum_c |q_c k_c| for its bound.
template <int kDeep, bool kApprox>
DS4A_DEVINL void score_rows(const IndexerArgs &a, const float (&qf)[2][8], long long lo, long long hi,
                           uint32_t *keys, long long kbase, float &bmax) {
    for (long long base = lo; base < hi; base += kDeep * kRowsPerCta) {
        RowLoads L[kDeep];
#pragma unroll
        for (int u = 0; u < kDeep; ++u) load_rows(a.k_idx, a.d_idx, base + u * kRowsPerCta, hi, L[u]);
#pragma unroll
        for (int u = 0; u < kDeep; ++u) {
            const long long bu = base + u * kRowsPerCta;
            if (bu < hi) {   // block-uniform
                if constexpr (kApprox) score_loaded_approx(qf, L[u], bu, hi, keys + (bu - kbase), bmax);
                else score_loaded(qf, L[u], bu, hi, keys + (bu - kbase));
            }
        }
    }
}

// Approximate scores of rows [lo, hi) into keys[j - lo], the key rows staged through
// shared memory with 16-byte cp.async and scored on the tensor cores: mma.sync
// m16n8k16 with a 16-row group as A and the query as column 0 of B, fp32 accumulation
// over the exact fp16 products.  A second product of the absolute values gives each
// row's sum_c |q_c k_c|; bmax collects the largest, and 2^-12 bmax bounds the error of
// every score (far above the accumulation error of d_idx <= 128 products, each rounded
// once).  Each of kScoreWarps warps runs its own pipeline over the groups
// warp, warp + kScoreWarps, ... (kWarpStages groups of 16 rows staged, two in flight
// while it scores the third) and writes its rows' keys itself: no block-wide barrier
// until the end.  Needs d_idx a multiple of 16, <= 128.  stage: kStageBytes bytes.
constexpr int kScoreWarps = 14;
constexpr int kWarpStages = 3;
constexpr int kGroupBytes = 16 * 256;   // 16 rows of up to 128 fp16
constexpr size_t kStageBytes = static_cast<size_t>(kScoreWarps) * kWarpStages * kGroupBytes;
static_assert(kScoreWarps <= kWarps, "scoring warps");
// the approximate path keeps the keys of up to this many rows per CTA in dynamic shared
// memory before the dependency wait (after the stages)
constexpr int kApproxStagedRows = 8192;
constexpr size_t kApproxDynBytes = kStageBytes + kApproxStagedRows * sizeof(uint32_t);
DS4A_DEVINL void score_rows_staged(const IndexerArgs &a, long long lo, long long hi, uint32_t *keys, float &bmax,
                                   unsigned char *stage) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp < kScoreWarps) {
        const int n_chunks = a.d_idx / 8;   // 16-byte chunks of a row
        const int ksteps = a.d_idx / 16;    // 16-wide k-steps
        // B fragments: the query in column 0 (lanes 0-3 of each k-step), zeros elsewhere
        uint32_t bq0[8], bq1[8], ba0[8], ba1[8];   // the query and its absolute values
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            bq0[s] = bq1[s] = ba0[s] = ba1[s] = 0u;
            if (s < ksteps && lane < 4) {
                const int k0 = s * 16 + 2 * lane;
                bq0[s] = *reinterpret_cast<const uint32_t *>(a.q_idx + k0);
                bq1[s] = *reinterpret_cast<const uint32_t *>(a.q_idx + k0 + 8);
                const __half2 x0 = __habs2(*reinterpret_cast<const __half2 *>(&bq0[s]));
                const __half2 x1 = __habs2(*reinterpret_cast<const __half2 *>(&bq1[s]));
                ba0[s] = *reinterpret_cast<const uint32_t *>(&x0);
                ba1[s] = *reinterpret_cast<const uint32_t *>(&x1);
            }
        }
        const long long n = hi - lo;
        const int n_groups = static_cast<int>((n + 15) / 16);
        const int my_groups = n_groups > warp ? (n_groups - warp + kScoreWarps - 1) / kScoreWarps : 0;
        unsigned char *mine = stage + static_cast<size_t>(warp) * kWarpStages * kGroupBytes;
        // chunk ch of row r sits at r * 256 + ((ch ^ (r & 7)) << 4): ldmatrix reads of 8
        // rows at one chunk column hit 8 different 16-byte bank groups
        auto issue = [&](int i) {   // this warp's i-th group
            if (i < my_groups) {
                const long long g0 = lo + static_cast<long long>(warp + i * kScoreWarps) * 16;
                unsigned char *dst = mine + (i % kWarpStages) * kGroupBytes;
#pragma unroll
                for (int m = 0; m < 8; ++m) {   // 16 rows x 16 chunks over 32 lanes
                    const int r = (lane >> 4) + 2 * m, ch = lane & 15;
                    if (ch < n_chunks) {
                        const long long j = g0 + r;
                        const bool valid = j < hi;
                        const uint32_t sdst =
                            static_cast<uint32_t>(__cvta_generic_to_shared(dst + r * 256 + ((ch ^ (r & 7)) << 4)));
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sdst),
                                     "l"(a.k_idx + (valid ? j : lo) * a.d_idx + ch * 8), "r"(valid ? 16 : 0)
                                     : "memory");
                    }
                }
            }
            cp_async_commit();   // one group per stage, empty past the last
        };
#pragma unroll
        for (int i = 0; i < kWarpStages - 1; ++i) issue(i);
        for (int i = 0; i < my_groups; ++i) {
            cp_async_wait<kWarpStages - 2>();   // group i has landed (this lane's copies)
            __syncwarp();                       // ... and every lane's; group i-1's stage is free
            issue(i + kWarpStages - 1);
            const unsigned char *src = mine + (i % kWarpStages) * kGroupBytes;
            float d[4] = {0.f, 0.f, 0.f, 0.f}, e4[4] = {0.f, 0.f, 0.f, 0.f};
            const int r = lane & 15;   // this lane's ldmatrix row
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (s < ksteps) {
                    const int ch = 2 * s + (lane >> 4);
                    uint32_t af[4], aa[4];
                    ldmatrix_x4(af[0], af[1], af[2], af[3], src + r * 256 + ((ch ^ (r & 7)) << 4));
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2 x = __habs2(*reinterpret_cast<const __half2 *>(&af[e]));
                        aa[e] = *reinterpret_cast<const uint32_t *>(&x);
                    }
                    mma_16816(d, af, bq0[s], bq1[s]);
                    mma_16816(e4, aa, ba0[s], ba1[s]);
                }
            }
            if ((lane & 3) == 0) {   // column 0: rows lane/4 and lane/4 + 8 of the group
                const long long j = lo + static_cast<long long>(warp + i * kScoreWarps) * 16 + (lane >> 2);
                if (j < hi) {
                    keys[j - lo] = float_key(d[0]);
                    bmax = fmaxf(bmax, e4[0]);
                }
                if (j + 8 < hi) {
                    keys[j + 8 - lo] = float_key(d[2]);
                    bmax = fmaxf(bmax, e4[2]);
                }
            }
        }
        cp_async_wait<0>();
    }
    __syncthreads();
}

// The sessions of a batched decode step: session s's inputs sit at fixed strides
// from session 0's and its position is pos[s] (device memory, read early).
struct DecodeBatch {
    const long long *pos;     // nullptr: one session, at IndexerArgs::q_pos0
    long long q_stride;       // elements between the sessions' indexer queries
    long long k_stride;       // elements between the sessions' indexer keys
    long long out_stride;     // elements between the sessions' kept-row lists
    long long ws_stride;      // bytes between the sessions' workspaces
    const uint16_t *ring_k;   // compressor: the new token is slot pos % W of the session's ring
    const uint16_t *ring_v;
    long long ring_stride;    // elements between the sessions' rings
    long long state_stride;   // floats between the sessions' compressor states
    long long comp_stride;    // elements between the sessions' compressed rows
    long long cap;            // compressed rows allocated per session
    unsigned int *err;
    int W;
    int comp_cta0;            // the compressor's update runs in scoring CTA 0 (no CTA of its own)
};

// one query per session: CTA x < n_score scores rows [x*rows_per_cta, (x+1)*rows_per_cta)
// in 64-row slices; the last of them to finish selects.  With kCompress the grid has
// one more CTA per session, which feeds the query's token to the layer's compressor:
// that update reads nothing the selection writes and vice versa.  blockIdx.y is the
// session of a batched step.
constexpr int kBandMaxRows = kThreads * kMaxItems;   // approximate path: rows per session

// shared memory of the exact select, and of the band select of the approximate path
struct ExactSmem {
    SelectSmem sm;
};
union ApproxSmem {
    SelectSmem sm;
    sel::BandSmem<kThreads, kBandMaxRows> band;
};

// kFold: the compressor's update runs in scoring CTA 0 (DecodeBatch::comp_cta0).  The
// single-session launches are instantiated without the batched-only paths: code and
// shared memory they never use measured 0.4 us slower on a decode step.
// kKeyRow: one session whose compressor pools the tokens' indexer keys (c.ki): the
// compressor's CTA also scores a row its token completes (a separate instantiation, so
// that the other launches carry none of its code).
template <bool kCompress, int kDeep, bool kApprox, bool kFold, int kSelItems = 0, bool kKeyRow = false>
__global__ void __launch_bounds__(kThreads, 1) indexer_decode_kernel(IndexerArgs a, int rows_per_cta,
                                                                     cmp::CompressArgs c, DecodeBatch bt) {
    __shared__ typename std::conditional<kApprox, ApproxSmem, ExactSmem>::type u;
    SelectSmem &sm = u.sm;
    __shared__ bool s_last;
    __shared__ uint32_t s_keys[kStagedRows];
    __shared__ float s_red[kWarps];
    bool comp_skip = false;     // the token would complete a row past the session's capacity
    if (bt.pos != nullptr) {
        const long long sid = blockIdx.y;
        const long long p = bt.pos[sid];
        a.q_pos0 = p;
        a.q_idx += sid * bt.q_stride;
        a.k_idx += sid * bt.k_stride;
        a.out_idx += sid * bt.out_stride;
        if (a.out_n) a.out_n += sid;
        a.ws += sid * bt.ws_stride;
        if constexpr (kCompress) {
            if ((p + 1) / c.ratio > bt.cap) {
                // the row this token completes is past the session's capacity: no update
                comp_skip = true;
                if (blockIdx.x == (kFold ? 0u : gridDim.x - 1) && threadIdx.x == 0)
                    record_error(bt.err, DS4A_ERR_CAPACITY);
                if (!kFold && blockIdx.x == gridDim.x - 1) return;
            }
            const long long slot = (p % bt.W) * c.D;
            c.pos = p;
            c.k = bt.ring_k + sid * bt.ring_stride + slot;
            c.v = bt.ring_v + sid * bt.ring_stride + slot;
            c.state += sid * bt.state_stride;
            c.comp_k += sid * bt.comp_stride;
            c.comp_v += sid * bt.comp_stride;
        }
    }
    // Pooled indexer keys (c.ki, one session): the compressor's CTA also pools the token's
    // indexer key, and when the token completes a row it writes that row's key, scores it
    // (the exact key, as the scoring CTAs compute it) into the workspace and takes a
    // ticket like a scoring CTA; the scoring CTAs leave that row to it.
    long long key_row = -1;
    if constexpr (kCompress && !kFold) {
        if constexpr (kKeyRow) {
            if ((a.q_pos0 + 1) % a.ratio == 0 && (a.q_pos0 + 1) / a.ratio <= a.n_rows)
                key_row = (a.q_pos0 + 1) / a.ratio - 1;
        }
        if (blockIdx.x == gridDim.x - 1) {
            static_assert(sizeof(sm.scan) >= kWarps * sizeof(float), "one float per warp");
            compress_one_token(c, reinterpret_cast<float *>(s_keys), reinterpret_cast<float *>(sm.scan));
            if (!kKeyRow || key_row < 0) return;
            __syncthreads();   // the row's key is in memory (this CTA's own writes)
            const uint32_t kx = sel::exact_key16<true>(a.q_idx, c.comp_ki + key_row * a.d_idx, a.d_idx,
                                                       threadIdx.x < 16);
            unsigned int *ticket = reinterpret_cast<unsigned int *>(a.ws);
            uint32_t *keys = reinterpret_cast<uint32_t *>(a.ws + kWsHeader);
            if (threadIdx.x == 0) {
                keys[key_row] = kx;
                unsigned int old;
                asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;\n" : "=r"(old) : "l"(ticket) : "memory");
                s_last = old == gridDim.x - 1;   // every scoring CTA and this one
            }
            __syncthreads();
            if (!s_last) return;
            select_topk_sized<kSelItems>(keys, static_cast<int>(visible_rows(a, 0)), a.k, a.out_idx, a.out_n, sm);
            if (threadIdx.x == 0) *ticket = 0u;
            return;
        }
    } else {
        (void)c;
    }
    // with comp_cta0, scoring CTA 0 also runs the compressor's update: its score before the
    // dependency wait, the running state and a completed row after it
    const bool comp_here = kCompress && kFold && blockIdx.x == 0 && !comp_skip;
    // tickets: the scoring CTAs, and the compressor's CTA when it scores a row
    const unsigned int n_score = (kCompress && !kFold) ? gridDim.x - (key_row < 0 ? 1u : 0u) : gridDim.x;
    (void)comp_skip;
    const long long n_vis = visible_rows(a, 0);
    const long long j0 = static_cast<long long>(blockIdx.x) * rows_per_cta;
    const long long j1 = min(key_row < 0 ? n_vis : key_row, j0 + rows_per_cta);
    // The query and the key rows complete before the query's token (j < floor(q_pos/ratio))
    // are inputs the kernel just ahead does not write, so up to kStagedRows of those rows
    // of the slice are scored into shared memory before waiting on the previous kernel.
    // A row the query's own token completes (which a compressor call just ahead may
    // write), the workspace and the output are read or written after the wait.
    extern __shared__ __align__(16) unsigned char dyn_smem[];   // approximate path: stages, then keys
    uint32_t *pre_keys = kApprox ? reinterpret_cast<uint32_t *>(dyn_smem + kStageBytes) : s_keys;
    const long long pre_cap = kApprox ? kApproxStagedRows : kStagedRows;
    const long long js = max(j0, min(min(j1, j0 + pre_cap), a.q_pos0 / a.ratio));
    float qf[2][8];
    float bmax = 0.f;   // approximate path: largest sum_c |q_c k_c| of this CTA's rows
    load_query(a.q_idx, a.d_idx, qf);
    if constexpr (kApprox) {
        if (a.d_idx % 16 == 0 && a.d_idx <= 128) score_rows_staged(a, j0, js, pre_keys, bmax, dyn_smem);
        else score_rows<kDeep, true>(a, qf, j0, js, pre_keys, j0, bmax);
    } else {
        score_rows<kDeep, false>(a, qf, j0, js, pre_keys, j0, bmax);
    }
    if constexpr (kCompress && !kFold && !kApprox && (kSelItems == 8 || kSelItems == 16)) {
        // Warm L2 with the compressed K and V rows the query most likely keeps: the
        // best `want` of this CTA's pre-scored rows, want = its even share of the k
        // kept rows plus 4.  A prefetch returns no data; attention gathers the kept
        // rows once the selection is done.
        const int nloc = static_cast<int>(js - j0);
        if (nloc > 0 && nloc <= 64) {   // the ranking costs nloc^2 / 512 compares a thread
            __syncthreads();   // pre_keys complete
            const long long share = (static_cast<long long>(nloc) * a.k + n_vis - 1) / n_vis;
            const int want = static_cast<int>(min(static_cast<long long>(nloc), share + 4));
            const int row_bytes = c.D * 2;
            // tpr threads (a power of two) rank each row, each against every tpr-th key
            int tpr = 1;
            while (tpr < 32 && tpr * 2 * nloc <= kThreads) tpr *= 2;
            for (int rb = 0; rb < nloc; rb += kThreads / tpr) {   // block-uniform trip count
                const int r = rb + static_cast<int>(threadIdx.x) / tpr, sub = threadIdx.x % tpr;
                int above = 0;
                if (r < nloc) {
                    const uint32_t kr = pre_keys[r];
                    for (int o = sub; o < nloc; o += tpr) {
                        const uint32_t ko = pre_keys[o];
                        above += (ko > kr) || (ko == kr && o < r);
                    }
                }
                for (int m = 1; m < tpr; m <<= 1) above += __shfl_xor_sync(0xffffffffu, above, m);
                if (r < nloc && sub == 0 && above < want) {
                    const char *pk = reinterpret_cast<const char *>(c.comp_k + (j0 + r) * c.D);
                    const char *pv = reinterpret_cast<const char *>(c.comp_v + (j0 + r) * c.D);
                    for (int off = 0; off < row_bytes; off += 128) {
                        prefetch_l2_line(pk + off);
                        prefetch_l2_line(pv + off);
                    }
                    prefetch_l2_line(pk + row_bytes - 1);
                    prefetch_l2_line(pv + row_bytes - 1);
                }
            }
        }
    }
    __shared__ float s_cw[1];   // kFold: the compressor's score of the step's token
    if constexpr (kFold) {
        if (comp_here) cmp::segment_scores<kThreads>(c, c.pos, c.pos + 1, s_cw);
    }
    pdl_wait();
    pdl_trigger();
    if constexpr (kFold) {
        if (comp_here)
            cmp::pool_segment<kThreads>(c, c.pos / c.ratio, c.pos, c.pos + 1, c.pos % c.ratio != 0, s_cw, s_red);
    }
    unsigned int *ticket = reinterpret_cast<unsigned int *>(a.ws);
    unsigned int *bmax_word = ticket + 1;   // approximate path: the session's largest sum_c |q_c k_c|
    uint32_t *keys = reinterpret_cast<uint32_t *>(a.ws + kWsHeader);
    __syncthreads();
    for (long long j = j0 + threadIdx.x; j < js; j += kThreads) keys[j] = pre_keys[j - j0];
    score_rows<kDeep, kApprox>(a, qf, js, j1, keys, 0, bmax);
    if constexpr (kApprox) {
        // non-negative floats order like their bit patterns: one atomicMax per CTA
        bmax = warp_max(bmax);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = bmax;
        __syncthreads();
        if (threadIdx.x == 0) {
            float m = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = fmaxf(m, s_red[w]);
            atomicMax(bmax_word, __float_as_uint(m));
        }
    }
    // one acquire-release atomic per CTA: releases this CTA's keys (ordered before it
    // by the barrier) and, for the last CTA, acquires everyone else's
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int old;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;\n" : "=r"(old) : "l"(ticket) : "memory");
        s_last = old == n_score - 1;
    }
    __syncthreads();
    if (!s_last) return;
    if constexpr (kApprox) {
        const int n = static_cast<int>(n_vis);
        if (a.out_n && threadIdx.x == 0) *a.out_n = n < a.k ? n : a.k;
        if (n <= a.k) {
            for (int i = threadIdx.x; i < a.k; i += kThreads) a.out_idx[i] = i < n ? i : -1;
        } else {
            // eps bounds |approximate - exact| score for every row: 2^-12 max_j sum_c |q_c k_jc|
            if (threadIdx.x == 0) u.band.eps = ldexpf(__uint_as_float(__ldcg(bmax_word)) * 1.01f, -12) + 1e-30f;
            __syncthreads();
            const float eps = u.band.eps;
            if constexpr (kSelItems != 0) {
                band_select_regs<kSelItems>(a, keys, n, eps, u.band);
            } else {
                if (n <= kThreads * 8) band_select_regs<8>(a, keys, n, eps, u.band);
                else if (n <= kThreads * 16) band_select_regs<16>(a, keys, n, eps, u.band);
                else band_select_regs<kMaxItems>(a, keys, n, eps, u.band);
            }
        }
        if (threadIdx.x == 0) *bmax_word = 0u;
    } else {
        select_topk_sized<kSelItems>(keys, static_cast<int>(n_vis), a.k, a.out_idx, a.out_n, sm);
    }
    if (threadIdx.x == 0) *ticket = 0u;
}

// many queries: one CTA per query
__global__ void __launch_bounds__(kThreads, 1) indexer_query_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint32_t skeys[];
    __shared__ SelectSmem sm;
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const long long n_vis = visible_rows(a, i);
    const bool in_smem = n_vis <= kSmemKeyCap;
    uint32_t *keys = in_smem ? skeys
                             : reinterpret_cast<uint32_t *>(a.ws + kWsHeader) + static_cast<size_t>(i) * a.n_rows;
    float qf[2][8];
    load_query(a.q_idx + static_cast<size_t>(i) * a.d_idx, a.d_idx, qf);
    for (long long base = 0; base < n_vis; base += kRowsPerCta) {
        RowLoads L;
        load_rows(a.k_idx, a.d_idx, base, n_vis, L);
        score_loaded(qf, L, base, n_vis, keys + base);
    }
    __syncthreads();
    int32_t *out = a.out_idx + static_cast<size_t>(i) * a.k;
    int32_t *out_n = a.out_n ? a.out_n + i : nullptr;
    if (in_smem) select_topk<false>(keys, static_cast<int>(n_vis), a.k, out, out_n, sm);
    else select_topk<true>(keys, static_cast<int>(n_vis), a.k, out, out_n, sm);
}

constexpr size_t kQuerySmem = kSmemKeyCap * sizeof(uint32_t);

}  // namespace

size_t indexer_ws_bytes(int n_q, long long n_rows, int k) {
    (void)k;
    size_t keys = 0;
    if (n_q <= 1) keys = static_cast<size_t>(n_rows);
    else if (n_rows > kSmemKeyCap) keys = static_cast<size_t>(n_q) * static_cast<size_t>(n_rows);
    size_t bytes = kWsHeader + keys * sizeof(uint32_t);
    // the tensor-core path for many queries keeps [n_q][rows] approximate scores and the key norms
    if (n_q > 1) {
        const size_t tc_bytes = indexer_prefill_tc_ws_bytes(n_q, n_rows);
        if (tc_bytes > bytes) bytes = tc_bytes;
    }
    return bytes;
}

// One decode query: 64-row slices spread so that the scoring grid is at most one
// CTA on each of `sms` SMs.
static unsigned decode_grid(long long q_pos, long long n_rows, int ratio, int sms, int &rows_per_cta) {
    long long n_vis = (q_pos + 1) / ratio;
    if (n_vis > n_rows) n_vis = n_rows;
    const long long slices = (n_vis + kRowsPerCta - 1) / kRowsPerCta;
    const long long per_cta = slices > sms ? (slices + sms - 1) / sms : 1;
    rows_per_cta = static_cast<int>(per_cta * kRowsPerCta);
    long long grid = (n_vis + rows_per_cta - 1) / rows_per_cta;
    return static_cast<unsigned>(grid < 1 ? 1 : grid);
}

static cudaError_t configure_indexer(const Ctx &c);

// the register-select size a one-query launch over n_vis rows needs (0: the run-time choice)
static int sel_items_for(long long n_vis) {
    if (n_vis <= kThreads * 8LL) return 8;
    if (n_vis <= kThreads * 16LL) return 16;
    if (n_vis <= kThreads * static_cast<long long>(kMaxItems)) return kMaxItems;
    return 0;
}

// a one-query decode kernel (kCompress: with the compressor's CTA; kKeyRow: that CTA pools
// indexer keys and scores the row its token completes) with the select its rows need
template <bool kCompress, bool kKeyRow = false>
static auto decode_kernel_for(long long n_vis) {
    switch (sel_items_for(n_vis)) {
        case 8: return indexer_decode_kernel<kCompress, 1, false, false, 8, kKeyRow>;
        case 16: return indexer_decode_kernel<kCompress, 1, false, false, 16, kKeyRow>;
        case kMaxItems: return indexer_decode_kernel<kCompress, 1, false, false, kMaxItems, kKeyRow>;
        default: return indexer_decode_kernel<kCompress, 1, false, false, 0, kKeyRow>;
    }
}

// a batched approximate-score launch with the band select its sessions' capacity needs
template <bool kFold>
static auto approx_kernel_for(long long cap) {
    switch (sel_items_for(cap)) {
        case 8: return indexer_decode_kernel<true, 4, true, kFold, 8>;
        case 16: return indexer_decode_kernel<true, 4, true, kFold, 16>;
        default: return indexer_decode_kernel<true, 4, true, kFold, kMaxItems>;
    }
}

cudaError_t launch_indexer(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                           int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                           int32_t *out_n, void *ws, const Ctx &c) {
    if (d_idx > kMaxDIdx || n_rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = configure_indexer(c);
    if (e != cudaSuccess) return e;
    IndexerArgs a{q_idx, k_idx, out_idx, out_n, static_cast<unsigned char *>(ws), n_rows, q_pos0,
                  n_q, d_idx, ratio, k};
    if (n_q == 1) {
        int rows_per_cta = 0;
        const unsigned grid = decode_grid(q_pos0, n_rows, ratio, c.num_sms, rows_per_cta);
        const long long n_vis = (q_pos0 + 1) / ratio < n_rows ? (q_pos0 + 1) / ratio : n_rows;
        return launch(decode_kernel_for<false>(n_vis), dim3(grid), dim3(kThreads), 0, c, 1, a, rows_per_cta,
                      cmp::CompressArgs{}, DecodeBatch{});
    }
    if (indexer_prefill_tc_ok(n_q, n_rows, d_idx))
        return launch_indexer_prefill_tc(q_idx, n_q, k_idx, n_rows, d_idx, q_pos0, ratio, k, out_idx, out_n, ws, c);
    return launch(indexer_query_kernel, dim3(static_cast<unsigned>(n_q)), dim3(kThreads), kQuerySmem, c, 1, a);
}

cudaError_t launch_indexer_compress(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows, int d_idx,
                                   long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                                   const uint16_t *k_new, const uint16_t *v_new, int D, const float *score_w,
                                   float *state, uint16_t *comp_k, uint16_t *comp_v, const Ctx &c,
                                   const uint16_t *k_idx_tok) {
    if (d_idx > kMaxDIdx || n_rows > 0x7fffffffLL || ratio > cmp::kMaxRatio || D > cmp::kMaxD)
        return cudaErrorInvalidValue;
    cudaError_t e = configure_indexer(c);
    if (e != cudaSuccess) return e;
    IndexerArgs a{q_idx, k_idx, out_idx, out_n, static_cast<unsigned char *>(ws), n_rows, q_pos,
                  1, d_idx, ratio, k};
    // with k_idx_tok the compressor also pools the tokens' indexer keys into k_idx
    const cmp::CompressArgs ca{k_new, v_new, score_w, state, comp_k, comp_v, q_pos, 1, D, ratio,
                               k_idx_tok, k_idx_tok ? const_cast<uint16_t *>(k_idx) : nullptr,
                               k_idx_tok ? d_idx : 0};
    int rows_per_cta = 0;
    // the scoring CTAs leave one SM for the compressor's CTA
    const unsigned grid = decode_grid(q_pos, n_rows, ratio, c.num_sms > 1 ? c.num_sms - 1 : 1, rows_per_cta);
    const long long n_vis = (q_pos + 1) / ratio < n_rows ? (q_pos + 1) / ratio : n_rows;
    return launch(k_idx_tok ? decode_kernel_for<true, true>(n_vis) : decode_kernel_for<true>(n_vis), dim3(grid + 1),
                  dim3(kThreads), 0, c, 1, a, rows_per_cta, ca, DecodeBatch{});
}

size_t indexer_batched_ws_stride(long long cap) {
    return (kWsHeader + static_cast<size_t>(cap) * sizeof(uint32_t) + 255) / 256 * 256;
}

cudaError_t launch_indexer_compress_batched(int B, const uint16_t *q_idx, const uint16_t *k_idx, long long cap,
                                           int d_idx, const long long *pos, int ratio, int k, int32_t *out_idx,
                                           int32_t *out_n, void *ws, const uint16_t *ring_k, const uint16_t *ring_v,
                                           int W, int D, const float *score_w, float *state, uint16_t *comp_k,
                                           uint16_t *comp_v, const Ctx &c) {
    if (d_idx > kMaxDIdx || cap > 0x7fffffffLL || ratio > cmp::kMaxRatio || D > cmp::kMaxD)
        return cudaErrorInvalidValue;
    cudaError_t e = configure_indexer(c);
    if (e != cudaSuccess) return e;
    IndexerArgs a{q_idx, k_idx, out_idx, out_n, static_cast<unsigned char *>(ws), cap, 0, 1, d_idx, ratio, k};
    const cmp::CompressArgs ca{nullptr, nullptr, score_w, state, comp_k, comp_v, 0, 1, D, ratio};
    // every session's CTAs in one wave when B allows: (SMs - B) / B scoring CTAs per
    // session and one compressor CTA each; or, from 32 sessions on (where the separate
    // CTAs would take a large share of the SMs), SMs / B scoring CTAs with the
    // compressor's update in each session's CTA 0 (64 sessions: 131 -> 84 us per step;
    // at 16 it measured slower).  The row split is sized for the largest row count (cap).
    const int per_sep = c.num_sms > 2 * B ? (c.num_sms - B) / B : 1;
    const int per_fold = c.num_sms / B > 1 ? c.num_sms / B : 1;
    const bool fold = B >= 32 && per_fold > per_sep && cap <= kBandMaxRows;   // folded: approximate path only
    DecodeBatch bt{pos, d_idx, cap * d_idx, k, static_cast<long long>(indexer_batched_ws_stride(cap)),
                   ring_k, ring_v, static_cast<long long>(W) * D, 2 + 2LL * D, cap * D, cap, c.err, W,
                   fold ? 1 : 0};
    int rows_per_cta = 0;
    const unsigned n_sc = decode_grid(cap * ratio, cap, ratio, fold ? per_fold : per_sep, rows_per_cta);
    const unsigned grid = fold ? n_sc - 1 : n_sc;   // the launches below add the compressor's CTA
    // approximate scores with an exact band when every session's rows fit the band select
    // and a CTA covers enough rows for the cheaper scoring to outweigh the band's rescoring;
    // exact scores otherwise, one 64-row batch per round when a CTA covers two at most
    if (cap <= kBandMaxRows && rows_per_cta >= 512) {
        if (fold)
            return launch(approx_kernel_for<true>(cap), dim3(grid + 1, B), dim3(kThreads), kApproxDynBytes, c, 1, a,
                          rows_per_cta, ca, bt);
        return launch(approx_kernel_for<false>(cap), dim3(grid + 1, B), dim3(kThreads), kApproxDynBytes, c, 1, a,
                      rows_per_cta, ca, bt);
    }
    if (rows_per_cta <= 2 * kRowsPerCta)
        return launch(indexer_decode_kernel<true, 1, false, false>, dim3(grid + 1, B), dim3(kThreads), 0, c, 1, a,
                      rows_per_cta, ca, bt);
    return launch(indexer_decode_kernel<true, 4, false, false>, dim3(grid + 1, B), dim3(kThreads), 0, c, 1, a,
                  rows_per_cta, ca, bt);
}

// kernel attributes, once per device and host thread
static cudaError_t configure_indexer(const Ctx &c) {
    (void)c;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kQuerySmem));
        for (long long n_vis : {1LL * kThreads * 8, 1LL * kThreads * 16, 1LL * kThreads * kMaxItems, 1LL << 40}) {
            for (auto kern : {decode_kernel_for<false>(n_vis), decode_kernel_for<true>(n_vis),
                              decode_kernel_for<true, true>(n_vis)})
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(indexer_decode_kernel<true, 1, false, false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        for (long long cap : {1LL * kThreads * 8, 1LL * kThreads * 16, 1LL * kThreads * kMaxItems}) {
            for (auto kern : {approx_kernel_for<false>(cap), approx_kernel_for<true>(cap)}) {
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kApproxDynBytes));
            }
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(indexer_decode_kernel<true, 4, false, false>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(indexer_query_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return cudaSuccess;
}

}  // namespace ds4a
