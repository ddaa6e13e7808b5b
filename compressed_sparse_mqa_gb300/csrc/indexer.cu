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
// Select.  Scores map to order-preserving u32 keys; a radix select over four
// 8-bit digits (per-warp shared-memory histograms) finds the k-th largest key;
// rows above it, then rows equal to it in ascending index order, are emitted in
// ascending index order with two block-wide scans.
//
// Decode (one query): a grid of CTAs sized to the SM count scores slices of the
// rows into the workspace; the last CTA to finish (atomic ticket, no waiting)
// runs the select and resets the ticket.  Prefill (many queries): one CTA per
// query scores its visible rows into shared memory and selects.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace ds4a {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 16;                        // threads per scored row
constexpr int kRowsPerPass = kThreads / kGroup;   // 32
constexpr int kMaxDIdx = 256;
constexpr size_t kWsHeader = 256;                 // ticket lives here
constexpr int kSmemKeyCap = 24576;                // keys staged in shared memory

struct SelectSmem {
    uint32_t hist[kWarps][256];
    uint32_t total[256];
    uint32_t scan[kWarps];
    uint32_t bin;
    uint32_t above;
};

// Score rows [j0, j1) of one query into keys[j - key_base].  q is staged once
// per thread: thread (group lane gl) owns 8-dim chunks gl and gl + 16.
__device__ void score_rows(const uint16_t *__restrict__ q, const uint16_t *__restrict__ kidx, int d_idx,
                           long long j0, long long j1, uint32_t *keys, long long key_base) {
    const int tid = threadIdx.x;
    const int gl = tid % kGroup;
    const int n_chunks = d_idx / 8;
    float qf[2][8];
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
    for (long long j = j0 + tid / kGroup; j < j1; j += kRowsPerPass) {
        float s = 0.f, c = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int ch = gl + cc * kGroup;
            if (ch < n_chunks) {
                uint4 raw = __ldg(reinterpret_cast<const uint4 *>(kidx + j * d_idx + ch * 8));
                const uint16_t *h = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float err;
                    two_sum(s, qf[cc][e] * h2f(h[e]), s, err);
                    c += err;
                }
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
        if (gl == 0) keys[j - key_base] = float_key(s + c);
    }
}

// Block-wide exclusive scan of one value per thread (kThreads threads).
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t *scratch, uint32_t &total) {
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
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = scratch[w];
        if (w < warp) before += t;
        all += t;
    }
    total = all;
    return before + incl - v;
}

// Keep the k largest of keys[0..n) (ties to the lower index); write them in
// ascending order to out[0..k), -1 past min(k, n); out_n (if given) = min(k, n).
__device__ void block_topk(const uint32_t *keys, int n, int k, int32_t *out, int32_t *out_n,
                           SelectSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (n <= k) {
        for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
        if (out_n && tid == 0) *out_n = n;
        return;
    }
    uint32_t prefix = 0, mask = 0, kk = static_cast<uint32_t>(k);
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < kWarps * 256; i += kThreads) (&sm.hist[0][0])[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t key = keys[i];
            if ((key & mask) == prefix) atomicAdd(&sm.hist[warp][(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t t = 0;
            for (int w = 0; w < kWarps; ++w) t += sm.hist[w][tid];
            sm.total[tid] = t;
        }
        __syncthreads();
        if (warp == 0) {
            // lane L covers bins 255-8L down to 248-8L (largest bins first)
            uint32_t cnt[8], lsum = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) { cnt[e] = sm.total[255 - 8 * lane - e]; lsum += cnt[e]; }
            uint32_t incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= kk);
            const int first = __ffs(hit) - 1;
            if (lane == first) {
                uint32_t before = incl - lsum;
                for (int e = 0; e < 8; ++e) {
                    if (before + cnt[e] >= kk) { sm.bin = 255 - 8 * lane - e; sm.above = before; break; }
                    before += cnt[e];
                }
            }
        }
        __syncthreads();
        kk -= sm.above;
        prefix |= sm.bin << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    // emit in ascending index order: thread t owns the contiguous range [t*C, t*C + C)
    const int C = (n + kThreads - 1) / kThreads;
    const int lo = tid * C, hi = min(n, lo + C);
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = keys[i];
        n_gt += key > prefix;
        n_eq += key == prefix;
    }
    uint32_t tot;
    const uint32_t eq_before = block_excl_scan(n_eq, sm.scan, tot);
    const uint32_t take = eq_before >= kk ? 0u : min(n_eq, kk - eq_before);
    const uint32_t pos0 = block_excl_scan(n_gt + take, sm.scan, tot);
    uint32_t p = pos0, taken = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = keys[i];
        if (key > prefix) out[p++] = i;
        else if (key == prefix && taken < take) { out[p++] = i; ++taken; }
    }
    if (out_n && tid == 0) *out_n = k;
}

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

__device__ __forceinline__ long long visible_rows(const IndexerArgs &a, int i) {
    const long long v = (a.q_pos0 + i + 1) / a.ratio;
    return v < a.n_rows ? v : a.n_rows;
}

// one query, many CTAs: score a slice each, the last CTA selects
__global__ void __launch_bounds__(kThreads) indexer_decode_kernel(IndexerArgs a, int rows_per_cta) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(smem_raw);
    __shared__ bool s_last;
    pdl_wait();
    pdl_trigger();
    unsigned int *ticket = reinterpret_cast<unsigned int *>(a.ws);
    uint32_t *keys = reinterpret_cast<uint32_t *>(a.ws + kWsHeader);
    const long long n_vis = visible_rows(a, 0);
    const long long j0 = static_cast<long long>(blockIdx.x) * rows_per_cta;
    const long long j1 = min(n_vis, j0 + rows_per_cta);
    if (j0 < j1) score_rows(a.q_idx, a.k_idx, a.d_idx, j0, j1, keys, 0);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // keys written by other CTAs: read through L2 (they were never cached in this SM's L1)
    uint32_t *skeys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelectSmem));
    const uint32_t *src = keys;
    if (n_vis <= kSmemKeyCap) {
        for (long long i = threadIdx.x; i < n_vis; i += kThreads) skeys[i] = __ldcg(keys + i);
        src = skeys;
        __syncthreads();
    }
    block_topk(src, static_cast<int>(n_vis), a.k, a.out_idx, a.out_n, sm);
    if (threadIdx.x == 0) *ticket = 0u;
}

// many queries: one CTA per query
__global__ void __launch_bounds__(kThreads) indexer_query_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(smem_raw);
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const long long n_vis = visible_rows(a, i);
    uint32_t *keys;
    if (n_vis <= kSmemKeyCap) keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelectSmem));
    else keys = reinterpret_cast<uint32_t *>(a.ws + kWsHeader) + static_cast<size_t>(i) * a.n_rows;
    score_rows(a.q_idx + static_cast<size_t>(i) * a.d_idx, a.k_idx, a.d_idx, 0, n_vis, keys, 0);
    __syncthreads();
    block_topk(keys, static_cast<int>(n_vis), a.k, a.out_idx + static_cast<size_t>(i) * a.k,
               a.out_n ? a.out_n + i : nullptr, sm);
}

constexpr size_t kSelectSmem = (sizeof(SelectSmem) + 15) / 16 * 16;
constexpr size_t kMaxSmem = kSelectSmem + kSmemKeyCap * sizeof(uint32_t);

}  // namespace

size_t indexer_ws_bytes(int n_q, long long n_rows, int k) {
    (void)k;
    const long long nq = n_q > 1 ? n_q : 1;
    return kWsHeader + static_cast<size_t>(nq) * static_cast<size_t>(n_rows) * sizeof(uint32_t);
}

cudaError_t launch_indexer(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                           int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                           int32_t *out_n, void *ws, const Ctx &c) {
    if (d_idx > kMaxDIdx || n_rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(indexer_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    IndexerArgs a{q_idx, k_idx, out_idx, out_n, static_cast<unsigned char *>(ws), n_rows, q_pos0,
                  n_q, d_idx, ratio, k};
    if (n_q == 1) {
        long long n_vis = (q_pos0 + 1) / ratio;
        if (n_vis > n_rows) n_vis = n_rows;
        long long grid = (n_vis + kRowsPerPass - 1) / kRowsPerPass;
        if (grid > c.num_sms) grid = c.num_sms;
        if (grid < 1) grid = 1;
        const int rows_per_cta = static_cast<int>((n_vis + grid - 1) / grid);
        return launch(indexer_decode_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kMaxSmem,
                      c, 1, a, rows_per_cta);
    }
    return launch(indexer_query_kernel, dim3(static_cast<unsigned>(n_q)), dim3(kThreads), kMaxSmem, c, 1, a);
}

}  // namespace ds4a
