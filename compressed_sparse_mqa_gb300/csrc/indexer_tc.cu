// indexer_tc.cu -- the prefill indexer on the 5th-generation tensor cores.
//
// "DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": on ratio-4
// layers a learned indexer keeps the top-512 compressed rows for every query of
// a prefill chunk.  For a chunk of T queries this is a [T x d] . [d x n_rows]
// score matrix followed by a per-query top-k.
//
// 1. indexer_scores_tc_kernel: tcgen05.mma (M = 128 queries, N = 256 rows,
//    K = d_idx, fp16 in, fp32 accumulate in tensor memory, two accumulator
//    buffers so the epilogue of one tile overlaps the MMAs of the next) writes
//    approximate scores s~ to the workspace, and the largest squared key norm
//    of every 256-row tile.
// 2. indexer_select_kernel: per query, the approximate scores s~ differ from the
//    exact scores s by at most eps = 2^-12 |q| max_j |k_j| (a bound far above the
//    tensor cores' fp32 accumulation error over d_idx <= 128 exact products).  Two
//    11-bit radix passes over s~ bracket the k-th largest s~ in [T_lo, T_hi].
//    Rows with s~ > T_hi + 2 eps + 4 ulp are kept for certain, rows with
//    s~ < T_lo - 2 eps - 4 ulp are dropped for certain; only the rows in between
//    (a handful) are rescored exactly (TwoSum over the exact fp16 products,
//    rounded once to binary32) and ranked (higher score, then lower index).  The
//    result is the exact top-k of the binary32-rounded exact scores.  If the band
//    is ever larger than its buffer (e.g. many equal keys), the query falls back
//    to exact scores for every row and an exact radix select.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"
#include "select.cuh"
#include "tcgen05.cuh"

namespace ds4a {
namespace {

constexpr int kTM = 128;                 // queries per tile (MMA M)
constexpr int kTN = 256;                 // rows per tile (MMA N)
constexpr int kGemmThreads = 128;

struct TcScoreArgs {
    const uint16_t *q_idx;
    const uint16_t *k_idx;
    float *scores;     // [n_q][ld]
    float *tile_kmax2; // [n_ntiles] largest squared key norm of each 256-row tile
    unsigned int *err;
    long long n_rows;
    long long early_rows;   // key rows below this may be read before the dependency wait
    int n_q;
    int ld;
    int n_ntiles;
    int n_split;
};

template <int DI>
__global__ void __launch_bounds__(kGemmThreads, 1) indexer_scores_tc_kernel(TcScoreArgs a) {
    constexpr int kAtoms = DI / 64;                 // 128-byte swizzle atoms along K
    constexpr int kChunks = DI / 8;                 // 16-byte chunks per row
    constexpr int kABytes = kAtoms * kTM * 128;
    constexpr int kBBytes = kAtoms * kTN * 128;
    constexpr uint32_t kIdesc = tc::idesc_f16_f32(kTM, kTN, false, false);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sa = smem;
    unsigned char *sb[2] = {smem + kABytes, smem + kABytes + kBBytes};
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_bar[2];
    __shared__ uint32_t s_kmax2;
    __shared__ float s_stage[kGemmThreads / 32][32 * 33];   // epilogue transpose, padded against bank conflicts

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kTM;
    const int ns = blockIdx.y;
    const int n_my = ns < a.n_ntiles ? (a.n_ntiles - ns + a.n_split - 1) / a.n_split : 0;

    if (tid == 0) {
        tc::mbar_init(&s_bar[0], 1);
        tc::mbar_init(&s_bar[1], 1);
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 2 * kTN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    auto load_b = [&](int it, int buf) {
        const long long row0 = static_cast<long long>(ns + it * a.n_split) * kTN;
        for (int i = tid; i < kTN * kChunks; i += kGemmThreads) {
            const int r = i / kChunks, c = i % kChunks;
            unsigned char *dst = sb[buf] + (c >> 3) * (kTN * 128) + tc::sw128_chunk(r, c & 7);
            const long long row = row0 + r;
            if (row < a.n_rows) cp_async16(dst, a.k_idx + row * DI + c * 8);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
    };
    // key rows complete before the chunk are cache state: the first tile is fetched before
    // waiting on the previous kernel when all of its rows are (later rows may be written by
    // the compressor call just ahead of this one)
    const bool early = n_my > 0 && static_cast<long long>(ns + 1) * kTN <= a.early_rows;
    if (early) load_b(0, 0);
    pdl_wait();
    pdl_trigger();
    if (n_my > 0 && !early) load_b(0, 0);
    for (int i = tid; i < kTM * kChunks; i += kGemmThreads) {
        const int r = i / kChunks, c = i % kChunks;
        unsigned char *dst = sa + (c >> 3) * (kTM * 128) + tc::sw128_chunk(r, c & 7);
        if (m0 + r < a.n_q) cp_async16(dst, a.q_idx + static_cast<long long>(m0 + r) * DI + c * 8);
        else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
    if (n_my > 1) {
        load_b(1, 1);
        cp_async_commit();
    }

    bool ok = true;
    // Epilogue: lane l of warp w holds query row 32w + l.  Each 32 x 32 block goes
    // through a padded shared tile so that a store instruction writes 128-byte runs
    // of four rows instead of 16 bytes of 32 rows.
    auto epilogue = [&](int it) {
        const int buf = it & 1;
        if (!tc::mbar_wait(&s_bar[buf], (it >> 1) & 1)) ok = false;
        tc::fence_after_sync();
        const long long col0 = static_cast<long long>(ns + it * a.n_split) * kTN;
        float *stg = s_stage[warp];
#pragma unroll 1
        for (int c0 = 0; c0 < kTN; c0 += 32) {
            uint32_t r[16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc::ld_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + buf * kTN + c0 + 16 * h, r);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[lane * 33 + 16 * h + j] = __uint_as_float(r[j]);
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = 4 * k + (lane >> 3), cg = 4 * (lane & 7);
                const int q = m0 + warp * 32 + row;
                const float *src = stg + row * 33 + cg;
                if (ok && q < a.n_q)
                    *reinterpret_cast<float4 *>(a.scores + static_cast<long long>(q) * a.ld + col0 + c0 + cg) =
                        make_float4(src[0], src[1], src[2], src[3]);
            }
            __syncwarp();
        }
    };

    for (int it = 0; it < n_my; ++it) {
        if (it == 0 && n_my > 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        tc::fence_proxy_async();
        __syncthreads();
        tc::fence_after_sync();
        const int buf = it & 1;
        if (tid == 0) {
#pragma unroll
            for (int s = 0; s < DI / 16; ++s) {
                const uint64_t da = tc::desc_sw128(tc::smem_u32(sa) + (s / 4) * (kTM * 128) + (s % 4) * 32, 16, 1024);
                const uint64_t db = tc::desc_sw128(tc::smem_u32(sb[buf]) + (s / 4) * (kTN * 128) + (s % 4) * 32, 16, 1024);
                tc::mma_f16(tmem + buf * kTN, da, db, kIdesc, s > 0 ? 1u : 0u);
            }
            tc::commit(&s_bar[buf]);
        }
        // largest squared norm of the tile's key rows (one M tile computes them)
        if (blockIdx.x == 0) {
            const long long row0 = static_cast<long long>(ns + it * a.n_split) * kTN;
            if (tid == 0) s_kmax2 = 0u;
            __syncthreads();
            float m2 = 0.f;
            for (int r = tid; r < kTN; r += kGemmThreads) {
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(sb[buf] + (c >> 3) * (kTN * 128) + tc::sw128_chunk(r, c & 7));
                    const uint16_t *h = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x = h2f(h[e]);
                        acc = fmaf(x, x, acc);
                    }
                }
                if (row0 + r < a.n_rows) m2 = fmaxf(m2, acc);
            }
            // non-negative floats order like their bit patterns
            atomicMax(&s_kmax2, __float_as_uint(warp_max(m2)));
            __syncthreads();
            if (tid == 0) a.tile_kmax2[ns + it * a.n_split] = __uint_as_float(s_kmax2);
        }
        if (it >= 1) {
            epilogue(it - 1);
            // MMA it-1 has completed: its B buffer takes tile it+1
            if (it + 1 < n_my) {
                load_b(it + 1, (it + 1) & 1);
                cp_async_commit();
            }
        }
        tc::fence_before_sync();
    }
    if (n_my > 0) epilogue(n_my - 1);
    if (!ok && tid == 0) record_error(a.err, DS4A_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 2 * kTN);
}

// ---- per-query select on approximate scores with an exact band ------------------------------

constexpr int kSelMaxRows = 8192;
constexpr int kBandCap = 1024;
constexpr int kBins = 2048;               // 11-bit digits

struct SelArgs {
    const uint16_t *q_idx;
    const uint16_t *k_idx;
    float *scores;          // [n_q][ld] approximate scores (overwritten by exact keys on fallback)
    const float *tile_kmax2;   // largest squared key norm of each 256-row tile
    int32_t *out_idx;
    int32_t *out_n;
    long long n_rows;
    long long q_pos0;
    int d_idx;
    int ratio;
    int k;
    int ld;
};

template <int NT>
struct SelSmem {
    uint32_t hist[kBins];
    uint32_t cnt[NT];
    uint32_t scan[NT / 32];
    int band_idx[kBandCap];
    uint32_t band_key[kBandCap];
    uint32_t sel_bits[kSelMaxRows / 32];
    uint32_t res[3], band_n, n_in;
    float eps;
};

DS4A_DEVINL float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// TwoSum-exact score of one row, computed by a group of 16 threads (all 32 lanes of
// every warp call this; `valid` masks the rows).
DS4A_DEVINL uint32_t exact_key16(const uint16_t *q, const uint16_t *krow, int d_idx, bool valid) {
    const int gl = threadIdx.x & 15;
    float s = 0.f, c = 0.f;
    for (int ch = gl; ch < d_idx / 8; ch += 16) {
        if (valid) {
            const uint4 qa = *reinterpret_cast<const uint4 *>(q + ch * 8);
            const uint4 ka = __ldg(reinterpret_cast<const uint4 *>(krow + ch * 8));
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

template <int NT, int ITEMS, int MIN_BLOCKS>
__global__ void __launch_bounds__(NT, MIN_BLOCKS) indexer_select_kernel(SelArgs a) {
    constexpr int kSelThreads = NT;
    __shared__ SelSmem<NT> sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    long long nv = (a.q_pos0 + i + 1) / a.ratio;
    const int n = static_cast<int>(nv < a.n_rows ? nv : a.n_rows);
    int32_t *out = a.out_idx + static_cast<size_t>(i) * a.k;
    if (a.out_n && tid == 0) a.out_n[i] = n < a.k ? n : a.k;
    if (n <= a.k) {
        for (int j = tid; j < a.k; j += kSelThreads) out[j] = j < n ? j : -1;
        return;
    }
    const uint16_t *q = a.q_idx + static_cast<size_t>(i) * a.d_idx;
    float *row = a.scores + static_cast<size_t>(i) * a.ld;

    uint32_t key[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * kSelThreads + tid;
        key[it] = j < n ? float_key(row[j]) : 0u;
    }
    // error bound of the approximate scores: |q| times the largest key norm of
    // the tiles holding the visible rows
    if (warp == 0) {
        float qn2 = 0.f;
        for (int c = lane; c < a.d_idx; c += 32) {
            const float x = h2f(q[c]);
            qn2 = fmaf(x, x, qn2);
        }
        float kmax2 = 0.f;
        for (int t = lane; t * kTN < n; t += 32) kmax2 = fmaxf(kmax2, a.tile_kmax2[t]);
        qn2 = warp_sum(qn2);
        kmax2 = warp_max(kmax2);
        if (lane == 0) sm.eps = ldexpf(sqrtf(qn2 * kmax2) * 1.01f, -12) + 1e-30f;
    }
    __syncthreads();
    const float eps = sm.eps;

    // bracket the k-th largest approximate score: bits 31..21, then 20..10
    uint32_t kk = static_cast<uint32_t>(a.k);
    sel::radix_pass<kSelThreads, ITEMS>(key, n, 0u, 0u, 21, 11, kk, sm.hist, sm.scan, sm.res);
    uint32_t prefix = sm.res[0] << 21, mask = 0xFFE00000u;
    kk -= sm.res[1];
    sel::radix_pass<kSelThreads, ITEMS>(key, n, prefix, mask, 10, 11, kk, sm.hist, sm.scan, sm.res);
    prefix |= sm.res[0] << 10;
    const uint32_t lo_key = prefix, hi_key = prefix | 0x3FFu;
    const float t_lo = key_to_float(lo_key), t_hi = key_to_float(hi_key);
    const float big = fmaxf(fabsf(t_lo), fabsf(t_hi));
    const float ulp = ldexpf(1.f, ilogbf(big > 0.f ? big : 1.f) - 23);
    const float margin = 2.f * eps + 4.f * ulp;
    const float in_thr = t_hi + margin, out_thr = t_lo - margin;

    // classify: certainly in, certainly out, or band (rescored exactly)
    if (tid == 0) {
        sm.band_n = 0;
        sm.n_in = 0;
    }
    for (int w = tid; w < ITEMS * kSelThreads / 32; w += kSelThreads) sm.sel_bits[w] = 0;
    __syncthreads();
    uint32_t flags = 0, my_in = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * kSelThreads + tid;
        if (j < n) {
            const float s = key_to_float(key[it]);
            if (s > in_thr) {
                flags |= 1u << it;
                ++my_in;
            } else if (s >= out_thr) {
                const uint32_t b = atomicAdd(&sm.band_n, 1u);
                if (b < kBandCap) sm.band_idx[b] = j;
            }
        }
    }
    my_in = __reduce_add_sync(0xffffffffu, my_in);
    if (lane == 0 && my_in) atomicAdd(&sm.n_in, my_in);
    __syncthreads();
    const uint32_t band_n = sm.band_n, n_in = sm.n_in;
    const bool fits = band_n <= kBandCap && n_in <= static_cast<uint32_t>(a.k) &&
                      n_in + band_n >= static_cast<uint32_t>(a.k);
    if (fits) {
        // exact keys of the band rows: 16 threads per row
        for (uint32_t b0 = 0; b0 < band_n; b0 += kSelThreads / 16) {
            const uint32_t b = b0 + tid / 16;
            const bool valid = b < band_n;
            const int j = valid ? sm.band_idx[b] : 0;
            const uint32_t kx = exact_key16(q, a.k_idx + static_cast<size_t>(j) * a.d_idx, a.d_idx, valid);
            if (valid && (tid & 15) == 0) sm.band_key[b] = kx;
        }
        __syncthreads();
        // keep the (k - n_in) best band rows: higher exact key, then lower index
        const uint32_t need = static_cast<uint32_t>(a.k) - n_in;
        for (uint32_t b = tid; b < band_n; b += kSelThreads) {
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
            if (lane == 0 && b) atomicOr(&sm.sel_bits[it * (kSelThreads / 32) + warp], b);
        }
        __syncthreads();
        sel::emit_bits<kSelThreads, ITEMS>(sm.sel_bits, sm.scan, out);
        return;
    }

    // fallback: exact keys for every visible row, then an exact radix select
    for (int b0 = 0; b0 < ITEMS * kSelThreads; b0 += kSelThreads / 16) {
        const int j = b0 + tid / 16;
        const uint32_t kx = exact_key16(q, a.k_idx + static_cast<size_t>(j < n ? j : 0) * a.d_idx, a.d_idx, j < n);
        if (j < n && (tid & 15) == 0) reinterpret_cast<uint32_t *>(row)[j] = kx;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * kSelThreads + tid;
        key[it] = j < n ? reinterpret_cast<const uint32_t *>(row)[j] : 0u;
    }
    const bool all_eq = sel::find_threshold<kSelThreads, ITEMS>(key, n, a.k, sm.hist, sm.scan, sm.res, prefix, mask, kk);
    sel::emit_topk_bits<kSelThreads, ITEMS>(key, n, prefix, mask, kk, all_eq, sm.cnt, sm.sel_bits, sm.scan, out);
}

constexpr int kSelNT = 256, kSelMinBlocks = 4;   // threads per query, CTAs per SM (<= 64 registers)

template <int DI>
constexpr size_t gemm_smem() { return (DI / 64) * (kTM + 2 * kTN) * 128 + 1024; }

}  // namespace

bool indexer_prefill_tc_ok(int n_q, long long n_rows, int d_idx) {
    return n_q >= 64 && (d_idx == 64 || d_idx == 128) && n_rows <= kSelMaxRows;
}

size_t indexer_prefill_tc_ws_bytes(int n_q, long long n_rows) {
    const long long ld = (n_rows + kTN - 1) / kTN * kTN;
    return 256 + static_cast<size_t>(n_q) * ld * sizeof(float);
}

cudaError_t launch_indexer_prefill_tc(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                                      int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                                      int32_t *out_n, void *ws, const Ctx &c) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_scores_tc_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(gemm_smem<64>()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(indexer_scores_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(gemm_smem<128>()));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int ld = static_cast<int>((n_rows + kTN - 1) / kTN * kTN);
    // workspace: 256-byte header holding the tile norms (<= 32 tiles), then the scores
    float *tile_kmax2 = static_cast<float *>(ws);
    float *scores = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) + 256);
    TcScoreArgs g;
    g.q_idx = q_idx;
    g.k_idx = k_idx;
    g.scores = scores;
    g.tile_kmax2 = tile_kmax2;
    g.err = c.err;
    g.n_rows = n_rows;
    g.early_rows = q_pos0 / ratio;
    g.n_q = n_q;
    g.ld = ld;
    g.n_ntiles = ld / kTN;
    const int n_mtiles = (n_q + kTM - 1) / kTM;
    g.n_split = c.num_sms / n_mtiles;
    if (g.n_split < 1) g.n_split = 1;
    if (g.n_split > g.n_ntiles) g.n_split = g.n_ntiles;
    const dim3 grid(n_mtiles, g.n_split);
    cudaError_t e = d_idx == 128
                        ? launch(indexer_scores_tc_kernel<128>, grid, dim3(kGemmThreads), gemm_smem<128>(), c, 1, g)
                        : launch(indexer_scores_tc_kernel<64>, grid, dim3(kGemmThreads), gemm_smem<64>(), c, 1, g);
    if (e != cudaSuccess) return e;
    SelArgs s{q_idx, k_idx, scores, tile_kmax2, out_idx, out_n, n_rows, q_pos0, d_idx, ratio, k, ld};
    const long long n_max = n_rows;
    if (n_max <= 8 * kSelNT) return launch(indexer_select_kernel<kSelNT, 8, kSelMinBlocks>, dim3(n_q), dim3(kSelNT), 0, c, 1, s);
    if (n_max <= 16 * kSelNT) return launch(indexer_select_kernel<kSelNT, 16, kSelMinBlocks>, dim3(n_q), dim3(kSelNT), 0, c, 1, s);
    return launch(indexer_select_kernel<kSelNT, kSelMaxRows / kSelNT, kSelMinBlocks>, dim3(n_q), dim3(kSelNT), 0, c, 1, s);
}

}  // namespace ds4a
