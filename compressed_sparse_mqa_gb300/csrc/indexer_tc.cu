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
constexpr int kGemmThreads = 256;   // two warps per TMEM lane quadrant

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
    // Epilogue: lane l of warp w holds query row 32 (w % 4) + l, columns of part w / 4.  Each 32 x 32 block goes
    // through a padded shared tile so that a store instruction writes 128-byte runs
    // of four rows instead of 16 bytes of 32 rows.
    constexpr int kColParts = kGemmThreads / 128;   // warps sharing a TMEM lane quadrant
    constexpr int kPartCols = kTN / kColParts;
    const int quad = warp & 3, cpart = warp >> 2;
    auto epilogue = [&](int it) {
        const int buf = it & 1;
        if (!tc::mbar_wait(&s_bar[buf], (it >> 1) & 1)) ok = false;
        tc::fence_after_sync();
        const long long col0 = static_cast<long long>(ns + it * a.n_split) * kTN;
        float *stg = s_stage[warp];
#pragma unroll 1
        for (int c0 = cpart * kPartCols; c0 < (cpart + 1) * kPartCols; c0 += 32) {
            uint32_t r[16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc::ld_x16(tmem + (static_cast<uint32_t>(quad * 32) << 16) + buf * kTN + c0 + 16 * h, r);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[lane * 33 + 16 * h + j] = __uint_as_float(r[j]);
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = 4 * k + (lane >> 3), cg = 4 * (lane & 7);
                const int q = m0 + quad * 32 + row;
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

template <int NT, int ITEMS, int MIN_BLOCKS>
__global__ void __launch_bounds__(NT, MIN_BLOCKS) indexer_select_kernel(SelArgs a) {
    constexpr int kSelThreads = NT;
    __shared__ sel::BandSmem<NT, kSelMaxRows> sm;
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
    sel::band_select<kSelThreads, ITEMS>(key, n, a.k, sm.eps, q, a.k_idx, a.d_idx, sm,
                                         reinterpret_cast<uint32_t *>(row), out);
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
