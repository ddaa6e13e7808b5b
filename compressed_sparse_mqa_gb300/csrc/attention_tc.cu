// attention_tc.cu -- prefill attention on the 5th-generation tensor cores.
//
// "DS4 (DwarfStar 4)", Architecture (64 query heads share one KV head, 128-token
// window) and Key Techniques, "KV attention compression" (one softmax over the
// raw window and the kept compressed rows): for query i and head h,
//   o_h = sum_j softmax_j(scale * q_h . K_j) V_j
// over the query's own key set (its window rows, then its selected rows).
//
// Because each query has its own key set, the 64 heads of one query are the only
// operand that is shared by all its keys.  The kernel therefore puts the KEYS on
// the 128-row M side of tcgen05.mma and the heads on N = 64:
//   S^T[key][head] = K[key][:] . Q[head][:]       (A = K tile, K-major; B = Q, K-major)
//   O^T[d][head]  += sum_key V[key][d] P^T[key][head]   (A = V tile, MN-major; B = P^T, MN-major)
// so both products run as M = 128 tiles.
//
// A query's key list is tile-aligned: its window tiles (raw rows), then its
// compressed-row tiles, each padded with zero rows.
//
// Warp roles (one persistent CTA per SM, each taking a contiguous block of queries;
// registers are rebalanced with setmaxnreg: 128 for softmax, 56 for the rest):
//   warps 0-7    softmax + epilogue: warp w reads TMEM lane quadrant w%4 (keys)
//                and heads 32*(w/4) .. +31; each warp keeps the running
//                references of its 32 heads in shared memory.  Per tile: x = s*scale - m
//                for its 32 scores, and one barrier-reduction per head half asks
//                whether any x exceeds 8 (log2 units); only then is the exact
//                tile max taken (redux.sync, then the 4 quadrants through shared
//                memory) and O^T in TMEM rescaled.  P^T (fp16) goes to one of two
//                shared buffers.  Per query: the per-head sums, then O^T / l from
//                TMEM to the output.
//   warp 8       row tables: the 32 lanes resolve the row of every key slot of
//                the next query (window rows, then sel entries) into one of two
//                shared tables, with a validity bit per slot.
//   warp 9       MMA issuer (one thread): S^T_0, S^T_1, then S^T_(c+2) (into the
//                TMEM buffer the softmax has just read S^T_c from) and
//                O^T += V^T_c P^T_c for each tile c; tcgen05.commit releases ring
//                stages and signals the softmax warps.
//   warps 10-23  TMA producers: fill a 5-stage ring of 128-byte-swizzled 32 KB
//                tiles in the order the MMAs consume them: K0, K1, K2, V0, K3,
//                V1, ..., V(n-2), V(n-1).  A tile of scattered rows is 64 tile::gather4 loads
//                (4 rows x 128 B each) shared out over the 14 warps -- a TMA
//                instruction holds its issuing warp for a while, so the gather
//                rate grows with the number of issuing warps; a full window tile
//                is two plain 2-D tile loads.  The query block Q rides with K0.
//                Completion is counted in bytes on each stage's mbarrier.
// All hand-offs are mbarriers with time-bounded waits; a wait that gives up
// records DS4A_ERR_TIMEOUT.  Warps that share a named barrier never leave their
// loops early: after a failed wait they skip the work but keep the structure.
#include <cuda.h>

#include "ds4a_common.cuh"
#include "ds4a_internal.h"
#include "tcgen05.cuh"

namespace ds4a {
namespace {

constexpr int kH = 64;                      // heads (MMA N)
constexpr int kD = 128;                     // head dim
constexpr int kTK = 128;                    // keys per tile (MMA M)
constexpr int kMaxTiles = 6;                // tiles per query
constexpr int kNS = 5;                      // ring stages
constexpr int kSoftWarps = 8;
constexpr int kTblWarp = kSoftWarps;        // row tables
constexpr int kMmaWarp = kTblWarp + 1;
constexpr int kIssWarp0 = kMmaWarp + 1;     // first TMA producer warp
constexpr int kIss = 14;                    // TMA producer warps
constexpr int kWarps = kIssWarp0 + kIss;    // 24 = 6 warpgroups
constexpr int kThreads = 32 * kWarps;
constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;   // 80
constexpr int kSoftRegs = 128, kOtherRegs = 56;
constexpr int kTileBytes = kTK * kD * 2;    // 32 KB: [2 atoms][128 rows][128 B]
constexpr int kQBytes = kH * kD * 2;        // 16 KB: [2 atoms][64 rows][128 B]
constexpr int kPBytes = kTK * kH * 2;       // 16 KB: [128 key rows][128 B]
constexpr int kGathers = kTK / 4 * 2;       // gather4 loads per tile (row groups x atom halves)
constexpr int kMaskWords = kMaxTiles * 4;   // validity bits per query, 32 slots a word
constexpr uint32_t kTmemCols = 256;         // S0 | S1 | O0 | O1, 64 columns each
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;             // lazy rescale threshold (log2 units)

static_assert(kWarps % 4 == 0 && kSoftWarps % 4 == 0, "the register split is per warpgroup");
static_assert(kSoftWarps * kSoftRegs + (kWarps - kSoftWarps) * kOtherRegs <= kWarps * kLaunchRegs,
              "the register split exceeds what the block is launched with");

struct Bars {
    uint64_t full[kNS], empty[kNS];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t q_empty;
    uint64_t tbl_full[2], tbl_empty[2];
};

struct SmemLayout {
    static constexpr int q = 0;
    static constexpr int p = q + kQBytes;                               // 2 buffers
    static constexpr int ring = p + 2 * kPBytes;
    static constexpr int tbl = ring + kNS * kTileBytes;                 // int [2][768] gather rows
    static constexpr int mask = tbl + 2 * kMaxTiles * kTK * 4;          // uint32 [2][24] slot validity
    static constexpr int red = mask + 2 * kMaskWords * 4;               // float [4][64] max, [4][64] sum, [64] 1/l
    static constexpr int bars = red + (2 * 4 * kH + kH) * 4;
    static constexpr int end = bars + static_cast<int>(sizeof(Bars));
};
constexpr size_t kSmemBytes = SmemLayout::end + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct Args {
    CUtensorMap map_raw_k, map_raw_v, map_comp_k, map_comp_v;   // one-row boxes (gathers)
    CUtensorMap map_win_k, map_win_v;                           // 128-row boxes (window tiles)
    CUtensorMap map_q;                                          // 64-row boxes
    const int32_t *sel;
    uint16_t *out;
    unsigned int *err;
    int n_comp;      // compressed rows (< 2^31 - 1)
    long long q_pos0;
    int n_raw;       // rows of the raw maps (n_prior + T): the zero-fill row
    int comp_oob;    // rows of the compressed maps: the zero-fill row
    int T;
    int n_prior;
    int window;
    int k_stride;
    int ratio;
    float scale_log2;
};

DS4A_DEVINL void ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
DS4A_DEVINL void st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
DS4A_DEVINL void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

DS4A_DEVINL void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(bar)) : "memory");
}
// named barriers 1 and 2: the four softmax warps of one head half (128 threads)
DS4A_DEVINL void half_barrier(int half) { asm volatile("bar.sync %0, 128;\n" ::"r"(1 + half) : "memory"); }
// the same barrier, returning whether any of the 128 threads passed pred = true
DS4A_DEVINL bool half_any(int half, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(1 + half)
        : "memory");
    return r != 0;
}
template <int N> DS4A_DEVINL void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <int N> DS4A_DEVINL void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }

// 2^x with the hardware approximation (flush-to-zero): the softmax numerators
// are rounded to fp16 right after, far coarser than its error
DS4A_DEVINL float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// lane l receives the max over the warp's 32 lanes of v[l] (see transpose_sum32)
DS4A_DEVINL float transpose_max32(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, s));
        }
    }
    return v[0];
}

// lane l receives the sum over the warp's 32 lanes of v[l] (a butterfly that
// halves the live values at each step: 31 shuffles in all)
DS4A_DEVINL float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

DS4A_DEVINL void expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(tc::smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// 2-D TMA tile load (x = column, y = row) completing on bar
DS4A_DEVINL void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(tc::smem_u32(dst)),
                 "l"(map), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
                 : "memory");
}
// four rows r.x .. r.w, columns x .. x+63, to 4 consecutive 128-byte rows at dst
DS4A_DEVINL void tma_gather4(uint32_t dst, const CUtensorMap *map, int x, int4 r, uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
                 "l"(map), "r"(x), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w), "r"(tc::smem_u32(bar))
                 : "memory");
}
DS4A_DEVINL void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(map) : "memory");
}

// The key list of query i: its window rows padded to whole tiles, then its
// compressed rows padded to whole tiles.
struct QueryKeys {
    int raw0;         // raw index of the first window row
    int n_w;          // window rows
    int n_sel;        // compressed-row slots
    int n_wt;         // window tiles
    int n_tiles;      // window tiles + compressed-row tiles
};
DS4A_DEVINL QueryKeys query_keys(const Args &a, int i) {
    QueryKeys k;
    const long long p = a.q_pos0 + i;
    const long long first = p - a.window + 1 > 0 ? p - a.window + 1 : 0;
    k.raw0 = static_cast<int>(first - (a.q_pos0 - a.n_prior));
    k.n_w = static_cast<int>(p - first + 1);
    k.n_sel = 0;
    if (a.ratio > 0) {
        if (a.sel) k.n_sel = a.k_stride;
        else {
            const long long nv = (p + 1) / a.ratio;
            k.n_sel = static_cast<int>(nv < a.n_comp ? nv : static_cast<long long>(a.n_comp));
        }
    }
    k.n_wt = (k.n_w + kTK - 1) / kTK;
    k.n_tiles = k.n_wt + (k.n_sel + kTK - 1) / kTK;
    return k;
}
// ring event e (0 .. 2n-1) of a query with n tiles, in the order the MMAs take
// them: K0, K1, then K(c+2), V(c) for c = 0 .. n-3, then V(n-2), V(n-1)
DS4A_DEVINL void ring_event(int e, int n, bool &is_v, int &tile) {
    if (e == 2 * n - 1) { is_v = true; tile = n - 1; }
    else if (e == 2 * n - 2 && n >= 2) { is_v = true; tile = n - 2; }
    else if (e < 2) { is_v = false; tile = e; }
    else if (e & 1) { is_v = true; tile = (e - 2) / 2; }
    else { is_v = false; tile = (e - 2) / 2 + 2; }
}


__global__ void __launch_bounds__(kThreads, 1) attn_prefill_tc_kernel(const __grid_constant__ Args a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *q_s = smem + SmemLayout::q;
    unsigned char *p_s = smem + SmemLayout::p;
    unsigned char *ring = smem + SmemLayout::ring;
    int *tbl = reinterpret_cast<int *>(smem + SmemLayout::tbl);
    uint32_t *mask = reinterpret_cast<uint32_t *>(smem + SmemLayout::mask);
    float *red_max = reinterpret_cast<float *>(smem + SmemLayout::red);   // [4][64]
    float *red_sum = red_max + 4 * kH;                                    // [4][64]
    float *red_inv = red_sum + 4 * kH;                                    // [64]
    Bars &bar = *reinterpret_cast<Bars *>(smem + SmemLayout::bars);
    __shared__ uint32_t s_tmem;
    __shared__ __align__(16) float s_alpha[kSoftWarps][32];
    __shared__ __align__(16) float s_mh[kSoftWarps][32];   // running reference per head (log2 units)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(&bar.full[s], kIss);
            tc::mbar_init(&bar.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bar.s_full[b], 1);
            tc::mbar_init(&bar.s_empty[b], kSoftWarps);
            tc::mbar_init(&bar.p_full[b], kSoftWarps);
            tc::mbar_init(&bar.p_empty[b], 1);
            tc::mbar_init(&bar.o_full[b], 1);
            tc::mbar_init(&bar.o_empty[b], kSoftWarps);
            tc::mbar_init(&bar.tbl_full[b], 32);
            tc::mbar_init(&bar.tbl_empty[b], kIss + kSoftWarps);
        }
        tc::mbar_init(&bar.q_empty, 1);
        tc::mbar_fence_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    // each CTA takes a contiguous block of queries: CTAs running side by side then
    // read windows spread over the whole chunk instead of the same few rows
    const int per_cta = (a.T + gridDim.x - 1) / gridDim.x;
    const int q_begin = blockIdx.x * per_cta;
    const int q_end = min(a.T, q_begin + per_cta);
    pdl_wait();
    pdl_trigger();
    bool ok = true;
    // a failed wait records the failure; later waits of this thread return at once
    auto wait = [&](uint64_t *b, uint32_t parity) {
        if (ok && !tc::mbar_wait(b, parity)) ok = false;
        return ok;
    };

    if (warp < kSoftWarps) {
        setmaxnreg_inc<kSoftRegs>();
        // ---------------- softmax + epilogue (warps 0-7) ----------------
        const int quad = warp & 3, half = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float c2 = a.scale_log2;
        uint32_t gs = 0, gp = 0;
        int t = 0;
        for (int i = q_begin; i < q_end; ++i, ++t) {
            const QueryKeys k = query_keys(a, i);
            const int n = k.n_tiles;
            const uint32_t obuf = static_cast<uint32_t>(t & 1);
            // validity of this warp's 32 keys in each tile, from the row table's bits
            const int b = t & 1;
            wait(&bar.tbl_full[b], static_cast<uint32_t>(t >> 1) & 1u);
            uint32_t vbits = 0;
            for (int c = 0; c < n; ++c) vbits |= ((mask[b * kMaskWords + c * 4 + quad] >> lane) & 1u) << c;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.tbl_empty[b]);
            float l_lane[32];   // this lane's key: partial softmax sums of the 32 heads
#pragma unroll
            for (int h = 0; h < 32; ++h) l_lane[h] = 0.f;
            float *mh = s_mh[warp];   // this warp's copy of the references of its 32 heads
            mh[lane] = -INFINITY;
            __syncwarp();
            for (int c = 0; c < n; ++c) {
                const uint32_t sb = static_cast<uint32_t>(gs & 1);
                wait(&bar.s_full[sb], static_cast<uint32_t>(gs >> 1) & 1u);
                tc::fence_after_sync();
                uint32_t r[32];
                ld_x32(tmem + lane_base + kColS + sb * kH + half * 32, r);
                tc::wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.s_empty[sb]);
                const bool valid = (vbits >> c) & 1u;
                float mx = -INFINITY;
#pragma unroll
                for (int h4 = 0; h4 < 8; ++h4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(mh + h4 * 4);
                    mx = fmaxf(mx, fmaf(__uint_as_float(r[h4 * 4 + 0]), c2, -m4.x));
                    mx = fmaxf(mx, fmaf(__uint_as_float(r[h4 * 4 + 1]), c2, -m4.y));
                    mx = fmaxf(mx, fmaf(__uint_as_float(r[h4 * 4 + 2]), c2, -m4.z));
                    mx = fmaxf(mx, fmaf(__uint_as_float(r[h4 * 4 + 3]), c2, -m4.w));
                }
                if (!valid) mx = -INFINITY;
                if (half_any(half, mx > kRescale)) {
                    // Some head grew past its reference: the exact tile max of each head
                    // over the 128 keys.  A transposing butterfly leaves lane l with the
                    // max of head l over this warp's 32 keys; the 4 quadrants meet in
                    // shared memory; lane l then updates the reference of head l.
                    float v[32];
#pragma unroll
                    for (int h = 0; h < 32; ++h) v[h] = valid ? __uint_as_float(r[h]) : -INFINITY;
                    red_max[quad * kH + half * 32 + lane] = transpose_max32(v, lane);
                    half_barrier(half);
                    float tm = red_max[half * 32 + lane];
#pragma unroll
                    for (int qd = 1; qd < 4; ++qd) tm = fmaxf(tm, red_max[qd * kH + half * 32 + lane]);
                    const float target = tm * c2;   // scale > 0: the max commutes with it
                    const float old = mh[lane];
                    float alpha = 1.f;
                    if (old == -INFINITY) {
                        mh[lane] = target;
                        alpha = 0.f;   // nothing accumulated yet
                    } else if (target > old + kRescale) {
                        alpha = ex2(old - target);
                        mh[lane] = target;
                    }
                    s_alpha[warp][lane] = alpha;
                    const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
                    __syncwarp();
                    if (rescale) {
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const float4 al = *reinterpret_cast<const float4 *>(&s_alpha[warp][h4 * 4]);
                            l_lane[h4 * 4 + 0] *= al.x;
                            l_lane[h4 * 4 + 1] *= al.y;
                            l_lane[h4 * 4 + 2] *= al.z;
                            l_lane[h4 * 4 + 3] *= al.w;
                        }
                    }
                    if (c > 0 && rescale) {
                        // O^T holds the earlier tiles once the previous PV is done
                        wait(&bar.p_empty[(gp - 1) & 1], static_cast<uint32_t>((gp - 1) >> 1) & 1u);
                        tc::fence_after_sync();
#pragma unroll
                        for (int part = 0; part < 2; ++part) {   // 16 columns at a time
                            uint32_t o[16];
                            const uint32_t oa = tmem + lane_base + kColO + obuf * kH + half * 32 + part * 16;
                            tc::ld_x16(oa, o);
                            tc::wait_ld();
#pragma unroll
                            for (int h4 = 0; h4 < 4; ++h4) {
                                const float4 al = *reinterpret_cast<const float4 *>(&s_alpha[warp][part * 16 + h4 * 4]);
                                o[h4 * 4 + 0] = __float_as_uint(__uint_as_float(o[h4 * 4 + 0]) * al.x);
                                o[h4 * 4 + 1] = __float_as_uint(__uint_as_float(o[h4 * 4 + 1]) * al.y);
                                o[h4 * 4 + 2] = __float_as_uint(__uint_as_float(o[h4 * 4 + 2]) * al.z);
                                o[h4 * 4 + 3] = __float_as_uint(__uint_as_float(o[h4 * 4 + 3]) * al.w);
                            }
                            st_x16(oa, o);
                        }
                        wait_st();
                    }
                }
                // p = 2^(s * scale - m) -> the P^T row (key) of this lane, 32 heads
                uint32_t pk[16];
#pragma unroll
                for (int h4 = 0; h4 < 8; ++h4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(mh + h4 * 4);
                    const float m[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                    for (int u = 0; u < 4; u += 2) {
                        const int h = h4 * 4 + u;
                        const float p0 = valid ? ex2(fmaf(__uint_as_float(r[h]), c2, -m[u])) : 0.f;
                        const float p1 = valid ? ex2(fmaf(__uint_as_float(r[h + 1]), c2, -m[u + 1])) : 0.f;
                        l_lane[h] += p0;
                        l_lane[h + 1] += p1;
                        pk[h / 2] = pack_half2(p0, p1);
                    }
                }
                const uint32_t pb = static_cast<uint32_t>(gp & 1);
                // the PV two tiles back has finished with this P buffer
                if (gp >= 2) wait(&bar.p_empty[pb], static_cast<uint32_t>((gp >> 1) - 1) & 1u);
                unsigned char *pbuf = p_s + pb * kPBytes;
                const int key = quad * 32 + lane;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int ch = half * 4 + q4;
                    *reinterpret_cast<uint4 *>(pbuf + key * 128 + ((ch ^ (key & 7)) << 4)) =
                        make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[pb]);
                ++gs;
                ++gp;
            }
            // ---- per-head sums, then O^T / l to the output ----
            const float part = transpose_sum32(l_lane, lane);   // head half*32 + lane, this warp's keys
            red_sum[quad * kH + half * 32 + lane] = part;
            half_barrier(half);
            float lsum = red_sum[half * 32 + lane];
#pragma unroll
            for (int qd = 1; qd < 4; ++qd) lsum += red_sum[qd * kH + half * 32 + lane];
            if (quad == 0) red_inv[half * 32 + lane] = 1.f / lsum;
            half_barrier(half);
            wait(&bar.o_full[obuf], static_cast<uint32_t>(t >> 1) & 1u);
            tc::fence_after_sync();
            uint32_t o[32];
            ld_x32(tmem + lane_base + kColO + obuf * kH + half * 32, o);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_empty[obuf]);
            // Stage the warp's 32 heads x 32 d through the part of the P buffer that
            // only this warp writes (rows 32*quad .., bytes 64*half ..; every PV of the
            // query has finished with it), then write 16 bytes per lane.
            unsigned char *stg = p_s + (gp & 1) * kPBytes;
            auto stg_chunk = [&](int h, int c16) {   // 16-byte chunk c16 (0..3) of head h's 64 bytes
                const int key = quad * 32 + h;
                return stg + key * 128 + (((half * 4 + c16) ^ (key & 7)) << 4);
            };
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
                const float4 iv = *reinterpret_cast<const float4 *>(red_inv + half * 32 + h4 * 4);
                const float inv[4] = {iv.x, iv.y, iv.z, iv.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint16_t *>(stg_chunk(h4 * 4 + u, lane >> 3) + (lane & 7) * 2) =
                        f2h(__uint_as_float(o[h4 * 4 + u]) * inv[u]);
            }
            __syncwarp();
            uint16_t *dst = a.out + (static_cast<size_t>(i) * kH + half * 32) * kD + quad * 32;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int h = k4 * 8 + (lane >> 2), c16 = lane & 3;
                *reinterpret_cast<uint4 *>(dst + h * kD + c16 * 8) = *reinterpret_cast<const uint4 *>(stg_chunk(h, c16));
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_dec<kOtherRegs>();
        // one lane waits for the warp, so that warp-wide steps stay converged
        auto warp_wait = [&](uint64_t *b, uint32_t parity) {
            bool r = true;
            if (lane == 0) r = wait(b, parity);
            r = __shfl_sync(0xffffffffu, r, 0);
            ok = ok && r;
            return r;
        };
        if (warp == kTblWarp) {
            // ---------------- row tables (double-buffered, one query each) ----------------
            // The sel entries of a query come in as int4 (four slots a lane), every
            // load in flight before any is used; the validity bits are then read
            // back from the finished table.
            constexpr int kVec = kMaxTiles * kTK / 4 / 32;
            int t = 0;
            for (int i = q_begin; i < q_end; ++i, ++t) {
                const int b = t & 1;
                if (t >= 2 && !warp_wait(&bar.tbl_empty[b], static_cast<uint32_t>((t >> 1) - 1) & 1u)) continue;
                const QueryKeys k = query_keys(a, i);
                int *tb = tbl + b * (kMaxTiles * kTK);
                uint32_t *mk = mask + b * kMaskWords;
                const int w_slots = k.n_wt * kTK;   // window slots
                const int n_slots = k.n_tiles * kTK;
                const int32_t *sp = a.sel ? a.sel + static_cast<size_t>(i) * a.k_stride : nullptr;
                const bool vec = sp && (reinterpret_cast<uintptr_t>(sp) & 15) == 0 && (k.n_sel & 3) == 0;
                int4 v[kVec];
#pragma unroll
                for (int m = 0; m < kVec; ++m) {
                    const int w = (lane + 32 * m) * 4;   // first of this lane's four compressed slots
                    if (sp && w < k.n_sel) {
                        if (vec) {
                            v[m] = __ldg(reinterpret_cast<const int4 *>(sp + w));
                        } else {
                            v[m].x = __ldg(sp + w);
                            v[m].y = w + 1 < k.n_sel ? __ldg(sp + w + 1) : -1;
                            v[m].z = w + 2 < k.n_sel ? __ldg(sp + w + 2) : -1;
                            v[m].w = w + 3 < k.n_sel ? __ldg(sp + w + 3) : -1;
                        }
                    } else {
                        v[m] = make_int4(w, w + 1, w + 2, w + 3);   // no sel: the visible rows in order
                    }
                }
                // window slots: consecutive raw rows, the zero row past the window
                for (int kx = lane; kx < w_slots; kx += 32) tb[kx] = kx < k.n_w ? k.raw0 + kx : a.n_raw;
#pragma unroll
                for (int m = 0; m < kVec; ++m) {
                    const int w = (lane + 32 * m) * 4;
                    if (w_slots + w < n_slots) {
                        const int e[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
                        int r[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const bool in_list = w + u < k.n_sel;
                            if (in_list && e[u] >= a.n_comp) record_error(a.err, DS4A_ERR_DEVICE_INDEX);
                            r[u] = in_list && e[u] >= 0 && e[u] < a.n_comp ? e[u] : a.comp_oob;
                        }
                        *reinterpret_cast<int4 *>(tb + w_slots + w) = make_int4(r[0], r[1], r[2], r[3]);
                    }
                }
                __syncwarp();
                for (int wd = 0; wd < k.n_tiles * 4; ++wd) {   // warp-uniform
                    const int kx = wd * 32 + lane;
                    const uint32_t m = __ballot_sync(0xffffffffu, tb[kx] != (kx < w_slots ? a.n_raw : a.comp_oob));
                    if (lane == 0) mk[wd] = m;
                }
                mbar_arrive(&bar.tbl_full[b]);
            }
        } else if (warp == kMmaWarp) {
            // ---------------- MMA issuer ----------------
            if (lane == 0) {
                constexpr uint32_t kIdS = tc::idesc_f16_f32(kTK, kH, false, false);
                constexpr uint32_t kIdO = tc::idesc_f16_f32(kTK, kH, true, true);
                uint32_t g = 0, gs = 0, gp = 0;
                int t = 0;
                for (int i = q_begin; i < q_end && ok; ++i, ++t) {
                    const QueryKeys k = query_keys(a, i);
                    const int n = k.n_tiles;
                    const uint32_t obuf = static_cast<uint32_t>(t & 1);
                    auto issue_pv = [&](int c) {
                        const uint32_t ev = g++;
                        const int s = static_cast<int>(ev % kNS);
                        const uint32_t pb = static_cast<uint32_t>(gp & 1);
                        wait(&bar.full[s], static_cast<uint32_t>(ev / kNS) & 1u);
                        wait(&bar.p_full[pb], static_cast<uint32_t>(gp >> 1) & 1u);
                        if (c == 0 && t >= 2) wait(&bar.o_empty[obuf], static_cast<uint32_t>((t >> 1) - 1) & 1u);
                        if (!ok) return;
                        tc::fence_after_sync();
                        const uint32_t va = tc::smem_u32(ring + s * kTileBytes);
                        const uint32_t pa = tc::smem_u32(p_s + pb * kPBytes);
#pragma unroll
                        for (int st = 0; st < kTK / 16; ++st) {
                            const uint64_t da = tc::desc_sw128(va + st * 2048, kTK * 128, 1024);
                            const uint64_t db = tc::desc_sw128(pa + st * 16 * 128, 8192, 1024);
                            tc::mma_f16(tmem + kColO + obuf * kH, da, db, kIdO, (c > 0 || st > 0) ? 1u : 0u);
                        }
                        tc::commit(&bar.p_empty[pb]);
                        tc::commit(&bar.empty[s]);
                        if (c == n - 1) tc::commit(&bar.o_full[obuf]);
                        ++gp;
                    };
                    // S^T_c = K_c Q^T into S buffer c % 2 (free once the softmax has read S_(c-2))
                    auto issue_s = [&](int c) {
                        const uint32_t ev = g++;
                        const int s = static_cast<int>(ev % kNS);
                        wait(&bar.full[s], static_cast<uint32_t>(ev / kNS) & 1u);
                        const uint32_t sb = static_cast<uint32_t>(gs & 1);
                        if (gs >= 2) wait(&bar.s_empty[sb], static_cast<uint32_t>((gs >> 1) - 1) & 1u);
                        if (!ok) return;
                        tc::fence_after_sync();
                        const uint32_t ka = tc::smem_u32(ring + s * kTileBytes), qb = tc::smem_u32(q_s);
#pragma unroll
                        for (int st = 0; st < kD / 16; ++st) {
                            const uint64_t da = tc::desc_sw128(ka + (st / 4) * (kTK * 128) + (st % 4) * 32, 16, 1024);
                            const uint64_t db = tc::desc_sw128(qb + (st / 4) * (kH * 128) + (st % 4) * 32, 16, 1024);
                            tc::mma_f16(tmem + kColS + sb * kH, da, db, kIdS, st > 0 ? 1u : 0u);
                        }
                        tc::commit(&bar.s_full[sb]);
                        tc::commit(&bar.empty[s]);
                        if (c == n - 1) tc::commit(&bar.q_empty);
                        ++gs;
                    };
                    // the scores run two tiles ahead of the PV products: S_(c+2) is on the
                    // tensor pipe while the softmax of tile c is still being computed
                    issue_s(0);
                    if (n > 1) issue_s(1);
                    for (int c = 0; c < n && ok; ++c) {
                        if (c + 2 < n) issue_s(c + 2);
                        if (ok) issue_pv(c);
                    }
                }
            }
            __syncwarp();
        } else {
            // ---------------- TMA producers (warps 10-23) ----------------
            const int j = warp - kIssWarp0;
            if (lane == 0) {
                const int u0 = j * kGathers / kIss, u1 = (j + 1) * kGathers / kIss;   // this warp's gathers
                const bool q_warp = j == 2 || j == 3;                                 // the two Q halves
                if (j == 0) {
                    prefetch_map(&a.map_q);
                    prefetch_map(&a.map_win_k);
                    prefetch_map(&a.map_win_v);
                    prefetch_map(&a.map_comp_k);
                    prefetch_map(&a.map_comp_v);
                }
                uint32_t g = 0;
                int t = 0;
                for (int i = q_begin; i < q_end && ok; ++i, ++t) {
                    const int b = t & 1;
                    const QueryKeys k = query_keys(a, i);
                    if (!wait(&bar.tbl_full[b], static_cast<uint32_t>(t >> 1) & 1u)) break;
                    const int *tb = tbl + b * (kMaxTiles * kTK);
                    for (int e = 0; e < 2 * k.n_tiles; ++e, ++g) {
                        const int s = static_cast<int>(g % kNS);
                        if (g >= kNS) wait(&bar.empty[s], static_cast<uint32_t>((g / kNS) - 1) & 1u);
                        const bool q_load = e == 0 && q_warp;
                        // the MMAs of the previous query are done with the Q block
                        if (q_load && t > 0) wait(&bar.q_empty, static_cast<uint32_t>(t - 1) & 1u);
                        if (!ok) break;
                        bool is_v;
                        int c;
                        ring_event(e, k.n_tiles, is_v, c);
                        // a window tile of 128 existing rows is contiguous: two tile loads
                        const bool win_tile = c < k.n_wt && (c + 1) * kTK <= k.n_w;
                        uint32_t bytes = q_load ? kQBytes / 2 : 0;
                        if (win_tile) bytes += j < 2 ? kTileBytes / 2 : 0;
                        else bytes += static_cast<uint32_t>(u1 - u0) * 512;
                        expect_tx(&bar.full[s], bytes);
                        unsigned char *dst = ring + s * kTileBytes;
                        if (q_load) tma_load_2d(q_s + (j - 2) * (kH * 128), &a.map_q, (j - 2) * 64, i * kH, &bar.full[s]);
                        if (win_tile) {
                            if (j < 2)
                                tma_load_2d(dst + j * (kTK * 128), is_v ? &a.map_win_v : &a.map_win_k, j * 64,
                                            k.raw0 + c * kTK, &bar.full[s]);
                        } else {
                            const CUtensorMap *map = c < k.n_wt ? (is_v ? &a.map_raw_v : &a.map_raw_k)
                                                                : (is_v ? &a.map_comp_v : &a.map_comp_k);
                            const uint32_t d0 = tc::smem_u32(dst);
                            for (int u = u0; u < u1; ++u) {
                                const int grp = u >> 1, hf = u & 1;
                                const int4 r4 = *reinterpret_cast<const int4 *>(tb + c * kTK + grp * 4);
                                tma_gather4(d0 + hf * (kTK * 128) + grp * 512, map, hf * 64, r4, &bar.full[s]);
                            }
                        }
                    }
                    // this warp's gathers of the query have taken their rows
                    mbar_arrive(&bar.tbl_empty[b]);
                }
            }
            __syncwarp();
        }
    }
    if (!ok) record_error(a.err, DS4A_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's tensor-map encoder, looked up once through the runtime
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// rows x 128 fp16 values, row-major; boxes of 64 columns x box_rows rows, 128-byte swizzle
bool encode_rows(CUtensorMap *m, const uint16_t *ptr, long long rows, uint32_t box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t box[2] = {64, box_rows}, es[2] = {1, 1};
    return encode_tiled()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_prefill_tc_ok(const uint16_t *q, const uint16_t *out, int T, int H, int D, int n_prior, int window,
                        long long max_sel, long long n_comp) {
    const long long tiles = (window + kTK - 1) / kTK + (max_sel + kTK - 1) / kTK;
    // TMA needs 16-byte aligned bases, the output is written 16 bytes at a time;
    // row coordinates are 32-bit
    return H == kH && D == kD && tiles <= kMaxTiles && (reinterpret_cast<uintptr_t>(q) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
           static_cast<long long>(n_prior) + T < (1LL << 31) - 1 && n_comp < (1LL << 31) - 1 &&
           static_cast<long long>(T) * kH < (1LL << 31) && encode_tiled() != nullptr;
}

cudaError_t launch_attn_prefill_tc(const uint16_t *q, int T, const uint16_t *raw_k, const uint16_t *raw_v,
                                   int n_prior, int window, const uint16_t *comp_k, const uint16_t *comp_v,
                                   long long n_comp, const int32_t *sel, int k_stride, long long q_pos0,
                                   int ratio, float scale, uint16_t *out, const Ctx &c) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    Args a{};
    const long long n_raw = static_cast<long long>(n_prior) + T;
    // with no compressed rows the compressed maps alias the raw ones and every slot reads the zero row
    const bool has_comp = n_comp > 0 && comp_k && comp_v;
    const long long comp_rows = has_comp ? n_comp : n_raw;
    if (!encode_rows(&a.map_q, q, static_cast<long long>(T) * kH, kH) ||
        !encode_rows(&a.map_raw_k, raw_k, n_raw, 1) || !encode_rows(&a.map_raw_v, raw_v, n_raw, 1) ||
        !encode_rows(&a.map_win_k, raw_k, n_raw, kTK) || !encode_rows(&a.map_win_v, raw_v, n_raw, kTK) ||
        !encode_rows(&a.map_comp_k, has_comp ? comp_k : raw_k, comp_rows, 1) ||
        !encode_rows(&a.map_comp_v, has_comp ? comp_v : raw_v, comp_rows, 1))
        return cudaErrorInvalidValue;
    a.sel = sel;
    a.out = out;
    a.err = c.err;
    a.n_comp = has_comp ? static_cast<int>(n_comp) : 0;
    a.q_pos0 = q_pos0;
    a.n_raw = static_cast<int>(n_raw);
    a.comp_oob = static_cast<int>(comp_rows);
    a.T = T;
    a.n_prior = n_prior;
    a.window = window;
    a.k_stride = k_stride;
    a.ratio = ratio;
    a.scale_log2 = scale * kLog2e;
    const int grid = T < c.num_sms ? T : c.num_sms;
    return launch(attn_prefill_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, c, 1, a);
}

}  // namespace ds4a
