constexpr long long kWinTag = 1LL << 62;
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
// Warp roles (one persistent CTA per SM, each taking a contiguous block of queries):
//   warps 8-10  producers: gather the key/value rows of each 128-key tile with
//               16-byte cp.async into a 5-stage ring of 128-byte-swizzled tiles
//               (about 160 KB in flight), in the order the MMAs consume them:
//               K0, K1, V0, K2, V1, ..., V(n-1); the query block Q rides with K0.
//               Each producer warp moves a third of every tile.
//   warp 11     MMA issuer (one thread): S^T_c into one of two TMEM buffers, then
//               O^T += V^T_(c-1) P^T_(c-1); tcgen05.commit releases ring stages
//               and signals the softmax warps.
//   warps 0-7   softmax + epilogue: warp w reads TMEM lane quadrant w%4 (keys)
//               and heads 32*(w/4) .. +31.  Per tile: the per-head max across
//               the 128 lanes (redux.sync on order-preserving keys, then the 4
//               quadrants through shared memory), a lazy online softmax (O^T in
//               TMEM is rescaled only when a head's max grows by more than 2^8),
//               P^T (fp16) to shared memory.  Per query: the per-head sums, then
//               O^T / l from TMEM to the output.
// All hand-offs are mbarriers with time-bounded waits; a wait that gives up
// records DS4A_ERR_TIMEOUT.  Warps that share a named barrier never leave their
// loops early: after a failed wait they skip the work but keep the structure.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"
#include "tcgen05.cuh"

namespace ds4a {
namespace {

constexpr int kH = 64;                      // heads (MMA N)
constexpr int kD = 128;                     // head dim
constexpr int kTK = 128;                    // keys per tile (MMA M)
constexpr int kMaxTiles = 6;                // keys per query <= 768
constexpr int kNS = 5;                      // ring stages
constexpr int kLag = kNS - 2;               // stages issued ahead of the oldest retired one
constexpr int kSoftWarps = 8;
constexpr int kProdWarps = 3;
constexpr int kProdWarp = 8;                // first producer warp
constexpr int kMmaWarp = kProdWarp + kProdWarps;
constexpr int kThreads = 32 * (kSoftWarps + kProdWarps + 1);
constexpr int kTileBytes = kTK * kD * 2;    // 32 KB: [2 atoms][128 rows][128 B]
constexpr int kQBytes = kH * kD * 2;        // 16 KB: [2 atoms][64 rows][128 B]
constexpr int kPBytes = kTK * kH * 2;       // 16 KB: [128 key rows][128 B]
constexpr uint32_t kTmemCols = 256;         // S0 | S1 | O0 | O1, 64 columns each
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;             // lazy rescale threshold (log2 units)

struct Bars {
    uint64_t full[kNS], empty[kNS];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, p_empty;
    uint64_t o_full[2], o_empty[2];
    uint64_t q_empty;
};

struct SmemLayout {
    static constexpr int q = 0;
    static constexpr int p = q + kQBytes;
    static constexpr int ring = p + kPBytes;
    static constexpr int tbl = ring + kNS * kTileBytes;                 // long long [768]
    static constexpr int red = tbl + kMaxTiles * kTK * 8;               // float [2][4][64] max, [4][64] sum
    static constexpr int bars = red + 3 * 4 * kH * 4;
    static constexpr int end = bars + static_cast<int>(sizeof(Bars));
};
constexpr size_t kSmemBytes = SmemLayout::end + 1024;

struct Args {
    const uint16_t *q;
    const uint16_t *raw_k;
    const uint16_t *raw_v;
    const uint16_t *comp_k;
    const uint16_t *comp_v;
    const int32_t *sel;
    uint16_t *out;
    unsigned int *err;
    long long n_comp;
    long long q_pos0;
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
DS4A_DEVINL void st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
DS4A_DEVINL void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

DS4A_DEVINL uint32_t redux_max_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;\n" : "=r"(r) : "r"(v));
    return r;
}
DS4A_DEVINL float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
DS4A_DEVINL void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(bar)) : "memory");
}
DS4A_DEVINL void softmax_barrier() { asm volatile("bar.sync 1, %0;\n" ::"n"(kSoftWarps * 32) : "memory"); }
DS4A_DEVINL void producer_barrier() { asm volatile("bar.sync 2, %0;\n" ::"n"(kProdWarps * 32) : "memory"); }

// The key list of query i: its window rows, then its compressed rows.
struct QueryKeys {
    long long raw0;   // raw index of the first window row
    int n_w;
    int n_sel;
    int n_tiles;
};
DS4A_DEVINL QueryKeys query_keys(const Args &a, int i) {
    QueryKeys k;
    const long long p = a.q_pos0 + i;
    const long long first = p - a.window + 1 > 0 ? p - a.window + 1 : 0;
    k.raw0 = first - (a.q_pos0 - a.n_prior);
    k.n_w = static_cast<int>(p - first + 1);
    k.n_sel = 0;
    if (a.ratio > 0) {
        if (a.sel) k.n_sel = a.k_stride;
        else {
            const long long nv = (p + 1) / a.ratio;
            k.n_sel = static_cast<int>(nv < a.n_comp ? nv : a.n_comp);
        }
    }
    k.n_tiles = (k.n_w + k.n_sel + kTK - 1) / kTK;
    return k;
}
// element offset of key kx's row (window rows tagged), -1 for padding (past the
// list, negative sel entries, or out-of-range rows, which are also recorded)
DS4A_DEVINL long long key_offset(const Args &a, int i, const QueryKeys &k, int kx, bool record) {
    if (kx < k.n_w) return kWinTag | ((k.raw0 + kx) * kD);
    if (kx >= k.n_w + k.n_sel) return -1;
    const long long j = a.sel ? static_cast<long long>(__ldg(a.sel + static_cast<size_t>(i) * a.k_stride + (kx - k.n_w)))
                              : static_cast<long long>(kx - k.n_w);
    if (j >= a.n_comp) {
        if (record) record_error(a.err, DS4A_ERR_DEVICE_INDEX);
        return -1;
    }
    return j >= 0 ? j * kD : -1;
}
// ring event e (0 .. 2n-1) of a query with n tiles: K0, K1, V0, K2, V1, ..., V(n-1)
DS4A_DEVINL void ring_event(int e, int n, bool &is_v, int &tile) {
    if (e == 0) { is_v = false; tile = 0; }
    else if (e == 2 * n - 1) { is_v = true; tile = n - 1; }
    else if (e & 1) { is_v = false; tile = (e + 1) / 2; }
    else { is_v = true; tile = e / 2 - 1; }
}

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_tc_kernel(Args a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *q_s = smem + SmemLayout::q;
    unsigned char *p_s = smem + SmemLayout::p;
    unsigned char *ring = smem + SmemLayout::ring;
    long long *tbl = reinterpret_cast<long long *>(smem + SmemLayout::tbl);
    float *red_max = reinterpret_cast<float *>(smem + SmemLayout::red);   // [2][4][64]
    float *red_sum = red_max + 2 * 4 * kH;                                // [4][64]
    Bars &bar = *reinterpret_cast<Bars *>(smem + SmemLayout::bars);
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(&bar.full[s], kProdWarps);
            tc::mbar_init(&bar.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bar.s_full[b], 1);
            tc::mbar_init(&bar.s_empty[b], kSoftWarps);
            tc::mbar_init(&bar.o_full[b], 1);
            tc::mbar_init(&bar.o_empty[b], kSoftWarps);
        }
        tc::mbar_init(&bar.p_full, kSoftWarps);
        tc::mbar_init(&bar.p_empty, 1);
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

    if (warp >= kProdWarp && warp < kMmaWarp) {
        // ---------------- producers: K/V tiles (and Q) into the ring ----------------
        const int pt = (warp - kProdWarp) * 32 + lane;   // 0 .. 95
        constexpr int kPT = kProdWarps * 32;
        long long g = 0;
        int pending = 0, t = 0;
        auto retire = [&](long long ev) {
            tc::fence_proxy_async();   // this lane's cp.async and zero stores -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.full[ev % kNS]);
        };
        for (int i = q_begin; i < q_end; ++i, ++t) {
            const QueryKeys k = query_keys(a, i);
            // the query's row table: every sel load issued before any is used
            constexpr int kPer = (kMaxTiles * kTK + kPT - 1) / kPT;
            long long offs[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int kx = pt + j * kPT;
                offs[j] = kx < k.n_tiles * kTK ? key_offset(a, i, k, kx, true) : -1;
            }
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int kx = pt + j * kPT;
                if (kx < k.n_tiles * kTK) tbl[kx] = offs[j];
            }
            producer_barrier();
            for (int e = 0; e < 2 * k.n_tiles; ++e, ++g) {
                const int s = static_cast<int>(g % kNS);
                if (g >= kNS) wait(&bar.empty[s], static_cast<uint32_t>((g / kNS) - 1) & 1u);
                bool is_v;
                int c;
                ring_event(e, k.n_tiles, is_v, c);
                if (e == 0 && t > 0) {
                    // The MMAs of the previous query need every stage issued so far:
                    // retire them all before waiting for those MMAs to free the Q block.
                    cp_async_wait<0>();
                    for (; pending > 0; --pending) retire(g - pending);
                    wait(&bar.q_empty, static_cast<uint32_t>(t - 1) & 1u);
                }
                if (!ok) continue;
                if (e == 0) {
                    for (int idx = pt; idx < kH * (kD / 8); idx += kPT) {
                        const int r = idx >> 4, ch = idx & 15;
                        cp_async16(q_s + (ch >> 3) * (kH * 128) + tc::sw128_chunk(r, ch & 7),
                                   a.q + (static_cast<size_t>(i) * kH + r) * kD + ch * 8);
                    }
                }
                unsigned char *dst = ring + s * kTileBytes;
                const uint16_t *raw = is_v ? a.raw_v : a.raw_k;
                const uint16_t *comp = is_v ? a.comp_v : a.comp_k;
                // all of this thread's sources first (table loads in flight together),
                // then the copies back to back
                constexpr int kChunksPer = (kTK * (kD / 8) + kPT - 1) / kPT;
                const uint16_t *src[kChunksPer];
#pragma unroll
                for (int j = 0; j < kChunksPer; ++j) {
                    const int idx = pt + j * kPT;
                    src[j] = nullptr;
                    if (idx < kTK * (kD / 8)) {
                        const int r = idx >> 4, ch = idx & 15;
                        const long long o = tbl[c * kTK + r];
                        if (o >= 0) src[j] = (o & kWinTag) ? raw + ((o & ~kWinTag) + ch * 8) : comp + (o + ch * 8);
                    }
                }
#pragma unroll
                for (int j = 0; j < kChunksPer; ++j) {
                    const int idx = pt + j * kPT;
                    if (idx < kTK * (kD / 8)) {
                        const int r = idx >> 4, ch = idx & 15;
                        unsigned char *d = dst + (ch >> 3) * (kTK * 128) + tc::sw128_chunk(r, ch & 7);
                        if (src[j]) cp_async16(d, src[j]);
                        else *reinterpret_cast<uint4 *>(d) = make_uint4(0, 0, 0, 0);
                    }
                }
                cp_async_commit();
                if (++pending > kLag) {
                    cp_async_wait<kLag>();
                    retire(g - kLag);
                    --pending;
                }
            }
            producer_barrier();   // the table is rewritten by the next query
        }
        cp_async_wait<0>();
        for (; pending > 0; --pending) retire(g - pending);
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t kIdS = tc::idesc_f16_f32(kTK, kH, false, false);
            constexpr uint32_t kIdO = tc::idesc_f16_f32(kTK, kH, true, true);
            long long g = 0, gs = 0, gp = 0;
            int t = 0;
            for (int i = q_begin; i < q_end && ok; ++i, ++t) {
                const QueryKeys k = query_keys(a, i);
                const int n = k.n_tiles;
                const uint32_t obuf = static_cast<uint32_t>(t & 1);
                auto issue_pv = [&](int c) {
                    const long long ev = g++;
                    const int s = static_cast<int>(ev % kNS);
                    wait(&bar.full[s], static_cast<uint32_t>(ev / kNS) & 1u);
                    wait(&bar.p_full, static_cast<uint32_t>(gp) & 1u);
                    if (c == 0 && t >= 2) wait(&bar.o_empty[obuf], static_cast<uint32_t>((t >> 1) - 1) & 1u);
                    if (!ok) return;
                    tc::fence_after_sync();
                    const uint32_t va = tc::smem_u32(ring + s * kTileBytes), pb = tc::smem_u32(p_s);
#pragma unroll
                    for (int st = 0; st < kTK / 16; ++st) {
                        const uint64_t da = tc::desc_sw128(va + st * 2048, kTK * 128, 1024);
                        const uint64_t db = tc::desc_sw128(pb + st * 16 * 128, 8192, 1024);
                        tc::mma_f16(tmem + kColO + obuf * kH, da, db, kIdO, (c > 0 || st > 0) ? 1u : 0u);
                    }
                    tc::commit(&bar.p_empty);
                    tc::commit(&bar.empty[s]);
                    if (c == n - 1) tc::commit(&bar.o_full[obuf]);
                    ++gp;
                };
                for (int c = 0; c < n && ok; ++c) {
                    const long long ev = g++;
                    const int s = static_cast<int>(ev % kNS);
                    wait(&bar.full[s], static_cast<uint32_t>(ev / kNS) & 1u);
                    const uint32_t sb = static_cast<uint32_t>(gs & 1);
                    if (gs >= 2) wait(&bar.s_empty[sb], static_cast<uint32_t>((gs >> 1) - 1) & 1u);
                    if (!ok) break;
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
                    if (c >= 1) issue_pv(c - 1);
                }
                if (ok) issue_pv(n - 1);
            }
        }
        __syncwarp();
    }
    else {
        // ---------------- softmax + epilogue (warps 0-7) ----------------
        const int quad = warp & 3, half = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t kNegInfKey = float_key(-INFINITY);
        long long gs = 0, gp = 0;
        int t = 0;
        for (int i = q_begin; i < q_end; ++i, ++t) {
            const QueryKeys k = query_keys(a, i);
            const int n = k.n_tiles;
            const uint32_t obuf = static_cast<uint32_t>(t & 1);
            uint32_t vbits = 0;
            for (int c = 0; c < n; ++c)
                if (key_offset(a, i, k, c * kTK + quad * 32 + lane, false) >= 0) vbits |= 1u << c;
            float mh = -INFINITY;   // running reference of head half*32 + lane (log2 units)
            float l_lane[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) l_lane[h] = 0.f;
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
                // tile max of each head across the 128 lanes: warp, then the 4 quadrants
                float *rm = red_max + (gs & 1) * (4 * kH);
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    const uint32_t m = redux_max_u32(valid ? float_key(__uint_as_float(r[h])) : kNegInfKey);
                    if (lane == h) rm[quad * kH + half * 32 + h] = key_to_float(m);
                }
                softmax_barrier();
                float tm = rm[half * 32 + lane];
#pragma unroll
                for (int qd = 1; qd < 4; ++qd) tm = fmaxf(tm, rm[qd * kH + half * 32 + lane]);
                const float target = tm * a.scale_log2;   // scale > 0: the max commutes with it
                float alpha = 1.f;
                bool grow = false;
                if (mh == -INFINITY) {
                    mh = target;
                } else if (target > mh + kRescale) {
                    alpha = exp2f(mh - target);
                    mh = target;
                    grow = true;
                }
                const bool any_grow = __any_sync(0xffffffffu, grow);
                // the PV of the previous tile has finished with P^T and with O^T
                if (gp >= 1) wait(&bar.p_empty, static_cast<uint32_t>(gp - 1) & 1u);
                tc::fence_after_sync();
                if (any_grow) {
#pragma unroll
                    for (int h = 0; h < 32; ++h) l_lane[h] *= __shfl_sync(0xffffffffu, alpha, h);
                    if (c > 0) {
                        uint32_t o[32];
                        const uint32_t oa = tmem + lane_base + kColO + obuf * kH + half * 32;
                        ld_x32(oa, o);
                        tc::wait_ld();
#pragma unroll
                        for (int h = 0; h < 32; ++h)
                            o[h] = __float_as_uint(__uint_as_float(o[h]) * __shfl_sync(0xffffffffu, alpha, h));
                        st_x32(oa, o);
                        wait_st();
                    }
                }
                // p = 2^(s * scale - m) -> the P^T row (key) of this lane, 32 heads
                const int key = quad * 32 + lane;
                uint32_t pk[16];
#pragma unroll
                for (int h = 0; h < 32; h += 2) {
                    const float m0 = __shfl_sync(0xffffffffu, mh, h), m1 = __shfl_sync(0xffffffffu, mh, h + 1);
                    const float p0 = valid ? exp2f(__uint_as_float(r[h]) * a.scale_log2 - m0) : 0.f;
                    const float p1 = valid ? exp2f(__uint_as_float(r[h + 1]) * a.scale_log2 - m1) : 0.f;
                    l_lane[h] += p0;
                    l_lane[h + 1] += p1;
                    pk[h / 2] = pack_half2(p0, p1);
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int ch = half * 4 + q4;
                    *reinterpret_cast<uint4 *>(p_s + key * 128 + ((ch ^ (key & 7)) << 4)) =
                        make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full);
                ++gs;
                ++gp;
            }
            // ---- per-head sums, then O^T / l to the output ----
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                float s = l_lane[h];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == h) red_sum[quad * kH + half * 32 + h] = s;
            }
            softmax_barrier();
            float lsum = red_sum[half * 32 + lane];
#pragma unroll
            for (int qd = 1; qd < 4; ++qd) lsum += red_sum[qd * kH + half * 32 + lane];
            const float inv = 1.f / lsum;
            wait(&bar.o_full[obuf], static_cast<uint32_t>(t >> 1) & 1u);
            tc::fence_after_sync();
            uint32_t o[32];
            ld_x32(tmem + lane_base + kColO + obuf * kH + half * 32, o);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_empty[obuf]);
            uint16_t *dst = a.out + (static_cast<size_t>(i) * kH + half * 32) * kD + quad * 32 + lane;
#pragma unroll
            for (int h = 0; h < 32; ++h) dst[h * kD] = f2h(__uint_as_float(o[h]) * __shfl_sync(0xffffffffu, inv, h));
            softmax_barrier();   // red_sum is rewritten by the next query
        }
    }
    if (!ok) record_error(a.err, DS4A_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool attn_prefill_tc_ok(int H, int D, long long max_keys) {
    return H == kH && D == kD && max_keys <= kMaxTiles * kTK;
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
    Args a{q, raw_k, raw_v, comp_k, comp_v, sel, out, c.err, n_comp, q_pos0, T, n_prior, window, k_stride,
           ratio, scale * kLog2e};
    const int grid = T < c.num_sms ? T : c.num_sms;
    return launch(attn_prefill_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, c, 1, a);
}

}  // namespace ds4a
