// attention.cu -- multi-query attention over the raw window and the compressed
// rows, as one softmax ("DS4 (DwarfStar 4)", Architecture: 64 heads, 1 KV head,
// 128-token sliding window; Key Techniques, "KV attention compression").
//
// For each head h: o_h = sum_j softmax_j(scale * q_h . K_j) V_j over the union of
// the window rows and the selected (or all visible) compressed rows.
//
// Tile engine (shared by decode and prefill).  A CTA of 8 warps walks a list of
// "virtual rows" (window rows first, then compressed rows through `sel`) in
// tiles of 64 (80 in some decode launches, below).  Each tile's K and V rows are gathered with 16-byte cp.async into
// a double-buffered, XOR-swizzled shared-memory tile.  Warp w owns heads
// 16(w%4) .. 16(w%4)+15 (the 64 heads of one query are the M dimension: they
// all share each K/V row, 64 flop per byte) and keys 32(w/4) .. +31 of each
// tile; it computes S = Q K^T and O += P V with mma.sync m16n8k16 (fp16 in,
// fp32 accumulate) and keeps an online softmax in the log2 domain.  16-key
// groups past the end of the list are skipped; rows that are padding (negative
// sel entries) get -inf logits and zero-filled K/V.  The two key halves of a
// head group are combined through shared memory at the end.
//
// Decode: one query, rows split across one thread-block cluster of 16 CTAs (8
// if 16 cannot be scheduled).  Inside a CTA the 8 warps split by head group x
// half of d instead (compute_tile_dsplit): both halves compute the same scores,
// and no partial state has to be combined across warps.  Each CTA stages its
// (O as fp16, m, l) of every head in its own shared memory and sends the rows of
// each owner's heads with one bulk copy into the owner's shared memory, counted in
// bytes on the owner's receive mbarrier; each CTA waits only for the bytes destined
// to it, then merges its own heads by log-sum-exp from local shared memory.  A
// cluster arrive at kernel start (after the receive barrier is armed), waited on
// just before the first copy, guarantees every peer is running and ready.  Window
// rows are cache state and, with the query, are gathered before waiting on the
// previous kernel.  No workspace, no second launch, no spin.  A tile costs a fixed
// part (row table, loads, softmax) well above its per-row work, so a one-session
// launch (and a batched compressor + attention launch) whose CTAs attend 65 .. 80
// rows takes them as one 80-row tile instead of 64 + a remainder.
// Prefill: one CTA per query walks the query's whole row list (the shapes the
// tensor-core kernel in attention_tc.cu does not take).
#include <cooperative_groups.h>

#include "compress_dev.cuh"
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace cg = cooperative_groups;

namespace ds4a {
namespace {

constexpr int kThreads = 256;    // 8 warps: 4 head groups x 2 key halves (decode: x 2 halves of d)
constexpr int kBN = 64;           // rows per tile
constexpr int kHalf = kBN / 2;    // keys per warp per tile
constexpr float kLog2e = 1.4426950408889634f;

// Where the virtual rows live: v < n_w -> window row wk/wv + v*D; otherwise the
// compressed row j = sel ? sel[v - n_w] : v - n_w (j < 0: padding; j >= n_comp:
// recorded as an index error and treated as padding).
struct RowSrc {
    const uint16_t *wk;
    const uint16_t *wv;
    const uint16_t *ck;
    const uint16_t *cv;
    const int32_t *sel;
    unsigned int *err;
    long long n_comp;
    int n_w;
};

template <int D, int BN = kBN>
struct Smem {
    uint16_t k[2][BN * D];
    uint16_t v[2][BN * D];
    long long off[2][BN];   // element offset of the row in the window (>=0, tagged) / comp arrays; -1 = padding
    int nvalid[2];          // rows of the tile inside the list (the rest is padding)
};

// Row offset encoding: bit 62 set -> window row.
constexpr long long kWinTag = 1LL << 62;

// byte offset of 16-byte chunk `ch` of row `r` in a swizzled tile
template <int D>
DS4A_DEVINL uint32_t swz(int r, int ch) {
    return static_cast<uint32_t>(r * (D * 2) + ((ch ^ (r & 7)) << 4));
}

template <int D, int BN = kBN>
DS4A_DEVINL void build_table(const RowSrc &s, int v0, int v_end, long long *off, int *nvalid) {
    const int t = threadIdx.x;
    if (t == 0) *nvalid = min(BN, v_end - v0);
    if (t < BN) {
        const int v = v0 + t;
        long long o = -1;
        if (v < v_end) {
            if (v < s.n_w) {
                o = kWinTag | (static_cast<long long>(v) * D);
            } else {
                const long long j = s.sel ? static_cast<long long>(__ldg(s.sel + (v - s.n_w)))
                                          : static_cast<long long>(v - s.n_w);
                if (j >= s.n_comp) record_error(s.err, DS4A_ERR_DEVICE_INDEX);
                else if (j >= 0) o = j * D;
            }
        }
        off[t] = o;
    }
}

template <int D, int BN = kBN>
DS4A_DEVINL void issue_loads(const RowSrc &s, const long long *off, uint16_t *kt, uint16_t *vt) {
    constexpr int kChunks = D / 8;
    unsigned char *kb = reinterpret_cast<unsigned char *>(kt);
    unsigned char *vb = reinterpret_cast<unsigned char *>(vt);
    for (int i = threadIdx.x; i < BN * kChunks; i += kThreads) {
        const int r = i / kChunks, ch = i % kChunks;
        const long long o = off[r];
        const uint32_t so = swz<D>(r, ch);
        if (o < 0) {
            *reinterpret_cast<uint4 *>(kb + so) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(vb + so) = make_uint4(0, 0, 0, 0);
        } else if (o & kWinTag) {
            const long long e = (o & ~kWinTag) + ch * 8;
            cp_async16(kb + so, s.wk + e);
            cp_async16(vb + so, s.wv + e);
        } else {
            const long long e = o + ch * 8;
            cp_async16(kb + so, s.ck + e);
            cp_async16(vb + so, s.cv + e);
        }
    }
}

// Bring rows [r0, r1) of a [*, D] fp16 array into L2: one bulk prefetch, which
// returns no data (a row another kernel writes afterwards is still read correctly).
template <int D>
DS4A_DEVINL void prefetch_rows_l2(const uint16_t *base, long long r0, long long r1) {
    if (r1 <= r0) return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(base + r0 * D),
                 "r"(static_cast<uint32_t>((r1 - r0) * D * 2))
                 : "memory");
}

// Per-warp running state: rows g and g+8 of the warp's 16 heads.
template <int D>
struct WarpState {
    float o[D / 8][4];
    float m[2];
    float l[2];
};

template <int D>
DS4A_DEVINL void load_q_frags(const uint16_t *q, int H, int h0, uint32_t (&qa)[D / 16][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int ra = h0 + g, rb = h0 + g + 8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int c0 = ks * 16 + 2 * t, c1 = c0 + 8;
        qa[ks][0] = ra < H ? *reinterpret_cast<const uint32_t *>(q + ra * D + c0) : 0u;
        qa[ks][1] = rb < H ? *reinterpret_cast<const uint32_t *>(q + rb * D + c0) : 0u;
        qa[ks][2] = ra < H ? *reinterpret_cast<const uint32_t *>(q + ra * D + c1) : 0u;
        qa[ks][3] = rb < H ? *reinterpret_cast<const uint32_t *>(q + rb * D + c1) : 0u;
    }
}

// One tile, keys kh*32 .. kh*32+31 of it: S = Q K^T, online softmax, O += P V.
template <int D>
DS4A_DEVINL void compute_tile(const uint32_t (&qa)[D / 16][4], const uint16_t *kt, const uint16_t *vt,
                              const long long *off, int nvalid, int kh, float scale_log2, WarpState<D> &st) {
    const int lane = threadIdx.x & 31, t = lane & 3;
    const int kbase = kh * kHalf;
    if (kbase >= nvalid) return;                                  // warp-uniform
    const int groups = min(2, (nvalid - kbase + 15) / 16);        // 16-key groups holding list rows
    const unsigned char *kb = reinterpret_cast<const unsigned char *>(kt);
    const unsigned char *vb = reinterpret_cast<const unsigned char *>(vt);
    float s[kHalf / 8][4];
#pragma unroll
    for (int nt = 0; nt < kHalf / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;

    // S = Q K^T: ldmatrix x4 gives b0/b1 for two key tiles (one 16-key group) at one k-step
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
            if (gq < groups) {
                const int key = kbase + gq * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(b0, b1, b2, b3, kb + swz<D>(key, ch));
                mma_16816(s[2 * gq], qa[ks], b0, b1);
                mma_16816(s[2 * gq + 1], qa[ks], b2, b3);
            }
        }
    }

    // scale into the log2 domain, mask padding rows, running max
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < kHalf / 8; ++nt) {
        const int kr = kbase + nt * 8 + 2 * t;
        const bool v0 = off[kr] >= 0, v1 = off[kr + 1] >= 0;
        s[nt][0] = v0 ? s[nt][0] * scale_log2 : -INFINITY;
        s[nt][1] = v1 ? s[nt][1] * scale_log2 : -INFINITY;
        s[nt][2] = v0 ? s[nt][2] * scale_log2 : -INFINITY;
        s[nt][3] = v1 ? s[nt][3] * scale_log2 : -INFINITY;
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float ref[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float m_new = fmaxf(st.m[r], mx[r]);
        ref[r] = m_new == -INFINITY ? 0.f : m_new;
        alpha[r] = exp2f(st.m[r] - ref[r]);
        st.m[r] = m_new;
        st.l[r] *= alpha[r];
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
        st.o[dn][0] *= alpha[0];
        st.o[dn][1] *= alpha[0];
        st.o[dn][2] *= alpha[1];
        st.o[dn][3] *= alpha[1];
    }
    uint32_t pa[kHalf / 16][4];
#pragma unroll
    for (int nt = 0; nt < kHalf / 8; ++nt) {
        const float p0 = exp2f(s[nt][0] - ref[0]), p1 = exp2f(s[nt][1] - ref[0]);
        const float p2 = exp2f(s[nt][2] - ref[1]), p3 = exp2f(s[nt][3] - ref[1]);
        st.l[0] += p0 + p1;
        st.l[1] += p2 + p3;
        const int kk = nt >> 1, hi = nt & 1;
        pa[kk][hi ? 2 : 0] = pack_half2(p0, p1);
        pa[kk][hi ? 3 : 1] = pack_half2(p2, p3);
    }
    // O += P V: ldmatrix.trans x4 gives b0/b1 for two d tiles at one 16-key step
#pragma unroll
    for (int kk = 0; kk < kHalf / 16; ++kk) {
        if (kk < groups) {
#pragma unroll
            for (int dn = 0; dn < D / 8; dn += 2) {
                const int key = kbase + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dn + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, vb + swz<D>(key, ch));
                mma_16816(st.o[dn], pa[kk], b0, b1);
                mma_16816(st.o[dn + 1], pa[kk], b2, b3);
            }
        }
    }
}

// Walk virtual rows [v_begin, v_end) of `src`, accumulating into `st`.  If
// `tile0_issued`, the caller has already built the first tile's table and
// issued (and committed) its loads.
template <int D>
__device__ void attend_range(const RowSrc &src, int v_begin, int v_end, const uint32_t (&qa)[D / 16][4],
                             bool has_heads, int kh, float scale_log2, Smem<D> &sm, WarpState<D> &st,
                             bool tile0_issued) {
    const int n_tiles = v_end > v_begin ? (v_end - v_begin + kBN - 1) / kBN : 0;
    if (n_tiles == 0) return;
    if (!tile0_issued) {
        build_table<D>(src, v_begin, v_end, sm.off[0], &sm.nvalid[0]);
        __syncthreads();
        issue_loads<D>(src, sm.off[0], sm.k[0], sm.v[0]);
        cp_async_commit();
    }
    for (int it = 0; it < n_tiles; ++it) {
        __syncthreads();
        if (it + 1 < n_tiles) {
            const int b = (it + 1) & 1;
            build_table<D>(src, v_begin + (it + 1) * kBN, v_end, sm.off[b], &sm.nvalid[b]);
            __syncthreads();
            issue_loads<D>(src, sm.off[b], sm.k[b], sm.v[b]);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int b = it & 1;
        if (has_heads) compute_tile<D>(qa, sm.k[b], sm.v[b], sm.off[b], sm.nvalid[b], kh, scale_log2, st);
    }
    __syncthreads();
}

template <int D>
DS4A_DEVINL void init_state(WarpState<D> &st) {
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[dn][e] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
}

// Combine the two key halves of each head group: warps 4..7 hand their state
// to warps 0..3 through shared memory (`xch` must hold 4*32*(D/2+4) floats).
template <int D>
DS4A_DEVINL void combine_halves(WarpState<D> &st, float *xch) {
    constexpr int kStride = D / 2 + 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= 4) {
        float *p = xch + ((warp - 4) * 32 + lane) * kStride;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
            for (int e = 0; e < 4; ++e) p[dn * 4 + e] = st.o[dn][e];
        p[D / 2 + 0] = st.m[0];
        p[D / 2 + 1] = st.m[1];
        p[D / 2 + 2] = st.l[0];
        p[D / 2 + 3] = st.l[1];
    }
    __syncthreads();
    if (warp < 4) {
        const float *p = xch + (warp * 32 + lane) * kStride;
        float wa[2], wb[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float mb = p[D / 2 + r];
            const float M = fmaxf(st.m[r], mb);
            wa[r] = st.m[r] == -INFINITY ? 0.f : exp2f(st.m[r] - M);
            wb[r] = mb == -INFINITY ? 0.f : exp2f(mb - M);
            st.l[r] = st.l[r] * wa[r] + p[D / 2 + 2 + r] * wb[r];
            st.m[r] = M;
        }
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            st.o[dn][0] = st.o[dn][0] * wa[0] + p[dn * 4 + 0] * wb[0];
            st.o[dn][1] = st.o[dn][1] * wa[0] + p[dn * 4 + 1] * wb[0];
            st.o[dn][2] = st.o[dn][2] * wa[1] + p[dn * 4 + 2] * wb[1];
            st.o[dn][3] = st.o[dn][3] * wa[1] + p[dn * 4 + 3] * wb[1];
        }
    }
    __syncthreads();
}

// ---- decode tile engine: warps split by head group x half of d ------------------------------
// Warp w owns heads 16(w%4) .. +15 and output columns d in [(w/4) D/2, (w/4 + 1) D/2): it
// computes S for all the tile's keys (the two d halves of a head group compute the same S
// and the same softmax state), and O += P V for its half of d only.  Nothing has to be
// combined across warps afterwards.

template <int D>
struct WarpStateH {
    float o[D / 16][4];   // rows g and g+8 of the warp's 16 heads, D/2 columns
    float m[2];
    float l[2];
};

template <int D, int BN = kBN>
DS4A_DEVINL void compute_tile_dsplit(const uint32_t (&qa)[D / 16][4], const uint16_t *kt, const uint16_t *vt,
                                     const long long *off, int nvalid, int dh, float scale_log2,
                                     WarpStateH<D> &st) {
    const int lane = threadIdx.x & 31, t = lane & 3;
    if (nvalid <= 0) return;
    const int groups = min(BN / 16, (nvalid + 15) / 16);   // 16-key groups holding list rows
    const unsigned char *kb = reinterpret_cast<const unsigned char *>(kt);
    const unsigned char *vb = reinterpret_cast<const unsigned char *>(vt);
    float s[BN / 8][4];
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
    // S = Q K^T over the tile: ldmatrix x4 gives b0/b1 for two key tiles (one 16-key group)
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int gq = 0; gq < BN / 16; ++gq) {
            if (gq < groups) {
                const int key = gq * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(b0, b1, b2, b3, kb + swz<D>(key, ch));
                mma_16816(s[2 * gq], qa[ks], b0, b1);
                mma_16816(s[2 * gq + 1], qa[ks], b2, b3);
            }
        }
    }
    // scale into the log2 domain, mask padding rows, running max
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) {
        const int kr = nt * 8 + 2 * t;
        const bool v0 = off[kr] >= 0, v1 = off[kr + 1] >= 0;
        s[nt][0] = v0 ? s[nt][0] * scale_log2 : -INFINITY;
        s[nt][1] = v1 ? s[nt][1] * scale_log2 : -INFINITY;
        s[nt][2] = v0 ? s[nt][2] * scale_log2 : -INFINITY;
        s[nt][3] = v1 ? s[nt][3] * scale_log2 : -INFINITY;
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float ref[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float m_new = fmaxf(st.m[r], mx[r]);
        ref[r] = m_new == -INFINITY ? 0.f : m_new;
        alpha[r] = exp2f(st.m[r] - ref[r]);
        st.m[r] = m_new;
        st.l[r] *= alpha[r];
    }
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
        st.o[dn][0] *= alpha[0];
        st.o[dn][1] *= alpha[0];
        st.o[dn][2] *= alpha[1];
        st.o[dn][3] *= alpha[1];
    }
    uint32_t pa[BN / 16][4];
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) {
        const float p0 = exp2f(s[nt][0] - ref[0]), p1 = exp2f(s[nt][1] - ref[0]);
        const float p2 = exp2f(s[nt][2] - ref[1]), p3 = exp2f(s[nt][3] - ref[1]);
        st.l[0] += p0 + p1;
        st.l[1] += p2 + p3;
        const int kk = nt >> 1, hi = nt & 1;
        pa[kk][hi ? 2 : 0] = pack_half2(p0, p1);
        pa[kk][hi ? 3 : 1] = pack_half2(p2, p3);
    }
    // O += P V over this warp's half of d: ldmatrix.trans x4 gives b0/b1 for two d tiles
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        if (kk < groups) {
#pragma unroll
            for (int dn = 0; dn < D / 16; dn += 2) {
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dh * (D / 16) + dn + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, vb + swz<D>(key, ch));
                mma_16816(st.o[dn], pa[kk], b0, b1);
                mma_16816(st.o[dn + 1], pa[kk], b2, b3);
            }
        }
    }
}

// Walk virtual rows [v_begin, v_end) with the d-split engine (as attend_range).
template <int D, int BN = kBN>
__device__ void attend_range_dsplit(const RowSrc &src, int v_begin, int v_end, const uint32_t (&qa)[D / 16][4],
                                    bool has_heads, int dh, float scale_log2, Smem<D, BN> &sm, WarpStateH<D> &st,
                                    bool tile0_issued) {
    const int n_tiles = v_end > v_begin ? (v_end - v_begin + BN - 1) / BN : 0;
    if (n_tiles == 0) return;
    if (!tile0_issued) {
        build_table<D, BN>(src, v_begin, v_end, sm.off[0], &sm.nvalid[0]);
        __syncthreads();
        issue_loads<D, BN>(src, sm.off[0], sm.k[0], sm.v[0]);
        cp_async_commit();
    }
    for (int it = 0; it < n_tiles; ++it) {
        __syncthreads();
        if (it + 1 < n_tiles) {
            const int b = (it + 1) & 1;
            build_table<D, BN>(src, v_begin + (it + 1) * BN, v_end, sm.off[b], &sm.nvalid[b]);
            __syncthreads();
            issue_loads<D, BN>(src, sm.off[b], sm.k[b], sm.v[b]);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int b = it & 1;
        if (has_heads) compute_tile_dsplit<D, BN>(qa, sm.k[b], sm.v[b], sm.off[b], sm.nvalid[b], dh, scale_log2, st);
    }
    __syncthreads();
}

// quad-reduce the per-lane partial sums of l
template <int D>
DS4A_DEVINL void finish_l(WarpState<D> &st) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
    }
}

// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
DS4A_DEVINL uint32_t cluster_addr(const void *local, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
    return r;
}
// bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this
// CTA's shared memory into another CTA's, counted in bytes on that CTA's mbarrier
DS4A_DEVINL void bulk_copy_to_cta(uint32_t raddr, const void *local, uint32_t bytes, uint32_t rbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     raddr),
                 "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(bytes), "r"(rbar)
                 : "memory");
}
DS4A_DEVINL void tc_mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))),
                 "r"(count));
}
// bounded wait (limit_ns of wall time) for phase 0 of a receive barrier
DS4A_DEVINL bool recv_wait(uint64_t *bar, uint64_t limit_ns) {
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done)
                     : "r"(b)
                     : "memory");
        if (done) return true;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(now));
        if (it == 0) t0 = now;
        else if (now - t0 > limit_ns) return false;
    }
}
constexpr uint64_t kRecvLimitNs = 1000000000ull;   // about a second
DS4A_DEVINL void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
DS4A_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

struct DecodeArgs {
    const uint16_t *q;
    uint16_t *out;
    RowSrc src;
    int H;
    int n_rows;        // n_win + n_sel
    float scale_log2;
    int comp_rank;     // with the compressor: the CTA that runs its update (the last row's CTA on a completing step, else 0)
    int comp_first;    // the update completes a block: its row is written before that CTA attends
    long long test_wait_ns;   // > 0 (test hook only): CTA 0 also waits this long on a barrier nobody completes
    // Batched decode: cluster blockIdx.y serves session s, whose inputs sit at fixed
    // strides from session 0's and whose position is pos[s] (device memory, read early).
    // The fields above are then session 0's pointers; the row counts, the window length
    // and the compressor's CTA follow from each session's position.
    const long long *pos;     // nullptr: one session, the fields above as given
    long long q_stride;       // elements between the sessions' q and out
    long long win_stride;     // elements between the sessions' window rings
    long long comp_stride;    // elements between the sessions' compressed rows
    long long sel_stride;     // entries between the sessions' kept-row lists
    long long state_stride;   // floats between the sessions' compressor states
    long long cap;            // compressed rows allocated per session
    int W;                    // ring length: window rows min(W, p + 1), slot p % W holds token p
    int ratio;                // 0: window only
    int n_sel_list;           // with sel: entries per list (-1 entries are skipped)
};

constexpr int kRecvRows = 80;   // >= cluster size * ceil(H / cluster size) for H <= 64
// one session's fused compressor + attention launch whose CTAs attend kBN+1 .. kBigBN rows
// each takes them as one tile (a tile costs a fixed part, row table, loads, softmax, far
// above its per-row work)
constexpr int kBigBN = 80;

template <int D, int BN = kBN>
__host__ __device__ constexpr size_t recv_offset() { return (sizeof(Smem<D, BN>) + 127) / 128 * 128; }
// One head's split-KV partial as exchanged between the CTAs of a cluster: O as D fp16
// (its rounding, 2^-11 relative, is far inside the output's fp16), then the running
// max m and sum l as fp32, padded to a 16-byte multiple for the bulk copies.
template <int D>
__host__ __device__ constexpr int part_bytes() { return 2 * D + 16; }
template <int D, int BN = kBN>
constexpr size_t decode_smem() { return recv_offset<D, BN>() + kRecvRows * part_bytes<D>(); }
template <int D>
constexpr size_t prefill_smem() { return sizeof(Smem<D>); }
static_assert(4 * 32 * (128 / 2 + 4) * sizeof(float) <= sizeof(Smem<128>), "exchange fits in the tiles");
static_assert(64 * part_bytes<128>() <= sizeof(Smem<128>) && 64 * part_bytes<64>() <= sizeof(Smem<64>),
              "the send rows of 64 heads fit in the tiles");
static_assert(part_bytes<128>() % 16 == 0 && part_bytes<64>() % 16 == 0, "bulk copies move 16-byte multiples");

// Log-sum-exp merge of the (O, m, l) rows every rank sent for heads [hb, hb + nh):
// recv[rank][local head] (part_bytes each); out[h] = sum_r w_r O_r / sum_r w_r l_r with
// w_r = 2^(m_r - max_r m_r).  First each (rank, head) weight w_r / sum_r w_r l_r, once
// (the ranks of a head are consecutive lanes of one warp), then every column's sum.
// wsh: cs * hpc floats of shared memory.  CS: the cluster size (0: runtime cs).
template <int D, int CS>
DS4A_DEVINL void merge_heads(const unsigned char *recv, int hpc, int hb, int nh, uint16_t *out, float *wsh,
                             int cs_rt = CS) {
    const int cs = CS > 0 ? CS : cs_rt;
    constexpr int RB = part_bytes<D>();
    // cs is a power of two <= 16: the ranks of head hh are lanes (hh * cs + r) % 32
    {
        const int t = threadIdx.x, r = t % cs, hh = t / cs;
        const bool valid = hh < nh;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (valid) ml = *reinterpret_cast<const float2 *>(recv + (r * hpc + hh) * RB + 2 * D);
        float M = ml.x;
        for (int o = 1; o < cs; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
        float den = w * ml.y;
        for (int o = 1; o < cs; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (valid) wsh[r * hpc + hh] = w / den;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nh * (D / 2); idx += kThreads) {   // 2 columns per item
        const int hh = idx / (D / 2), d = (idx % (D / 2)) * 2;
        float2 acc = make_float2(0.f, 0.f);
        auto add_rank = [&](int r) {
            const float w = wsh[r * hpc + hh];
            const float2 o = __half22float2(*reinterpret_cast<const __half2 *>(recv + (r * hpc + hh) * RB + 2 * d));
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
        };
        if constexpr (CS > 0) {
#pragma unroll
            for (int r = 0; r < CS; ++r) add_rank(r);
        } else {
            for (int r = 0; r < cs; ++r) add_rank(r);
        }
        *reinterpret_cast<uint32_t *>(out + (hb + hh) * D + d) = pack_half2(acc.x, acc.y);
    }
}

// kCompress: one CTA (a.comp_rank) also runs the compressor's update for the step's
// token (n_new = 1, arguments ca): its score before the dependency wait; the
// running state and, when the token completes a block, the pooled row after it.
// A completed row is the last row this call attends and a.comp_rank is the CTA
// that attends it, so that CTA writes the row before it attends its rows.  On the
// other steps CTA 0 updates the state after its partials are sent: its first tile
// (window rows) is gathered before the wait, so it finishes its tiles first and the
// update overlaps the other CTAs' tiles.  No other CTA reads what the compressor
// writes.
template <int D, bool kCompress, int BN = kBN>
__global__ void __launch_bounds__(kThreads, (kCompress || BN != kBN) ? 1 : 2)
    attn_decode_kernel(DecodeArgs a, cmp::CompressArgs ca) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<D, BN> &sm = *reinterpret_cast<Smem<D, BN> *>(smem_raw);
    unsigned char *recv = smem_raw + recv_offset<D, BN>();
    constexpr int RB = part_bytes<D>();
    __shared__ __align__(8) uint64_t s_recv_bar;
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    if (a.pos != nullptr) {   // batched: this cluster's session
        const long long sid = blockIdx.y;
        const long long p = a.pos[sid];
        a.q += sid * a.q_stride;
        a.out += sid * a.q_stride;
        a.src.wk += sid * a.win_stride;
        a.src.wv += sid * a.win_stride;
        a.src.ck += sid * a.comp_stride;
        a.src.cv += sid * a.comp_stride;
        if (a.src.sel) a.src.sel += sid * a.sel_stride;
        a.src.n_w = static_cast<int>(p + 1 < a.W ? p + 1 : a.W);
        long long n_sel = a.n_sel_list;
        if (!a.src.sel) {   // every visible row
            const long long nv = a.ratio > 0 ? (p + 1) / a.ratio : 0;
            n_sel = nv < a.cap ? nv : a.cap;
            a.src.n_comp = n_sel;
        }
        a.n_rows = a.src.n_w + static_cast<int>(n_sel);
        if constexpr (kCompress) {
            const long long slot = (p % a.W) * D;
            ca.pos = p;
            ca.k = a.src.wk + slot;
            ca.v = a.src.wv + slot;
            ca.state += sid * a.state_stride;
            ca.comp_k += sid * a.comp_stride;
            ca.comp_v += sid * a.comp_stride;
            const int chunk = (a.n_rows + cs - 1) / cs;
            a.comp_first = (p + 1) % a.ratio == 0;
            a.comp_rank = a.comp_first ? (a.n_rows - 1) / chunk : 0;
            if ((p + 1) / a.ratio > a.cap) {
                // the row this token completes is past the session's capacity: no update
                a.comp_rank = -1;
                if (rank == 0 && threadIdx.x == 0) record_error(a.src.err, DS4A_ERR_CAPACITY);
            }
        }
    }
    // heads [hb, hb + nh) are merged here: every CTA of the cluster sends (O, m, l) of
    // each of them, a row of part_bytes (16-byte multiple), into this CTA's receive buffer
    const int hpc = (a.H + cs - 1) / cs;
    const int hb = rank * hpc;
    const int nh = max(0, min(a.H, hb + hpc) - hb);
    if (threadIdx.x == 0) {
        tc_mbar_init(&s_recv_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(&s_recv_bar))),
                     "r"(static_cast<uint32_t>(cs * nh * RB))
                     : "memory");
    }
    // this CTA is running and its receive barrier is armed; waited on before the first copy is sent
    cluster_arrive_release();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int h0 = (warp & 3) * 16, dh = warp >> 2;   // head group, half of d
    const bool has_heads = h0 < a.H;
    const int chunk = (a.n_rows + cs - 1) / cs;
    const int v0 = min(a.n_rows, rank * chunk);
    const int v1 = min(a.n_rows, v0 + chunk);
    const bool comp_here = kCompress && rank == a.comp_rank;
    __shared__ float s_cw[1], s_cred[kThreads / 32];   // compressor: the token's score, per-warp maxima
    if (comp_here) cmp::segment_scores<kThreads>(ca, ca.pos, ca.pos + 1, s_cw);
    // a first tile of window rows only (cache state) is gathered before the dependency wait
    // (not by a CTA that writes a compressed row before it attends)
    const bool pre = v1 > v0 && min(v1, v0 + BN) <= a.src.n_w && !(comp_here && a.comp_first);
    if (pre) {
        build_table<D, BN>(a.src, v0, v1, sm.off[0], &sm.nvalid[0]);
        __syncthreads();
        issue_loads<D, BN>(a.src, sm.off[0], sm.k[0], sm.v[0]);
        cp_async_commit();
    }
    if (a.pos == nullptr && threadIdx.x < 4) {
        // one session: warm L2 with the rows this CTA gathers after the dependency wait
        // (window rows past the first tile; compressed rows when every row is attended,
        // since a kept-row list is known only after the wait)
        const int pv0 = pre ? min(v1, v0 + BN) : v0;
        const int nw = a.src.n_w;
        if (threadIdx.x < 2) {
            prefetch_rows_l2<D>(threadIdx.x ? a.src.wv : a.src.wk, pv0, min(v1, nw));
        } else if (!a.src.sel) {
            const long long c0 = max(pv0, nw) - nw, c1 = min(static_cast<long long>(v1 - nw), a.src.n_comp);
            prefetch_rows_l2<D>(threadIdx.x == 3 ? a.src.cv : a.src.ck, c0, c1);
        }
    }
    // the query is an input no kernel of this library writes: loaded before the wait too
    uint32_t qa[D / 16][4];
    load_q_frags<D>(a.q, a.H, h0, qa);
    pdl_wait();
    pdl_trigger();
    if (comp_here && a.comp_first) {
        cmp::pool_segment<kThreads>(ca, ca.pos / ca.ratio, ca.pos, ca.pos + 1, ca.pos % ca.ratio != 0, s_cw, s_cred);
        __threadfence();   // the row is in memory before this CTA's own row loads read it
        __syncthreads();
    }
    WarpStateH<D> st;
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[dn][e] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
    attend_range_dsplit<D, BN>(a.src, v0, v1, qa, has_heads, dh, a.scale_log2, sm, st, pre);
#pragma unroll
    for (int r = 0; r < 2; ++r) {   // quad-reduce the per-lane partial sums of l
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
    }

    // Stage (O, m, l) of each head in this CTA's own shared memory, send[h] (part_bytes
    // each; the tiles are free once every warp is past them), then send the rows of
    // each owner's heads with one bulk copy into recv[this rank] there; the copies
    // complete on the owner's receive barrier.
    unsigned char *send = smem_raw;
    __syncthreads();
    if (has_heads) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int h = h0 + g + 8 * r;
            if (h < a.H) {
                unsigned char *row = send + h * RB;
#pragma unroll
                for (int dn = 0; dn < D / 16; ++dn)
                    *reinterpret_cast<__half2 *>(row + 2 * (dh * (D / 2) + dn * 8 + 2 * t)) =
                        __floats2half2_rn(st.o[dn][2 * r], st.o[dn][2 * r + 1]);
                if (t == 0 && dh == 0) *reinterpret_cast<float2 *>(row + 2 * D) = make_float2(st.m[r], st.l[r]);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");   // the copies read through the async proxy
    __syncthreads();
    cluster_wait();   // every CTA's receive barrier is armed
    // lane 0 of each warp sends the rows of owners warp, warp + 8, ...: the copies are
    // issued in parallel rather than one after another by one thread
    if (lane == 0) {
        for (int o = warp; o < cs; o += kThreads / 32) {
            const int nho = min(a.H, (o + 1) * hpc) - o * hpc;
            if (nho > 0)
                bulk_copy_to_cta(cluster_addr(recv + rank * hpc * RB, o), send + o * hpc * RB,
                                 static_cast<uint32_t>(nho * RB), cluster_addr(&s_recv_bar, o));
        }
        asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
    }
    if (comp_here && !a.comp_first)   // off the critical path: while the partials travel
        cmp::pool_segment<kThreads>(ca, ca.pos / ca.ratio, ca.pos, ca.pos + 1, ca.pos % ca.ratio != 0, s_cw, s_cred);
    // every byte destined for this CTA has landed
    if (!recv_wait(&s_recv_bar, kRecvLimitNs)) record_error(a.src.err, DS4A_ERR_TIMEOUT);
    if (a.test_wait_ns > 0 && rank == 0) {
        // Test hook: the bounded wait's give-up path, exercised with nothing in flight.
        // Every copy destined for this CTA has landed (the wait above completed), and
        // this barrier, armed for one arrival that no thread makes, never completes.
        __shared__ __align__(8) uint64_t s_never_bar;
        if (threadIdx.x == 0) tc_mbar_init(&s_never_bar, 1);
        __syncthreads();
        if (!recv_wait(&s_never_bar, static_cast<uint64_t>(a.test_wait_ns))) record_error(a.src.err, DS4A_ERR_TIMEOUT);
    }

    // merge this CTA's heads from local shared memory (the loop over the cluster's ranks
    // unrolled for the usual cluster sizes)
    __shared__ float s_w[kRecvRows];   // the merge's (rank, head) weights
    if (cs == 16) merge_heads<D, 16>(recv, hpc, hb, nh, a.out, s_w);
    else if (cs == 8) merge_heads<D, 8>(recv, hpc, hb, nh, a.out, s_w);
    else merge_heads<D, 0>(recv, hpc, hb, nh, a.out, s_w, cs);
    // this CTA's outgoing copies (each issuing lane's) have finished reading its shared memory
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

struct PrefillArgs {
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
    int H;
    int n_prior;
    int window;
    int k_stride;
    int ratio;
    float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads) attn_prefill_kernel(PrefillArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int h0 = (warp & 3) * 16, kh = warp >> 2;
    const bool has_heads = h0 < a.H;
    const int i = blockIdx.x;
    const long long p = a.q_pos0 + i;
    pdl_wait();
    pdl_trigger();

    // window: positions max(0, p-window+1) .. p; raw index = position - (q_pos0 - n_prior)
    const long long first = p - a.window + 1 > 0 ? p - a.window + 1 : 0;
    const long long raw0 = first - (a.q_pos0 - a.n_prior);
    RowSrc src;
    src.wk = a.raw_k + raw0 * D;
    src.wv = a.raw_v + raw0 * D;
    src.ck = a.comp_k;
    src.cv = a.comp_v;
    src.err = a.err;
    src.n_comp = a.n_comp;
    src.n_w = static_cast<int>(p - first + 1);
    int n_sel = 0;
    src.sel = nullptr;
    if (a.ratio > 0) {
        if (a.sel) {
            src.sel = a.sel + static_cast<size_t>(i) * a.k_stride;
            n_sel = a.k_stride;
        } else {
            const long long nv = (p + 1) / a.ratio;
            n_sel = static_cast<int>(nv < a.n_comp ? nv : a.n_comp);
        }
    }
    const uint16_t *q = a.q + static_cast<size_t>(i) * a.H * D;
    uint32_t qa[D / 16][4];
    load_q_frags<D>(q, a.H, h0, qa);
    WarpState<D> st;
    init_state<D>(st);
    attend_range<D>(src, 0, src.n_w + n_sel, qa, has_heads, kh, a.scale_log2, sm, st, false);
    combine_halves<D>(st, reinterpret_cast<float *>(smem_raw));
    finish_l<D>(st);
    if (warp < 4 && has_heads) {
        uint16_t *o = a.out + static_cast<size_t>(i) * a.H * D;
        const float inv0 = 1.f / st.l[0], inv1 = 1.f / st.l[1];
        const int ra = h0 + g, rb = h0 + g + 8;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = dn * 8 + 2 * t;
            if (ra < a.H)
                *reinterpret_cast<uint32_t *>(o + ra * D + d) = pack_half2(st.o[dn][0] * inv0, st.o[dn][1] * inv0);
            if (rb < a.H)
                *reinterpret_cast<uint32_t *>(o + rb * D + d) = pack_half2(st.o[dn][2] * inv1, st.o[dn][3] * inv1);
        }
    }
}

template <int D>
cudaError_t configure(int &cluster, int *active16 = nullptr, int *active8 = nullptr, int *active4 = nullptr) {
    static thread_local int configured_device = -1;
    static thread_local int cluster_size = 16;
    static thread_local int n_active16 = 0, n_active8 = 0, n_active4 = 0;   // clusters of 16 / 8 / 4 resident at once
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaSuccess;
        for (auto kern : {attn_decode_kernel<D, false>, attn_decode_kernel<D, true>}) {
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(decode_smem<D>()));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
        }
        for (auto kern : {attn_decode_kernel<D, false, kBigBN>, attn_decode_kernel<D, true, kBigBN>}) {
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(decode_smem<D, kBigBN>()));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(prefill_smem<D>()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_prefill_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        // largest cluster (16, else 8) that the device can schedule with this footprint
        cluster_size = 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = decode_smem<D>();
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 16;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n_clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&n_clusters, attn_decode_kernel<D, false>, &cfg) == cudaSuccess &&
            n_clusters > 0)
            cluster_size = 16;
        n_active16 = n_clusters > 0 ? n_clusters : 0;
        cudaGetLastError();
        attr.val.clusterDim.x = 8;
        cfg.gridDim = dim3(8);
        n_clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&n_clusters, attn_decode_kernel<D, false>, &cfg) != cudaSuccess)
            n_clusters = 0;
        n_active8 = n_clusters;
        cudaGetLastError();
        attr.val.clusterDim.x = 4;
        cfg.gridDim = dim3(4);
        n_clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&n_clusters, attn_decode_kernel<D, false>, &cfg) != cudaSuccess)
            n_clusters = 0;
        n_active4 = n_clusters;
        cudaGetLastError();
        configured_device = dev;
    }
    cluster = cluster_size;
    if (active16) *active16 = n_active16;
    if (active8) *active8 = n_active8;
    if (active4) *active4 = n_active4;
    return cudaSuccess;
}

// Cluster size of a batched launch of B sessions of at most `rows` rows each.  The
// clusters run in waves of `active` resident clusters, and a CTA's time grows with the
// kBN-row tiles it attends on top of a fixed part (row table, exchange, merge) worth
// about five tiles; the size with the smallest waves x (5 + tiles) wins, the larger
// size on a tie.  Measured on 640-row sessions: 16 sessions run best in clusters of
// 8 (12.4 us, against 16.0 in 16 and 13.4 in 4), 64 sessions in clusters of 4 (20.7 us,
// against 27.9 in 8; clusters of 2 gave 22.8).
int batched_cluster(int B, long long rows, int largest, int active16, int active8, int active4) {
    int best = largest;
    long long best_cost = -1;
    for (int cs : {16, 8, 4}) {
        const int active = cs == 16 ? active16 : cs == 8 ? active8 : active4;
        if (cs > largest || active <= 0) continue;
        const long long waves = (B + active - 1) / active;
        const long long tiles = (rows + static_cast<long long>(kBN) * cs - 1) / (static_cast<long long>(kBN) * cs);
        const long long cost = waves * (5 + tiles);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = cs;
        }
    }
    return best;
}

}  // namespace

cudaError_t launch_attn_decode(const uint16_t *q, int H, int D, const uint16_t *win_k,
                               const uint16_t *win_v, int n_win, const uint16_t *comp_k,
                               const uint16_t *comp_v, long long n_comp, const int32_t *sel,
                               int n_sel, float scale, uint16_t *out, const Ctx &c) {
    DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.src = RowSrc{win_k, win_v, comp_k, comp_v, sel, c.err, n_comp, n_win};
    a.H = H;
    a.n_rows = n_win + n_sel;
    a.scale_log2 = scale * kLog2e;
    a.comp_rank = -1;
    a.comp_first = 0;
    a.test_wait_ns = test_wait_limit_ns();
    int cluster = 16;
    cudaError_t e = D == 128 ? configure<128>(cluster) : configure<64>(cluster);
    if (e != cudaSuccess) return e;
    // CTAs that attend 65 .. 80 rows take them as one 80-row tile (as the fused launch does)
    const int chunk = (a.n_rows + cluster - 1) / cluster;
    const bool big = chunk > kBN && chunk <= kBigBN;
    if (D == 128)
        return big ? launch(attn_decode_kernel<128, false, kBigBN>, dim3(cluster), dim3(kThreads),
                            decode_smem<128, kBigBN>(), c, cluster, a, cmp::CompressArgs{})
                   : launch(attn_decode_kernel<128, false>, dim3(cluster), dim3(kThreads), decode_smem<128>(), c,
                            cluster, a, cmp::CompressArgs{});
    return big ? launch(attn_decode_kernel<64, false, kBigBN>, dim3(cluster), dim3(kThreads), decode_smem<64, kBigBN>(),
                        c, cluster, a, cmp::CompressArgs{})
               : launch(attn_decode_kernel<64, false>, dim3(cluster), dim3(kThreads), decode_smem<64>(), c, cluster, a,
                        cmp::CompressArgs{});
}

cudaError_t launch_compress_attn_decode(const uint16_t *k_new, const uint16_t *v_new, const float *score_w, int ratio,
                                        long long pos, float *state, const uint16_t *q, int H, int D,
                                        const uint16_t *win_k, const uint16_t *win_v, int n_win, uint16_t *comp_k,
                                        uint16_t *comp_v, float scale, uint16_t *out, const Ctx &c) {
    if (ratio > cmp::kMaxRatio || D > cmp::kMaxD) return cudaErrorInvalidValue;
    const long long n_vis = (pos + 1) / ratio;   // every visible row, the one this step may complete included
    DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.src = RowSrc{win_k, win_v, comp_k, comp_v, nullptr, c.err, n_vis, n_win};
    a.H = H;
    a.n_rows = n_win + static_cast<int>(n_vis);
    a.scale_log2 = scale * kLog2e;
    a.comp_first = (pos + 1) % ratio == 0;
    a.test_wait_ns = test_wait_limit_ns();
    const cmp::CompressArgs ca{k_new, v_new, score_w, state, comp_k, comp_v, pos, 1, D, ratio};
    int cluster = 16;
    cudaError_t e = D == 128 ? configure<128>(cluster) : configure<64>(cluster);
    if (e != cudaSuccess) return e;
    // the CTA that attends the last row (the row a completing step writes), as the kernel splits the rows
    const int chunk = (a.n_rows + cluster - 1) / cluster;
    a.comp_rank = a.comp_first ? (a.n_rows - 1) / chunk : 0;
    const bool big = chunk > kBN && chunk <= kBigBN;
    if (D == 128)
        return big ? launch(attn_decode_kernel<128, true, kBigBN>, dim3(cluster), dim3(kThreads),
                            decode_smem<128, kBigBN>(), c, cluster, a, ca)
                   : launch(attn_decode_kernel<128, true>, dim3(cluster), dim3(kThreads), decode_smem<128>(), c,
                            cluster, a, ca);
    return big ? launch(attn_decode_kernel<64, true, kBigBN>, dim3(cluster), dim3(kThreads), decode_smem<64, kBigBN>(),
                        c, cluster, a, ca)
               : launch(attn_decode_kernel<64, true>, dim3(cluster), dim3(kThreads), decode_smem<64>(), c, cluster, a,
                        ca);
}

cudaError_t launch_attn_decode_batched(int B, const uint16_t *q, int H, int D, const uint16_t *ring_k,
                                       const uint16_t *ring_v, int W, const long long *pos, const uint16_t *comp_k,
                                       const uint16_t *comp_v, long long cap, const int32_t *sel, int n_sel,
                                       int ratio, float scale, uint16_t *out, const float *score_w, float *state,
                                       const Ctx &c) {
    if (state != nullptr && (ratio > cmp::kMaxRatio || D > cmp::kMaxD)) return cudaErrorInvalidValue;
    DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.src = RowSrc{ring_k, ring_v, comp_k, comp_v, sel, c.err, cap, W};
    a.H = H;
    a.scale_log2 = scale * kLog2e;
    a.comp_rank = -1;
    a.test_wait_ns = test_wait_limit_ns();
    a.pos = pos;
    a.q_stride = static_cast<long long>(H) * D;
    a.win_stride = static_cast<long long>(W) * D;
    a.comp_stride = cap * D;
    a.sel_stride = n_sel;
    a.state_stride = 2 + 2LL * D;
    a.cap = cap;
    a.W = W;
    a.ratio = ratio;
    a.n_sel_list = sel ? n_sel : 0;
    int cluster = 16, active16 = 0, active8 = 0, active4 = 0;
    cudaError_t e = D == 128 ? configure<128>(cluster, &active16, &active8, &active4)
                             : configure<64>(cluster, &active16, &active8, &active4);
    if (e != cudaSuccess) return e;
    const long long rows = W + (sel ? static_cast<long long>(n_sel) : cap);   // the largest session's
    cluster = batched_cluster(B, rows, cluster, active16, active8, active4);
    const dim3 grid(cluster, B);
    if (state != nullptr) {   // the compressor's update for each session's token, in the same launch
        const cmp::CompressArgs ca{nullptr, nullptr, score_w, state, const_cast<uint16_t *>(comp_k),
                                   const_cast<uint16_t *>(comp_v), 0, 1, D, ratio};
        // one 80-row tile when the largest session's CTAs attend 65 .. 80 rows, as the
        // one-session launch does (a session that fits 64 rows gets the same bits either way)
        const long long chunk = (rows + cluster - 1) / cluster;
        const bool big = chunk > kBN && chunk <= kBigBN;
        if (D == 128)
            return big ? launch(attn_decode_kernel<128, true, kBigBN>, grid, dim3(kThreads),
                                decode_smem<128, kBigBN>(), c, cluster, a, ca)
                       : launch(attn_decode_kernel<128, true>, grid, dim3(kThreads), decode_smem<128>(), c, cluster,
                                a, ca);
        return big ? launch(attn_decode_kernel<64, true, kBigBN>, grid, dim3(kThreads), decode_smem<64, kBigBN>(), c,
                            cluster, a, ca)
                   : launch(attn_decode_kernel<64, true>, grid, dim3(kThreads), decode_smem<64>(), c, cluster, a,
                            ca);
    }
    if (D == 128)
        return launch(attn_decode_kernel<128, false>, grid, dim3(kThreads), decode_smem<128>(), c, cluster, a,
                      cmp::CompressArgs{});
    return launch(attn_decode_kernel<64, false>, grid, dim3(kThreads), decode_smem<64>(), c, cluster, a,
                  cmp::CompressArgs{});
}

cudaError_t launch_attn_prefill(const uint16_t *q, int T, int H, int D, const uint16_t *raw_k,
                                const uint16_t *raw_v, int n_prior, int window,
                                const uint16_t *comp_k, const uint16_t *comp_v, long long n_comp,
                                const int32_t *sel, int k_stride, long long q_pos0, int ratio,
                                float scale, uint16_t *out, const Ctx &c) {
    // the most selected (or visible) compressed rows of any query
    long long max_sel = 0;
    if (ratio > 0) {
        if (sel) max_sel = k_stride;
        else {
            const long long nv = (q_pos0 + T) / ratio;
            max_sel = nv < n_comp ? nv : n_comp;
        }
    }
    if (attn_prefill_tc_ok(q, out, T, H, D, n_prior, window, max_sel, n_comp))
        return launch_attn_prefill_tc(q, T, raw_k, raw_v, n_prior, window, comp_k, comp_v, n_comp, sel, k_stride,
                                      q_pos0, ratio, scale, out, c);
    PrefillArgs a{q, raw_k, raw_v, comp_k, comp_v, sel, out, c.err, n_comp, q_pos0,
                  H, n_prior, window, k_stride, ratio, scale * kLog2e};
    int cluster = 16;
    cudaError_t e;
    if (D == 128) {
        if ((e = configure<128>(cluster)) != cudaSuccess) return e;
        return launch(attn_prefill_kernel<128>, dim3(T), dim3(kThreads), prefill_smem<128>(), c, 1, a);
    }
    if ((e = configure<64>(cluster)) != cudaSuccess) return e;
    return launch(attn_prefill_kernel<64>, dim3(T), dim3(kThreads), prefill_smem<64>(), c, 1, a);
}

}  // namespace ds4a
