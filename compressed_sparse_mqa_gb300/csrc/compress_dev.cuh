// compress_dev.cuh -- device routines of the KV compressor, shared by the
// compressor kernel and by the decode kernel that runs the indexer and the
// one-token compressor update in one launch.
//
// "DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": pooled row of
// block b = sum_t a_t [k_t ; v_t], a = softmax_t(w . k_t); the running state of
// the open block is (m, l, acc_k[D], acc_v[D]): running max of the scores, sum of
// exp(s - m), and the exp(s - m)-weighted sums of K and V.  With per-token indexer
// keys (ki != nullptr) the same weights also pool them into the block's indexer
// key, and the state carries their weighted sum too: (m, l, acc_k[D], acc_v[D],
// acc_ki[DI]).  NT: threads of the calling block (every thread calls these
// routines: they synchronise the block).
#pragma once

#include "ds4a_common.cuh"

namespace ds4a {
namespace cmp {

constexpr int kMaxRatio = 1024;
constexpr int kMaxD = 256;

struct CompressArgs {
    const uint16_t *k;
    const uint16_t *v;
    const float *w;
    float *state;
    uint16_t *comp_k;
    uint16_t *comp_v;
    long long pos;
    int n_new;
    int D;
    int ratio;
    const uint16_t *ki = nullptr;   // [n_new, DI] per-token indexer keys, or nullptr
    uint16_t *comp_ki = nullptr;    // [cap, DI] pooled indexer keys
    int DI = 0;
};

// Scores s_i = w . k_i of tokens [t0, t1) into s_w: one warp per token, lanes
// over 8-dim chunks.  Reads only the caller's inputs (k, w).
template <int NT>
__device__ void segment_scores(const CompressArgs &a, long long t0, long long t1, float *s_w) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = a.D;
    const int n = static_cast<int>(t1 - t0);
    const uint16_t *kb = a.k + (t0 - a.pos) * D;
    for (int i = warp; i < n; i += NT / 32) {
        float acc = 0.f;
        for (int ch = lane; ch < D / 8; ch += 32) {
            uint4 raw = *reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(i) * D + ch * 8);
            const uint16_t *h = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(a.w[ch * 8 + e], h2f(h[e]), acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) s_w[i] = acc;
    }
    __syncthreads();
}

// Pool tokens [t0, t1) of block b (t1 - t0 <= ratio) whose scores are in s_w.  If
// `resume`, continue from the stored running state.  If t1 closes the block,
// write row b, else store the running state.
template <int NT>
__device__ void pool_segment(const CompressArgs &a, long long b, long long t0, long long t1,
                             bool resume, float *s_w, float *s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = a.D;
    const int n = static_cast<int>(t1 - t0);
    const uint16_t *kb = a.k + (t0 - a.pos) * D;
    const uint16_t *vb = a.v + (t0 - a.pos) * D;

    // segment max
    float m = -INFINITY;
    for (int i = tid; i < n; i += NT) m = fmaxf(m, s_w[i]);
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float m_seg = s_red[0];
#pragma unroll
    for (int wi = 1; wi < NT / 32; ++wi) m_seg = fmaxf(m_seg, s_red[wi]);

    float m_old = -INFINITY, l_old = 0.f;
    if (resume) { m_old = a.state[0]; l_old = a.state[1]; }
    const float m_new = fmaxf(m_old, m_seg);
    const float c_old = resume ? __expf(m_old - m_new) : 0.f;
    __syncthreads();   // everyone has read s_red before it is reused
    for (int i = tid; i < n; i += NT) s_w[i] = __expf(s_w[i] - m_new);
    __syncthreads();

    // l = c_old * l_old + sum_i e_i  (every thread sums in the same order)
    float l = c_old * l_old;
    for (int i = 0; i < n; ++i) l += s_w[i];

    const bool closes = (t1 % a.ratio) == 0;
    for (int d = tid; d < D; d += NT) {
        float ak = 0.f, av = 0.f;
        if (resume) { ak = c_old * a.state[2 + d]; av = c_old * a.state[2 + D + d]; }
        for (int i = 0; i < n; ++i) {
            const float e = s_w[i];
            ak = fmaf(e, h2f(kb[static_cast<size_t>(i) * D + d]), ak);
            av = fmaf(e, h2f(vb[static_cast<size_t>(i) * D + d]), av);
        }
        if (closes) {
            const float inv = 1.f / l;
            a.comp_k[b * D + d] = f2h(ak * inv);
            a.comp_v[b * D + d] = f2h(av * inv);
        } else {
            a.state[2 + d] = ak;
            a.state[2 + D + d] = av;
        }
    }
    if (a.ki != nullptr) {   // the indexer keys, pooled with the same weights
        const int DI = a.DI;
        const uint16_t *ib = a.ki + (t0 - a.pos) * DI;
        for (int d = tid; d < DI; d += NT) {
            float ai = resume ? c_old * a.state[2 + 2 * D + d] : 0.f;
            for (int i = 0; i < n; ++i) ai = fmaf(s_w[i], h2f(ib[static_cast<size_t>(i) * DI + d]), ai);
            if (closes) a.comp_ki[b * DI + d] = f2h(ai * (1.f / l));
            else a.state[2 + 2 * D + d] = ai;
        }
    }
    if (!closes && tid == 0) { a.state[0] = m_new; a.state[1] = l; }
    __syncthreads();
}

}  // namespace cmp
}  // namespace ds4a
