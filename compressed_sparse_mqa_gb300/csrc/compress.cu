// compress.cu -- the KV compressor: softmax-of-score pooling of every block of
// `ratio` tokens into one compressed K row and one V row.
//
// "DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": the
// compressor keeps a rolling score/KV state and appends a pooled row at every
// ratio boundary; prefill runs it over the chunk, decode one token at a time.
// Pooled row of block b: sum_t a_t [k_t ; v_t], a = softmax_t(w . k_t).
//
// Work split: one CTA of 128 threads per block touched by the call.  Blocks that
// start inside the call and complete inside it are pooled directly (one CTA
// each, in parallel).  The at most two "edge" blocks -- the one left open by
// the previous call (its running state is read) and the one this call leaves
// open (its running state is written) -- are both handled by CTA 0, in that
// order, so the state buffer is never read and written by different CTAs.
// The running state is (m, l, acc_k[D], acc_v[D]): running max of the scores,
// sum of exp(s - m), and the exp(s - m)-weighted sums of K and V.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace ds4a {
namespace {

constexpr int kThreads = 128;
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
};

// Scores s_i = w . k_i of tokens [t0, t1) into s_w: one warp per token, lanes
// over 8-dim chunks.  Reads only the caller's inputs (k, w).
__device__ void segment_scores(const CompressArgs &a, long long t0, long long t1, float *s_w) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = a.D;
    const int n = static_cast<int>(t1 - t0);
    const uint16_t *kb = a.k + (t0 - a.pos) * D;
    for (int i = warp; i < n; i += kThreads / 32) {
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
__device__ void pool_segment(const CompressArgs &a, long long b, long long t0, long long t1,
                             bool resume, float *s_w, float *s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = a.D;
    const int n = static_cast<int>(t1 - t0);
    const uint16_t *kb = a.k + (t0 - a.pos) * D;
    const uint16_t *vb = a.v + (t0 - a.pos) * D;

    // segment max
    float m = -INFINITY;
    for (int i = tid; i < n; i += kThreads) m = fmaxf(m, s_w[i]);
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float m_seg = s_red[0];
#pragma unroll
    for (int wi = 1; wi < kThreads / 32; ++wi) m_seg = fmaxf(m_seg, s_red[wi]);

    float m_old = -INFINITY, l_old = 0.f;
    if (resume) { m_old = a.state[0]; l_old = a.state[1]; }
    const float m_new = fmaxf(m_old, m_seg);
    const float c_old = resume ? __expf(m_old - m_new) : 0.f;
    __syncthreads();   // everyone has read s_red before it is reused
    for (int i = tid; i < n; i += kThreads) s_w[i] = __expf(s_w[i] - m_new);
    __syncthreads();

    // l = c_old * l_old + sum_i e_i  (every thread sums in the same order)
    float l = c_old * l_old;
    for (int i = 0; i < n; ++i) l += s_w[i];

    const bool closes = (t1 % a.ratio) == 0;
    for (int d = tid; d < D; d += kThreads) {
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
    if (!closes && tid == 0) { a.state[0] = m_new; a.state[1] = l; }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
    __shared__ float s_w[kMaxRatio];
    __shared__ float s_red[kThreads / 32];
    const long long r = a.ratio;
    const long long end = a.pos + a.n_new;
    const long long b_first = a.pos / r, b_last = (end - 1) / r;
    const bool first_open = (a.pos % r) != 0;
    const bool last_open = (end % r) != 0;
    const long long fc_lo = b_first + (first_open ? 1 : 0);
    // this CTA's segments: [t0a, t1a) of block ba (resumed if CTA 0 continues the
    // open block), then for CTA 0 possibly the block this call leaves open
    long long ba, t0a, t1a;
    bool resume_a;
    if (blockIdx.x == 0) {
        if (first_open) {
            ba = b_first;
            t0a = a.pos;
            t1a = (b_first + 1) * r < end ? (b_first + 1) * r : end;
            resume_a = true;
        } else {
            ba = b_last;
            t0a = b_last * r;
            t1a = end;
            resume_a = false;
        }
    } else {
        ba = fc_lo + blockIdx.x - 1;
        t0a = ba * r;
        t1a = (ba + 1) * r;
        resume_a = false;
    }
    const bool has_a = blockIdx.x != 0 || first_open || last_open;
    // The scores read only the caller's inputs: computed before waiting on the
    // previous kernel; the running state and the outputs are touched after it.
    if (has_a) segment_scores(a, t0a, t1a, s_w);
    pdl_wait();
    pdl_trigger();
    if (has_a) pool_segment(a, ba, t0a, t1a, resume_a, s_w, s_red);
    if (blockIdx.x == 0 && first_open && last_open && b_last != b_first) {
        segment_scores(a, b_last * r, end, s_w);
        pool_segment(a, b_last, b_last * r, end, false, s_w, s_red);
    }
}

}  // namespace

cudaError_t launch_compress(const uint16_t *k, const uint16_t *v, int n_new, int D, const float *w,
                            int ratio, long long pos, float *state, uint16_t *comp_k,
                            uint16_t *comp_v, const Ctx &c) {
    if (n_new <= 0) return cudaSuccess;
    if (ratio > kMaxRatio || D > kMaxD) return cudaErrorInvalidValue;
    const long long end = pos + n_new;
    const long long b_first = pos / ratio, b_last = (end - 1) / ratio;
    const bool first_open = (pos % ratio) != 0;
    const bool last_open = (end % ratio) != 0;
    long long n_fc = (b_last - (last_open ? 1 : 0)) - (b_first + (first_open ? 1 : 0)) + 1;
    if (n_fc < 0) n_fc = 0;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        // same shared-memory carveout as the other ds4a kernels: no reconfiguration between them
        cudaError_t e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CompressArgs a{k, v, w, state, comp_k, comp_v, pos, n_new, D, ratio};
    return launch(compress_kernel, dim3(static_cast<unsigned>(1 + n_fc)), dim3(kThreads), 0, c, 1, a);
}

}  // namespace ds4a
