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
#include "compress_dev.cuh"
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace ds4a {
namespace {

using cmp::CompressArgs;
using cmp::kMaxD;
using cmp::kMaxRatio;

constexpr int kThreads = 128;

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
    if (has_a) cmp::segment_scores<kThreads>(a, t0a, t1a, s_w);
    pdl_wait();
    pdl_trigger();
    if (has_a) cmp::pool_segment<kThreads>(a, ba, t0a, t1a, resume_a, s_w, s_red);
    if (blockIdx.x == 0 && first_open && last_open && b_last != b_first) {
        cmp::segment_scores<kThreads>(a, b_last * r, end, s_w);
        cmp::pool_segment<kThreads>(a, b_last, b_last * r, end, false, s_w, s_red);
    }
}

}  // namespace

cudaError_t launch_compress(const uint16_t *k, const uint16_t *v, int n_new, int D, const float *w,
                            int ratio, long long pos, float *state, uint16_t *comp_k,
                            uint16_t *comp_v, const Ctx &c, const uint16_t *ki, uint16_t *comp_ki, int DI) {
    if (n_new <= 0) return cudaSuccess;
    if (ratio > kMaxRatio || D > kMaxD || DI > kMaxD) return cudaErrorInvalidValue;
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
    CompressArgs a{k, v, w, state, comp_k, comp_v, pos, n_new, D, ratio, ki, comp_ki, ki ? DI : 0};
    return launch(compress_kernel, dim3(static_cast<unsigned>(1 + n_fc)), dim3(kThreads), 0, c, 1, a);
}

}  // namespace ds4a
