// ds4a_internal.h -- launchers behind the C ABI (one per kernel family).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ds4a {

struct Ctx {
    cudaStream_t stream;
    unsigned int *err;   // device error word of the current device
    int num_sms;
    bool pdl;            // launch with programmatic stream serialization
};

// ki/comp_ki/DI: per-token indexer keys pooled with the same weights (ki = nullptr: none)
cudaError_t launch_compress(const uint16_t *k, const uint16_t *v, int n_new, int D, const float *w,
                            int ratio, long long pos, float *state, uint16_t *comp_k,
                            uint16_t *comp_v, const Ctx &c, const uint16_t *ki = nullptr,
                            uint16_t *comp_ki = nullptr, int DI = 0);

size_t indexer_ws_bytes(int n_q, long long n_rows, int k);

// test hook (ds4a_test_set_wait_limit): 0, or the limit of the extra never-completed wait
long long test_wait_limit_ns();
cudaError_t launch_indexer(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                           int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                           int32_t *out_n, void *ws, const Ctx &c);

// one decode query's indexer and the one-token compressor update of the same step,
// in one launch (the compressor's arguments as launch_compress with n_new = 1, pos = q_pos)
// k_idx_tok != nullptr: the compressor also pools the tokens' indexer keys into k_idx
// (ds4a_compress_append_keys), and a row the token completes is ranked by its pooled key
cudaError_t launch_indexer_compress(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows, int d_idx,
                                   long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                                   const uint16_t *k_new, const uint16_t *v_new, int D, const float *score_w,
                                   float *state, uint16_t *comp_k, uint16_t *comp_v, const Ctx &c,
                                   const uint16_t *k_idx_tok = nullptr);

// batched decode (B sessions, positions pos[B] in device memory): the indexer query
// and the compressor update of each session's token; workspace bytes per session
size_t indexer_batched_ws_stride(long long cap);
cudaError_t launch_indexer_compress_batched(int B, const uint16_t *q_idx, const uint16_t *k_idx, long long cap,
                                           int d_idx, const long long *pos, int ratio, int k, int32_t *out_idx,
                                           int32_t *out_n, void *ws, const uint16_t *ring_k, const uint16_t *ring_v,
                                           int W, int D, const float *score_w, float *state, uint16_t *comp_k,
                                           uint16_t *comp_v, const Ctx &c);
// batched decode attention; state != nullptr: with each session's compressor update
cudaError_t launch_attn_decode_batched(int B, const uint16_t *q, int H, int D, const uint16_t *ring_k,
                                       const uint16_t *ring_v, int W, const long long *pos, const uint16_t *comp_k,
                                       const uint16_t *comp_v, long long cap, const int32_t *sel, int n_sel,
                                       int ratio, float scale, uint16_t *out, const float *score_w, float *state,
                                       const Ctx &c);

// tensor-core prefill indexer (many queries): availability, workspace, launch
bool indexer_prefill_tc_ok(int n_q, long long n_rows, int d_idx);
size_t indexer_prefill_tc_ws_bytes(int n_q, long long n_rows);
cudaError_t launch_indexer_prefill_tc(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                                      int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                                      int32_t *out_n, void *ws, const Ctx &c);

cudaError_t launch_attn_decode(const uint16_t *q, int H, int D, const uint16_t *win_k,
                               const uint16_t *win_v, int n_win, const uint16_t *comp_k,
                               const uint16_t *comp_v, long long n_comp, const int32_t *sel,
                               int n_sel, float scale, uint16_t *out, const Ctx &c);

// the compressor's update for one decode token (as launch_compress with n_new = 1) and attention over the
// window and every visible compressed row floor((pos+1)/ratio), in one launch
cudaError_t launch_compress_attn_decode(const uint16_t *k_new, const uint16_t *v_new, const float *score_w, int ratio,
                                        long long pos, float *state, const uint16_t *q, int H, int D,
                                        const uint16_t *win_k, const uint16_t *win_v, int n_win, uint16_t *comp_k,
                                        uint16_t *comp_v, float scale, uint16_t *out, const Ctx &c);

// tensor-core prefill attention (64 heads, head_dim 128, <= 768 keys per query)
// the tensor-core prefill path takes H = 64, D = 128, 16-byte aligned queries and outputs, and
// key lists of at most 6 tiles of 128 (window tiles + selected-row tiles)
bool attn_prefill_tc_ok(const uint16_t *q, const uint16_t *out, int T, int H, int D, int n_prior, int window,
                        long long max_sel, long long n_comp);
cudaError_t launch_attn_prefill_tc(const uint16_t *q, int T, const uint16_t *raw_k, const uint16_t *raw_v,
                                   int n_prior, int window, const uint16_t *comp_k, const uint16_t *comp_v,
                                   long long n_comp, const int32_t *sel, int k_stride, long long q_pos0,
                                   int ratio, float scale, uint16_t *out, const Ctx &c);

cudaError_t launch_attn_prefill(const uint16_t *q, int T, int H, int D, const uint16_t *raw_k,
                                const uint16_t *raw_v, int n_prior, int window,
                                const uint16_t *comp_k, const uint16_t *comp_v, long long n_comp,
                                const int32_t *sel, int k_stride, long long q_pos0, int ratio,
                                float scale, uint16_t *out, const Ctx &c);

// ds4a_decode_layer_step's input kernel: up to kIngestSegs copies from device-visible
// (page-locked, mapped) host memory into device arrays; sizes are even byte counts
constexpr int kIngestSegs = 6;
struct IngestSeg {
    const void *src;
    void *dst;
    unsigned bytes;
};
struct IngestArgs {
    IngestSeg seg[kIngestSegs];
    int n;
};
cudaError_t launch_ingest(const IngestArgs &a, const Ctx &c);

// measurement kernel: gather n_idx rows table[idx[i]] (D fp16 each) into shared memory
cudaError_t launch_gather_probe(const uint16_t *table, long long n_table, int D, const int32_t *idx, long long n_idx,
                                unsigned int *sink, const Ctx &c);

// Launch helper: optional programmatic-dependent-launch attribute, optional cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, const Ctx &c,
                   int cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ds4a
