// ds4a_api.cu -- the C ABI: argument validation, per-device setup, dispatch to
// the kernel launchers, status strings and the device error word.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace {

// First error recorded by a kernel on this device (0 = none).
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;

// Filled once per device under g_mu; `ready` is stored with release order after the
// fields, and read with acquire order, so a thread that sees it set also sees them.
struct DeviceInfo {
    unsigned int *err = nullptr;
    int num_sms = 0;
    std::atomic<bool> ready{false};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

bool pdl_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("DS4A_PDL");
        return !(e && std::strcmp(e, "0") == 0);
    }();
    return on;
}

int make_ctx(void *stream, ds4a::Ctx &c) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DS4A_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return DS4A_ERR_CUDA;
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return DS4A_ERR_CUDA;
            d.err = static_cast<unsigned int *>(p);
            d.num_sms = sms;
            d.ready.store(true, std::memory_order_release);
        }
    }
    c.stream = static_cast<cudaStream_t>(stream);
    c.err = d.err;
    c.num_sms = d.num_sms;
    c.pdl = pdl_enabled();
    return DS4A_OK;
}

std::atomic<long long> g_test_wait_ns{0};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return DS4A_OK;
    cudaGetLastError();   // clear the sticky-free launch error
    return e == cudaErrorInvalidValue ? DS4A_ERR_UNSUPPORTED : DS4A_ERR_CUDA;
}

}  // namespace

long long ds4a::test_wait_limit_ns() { return g_test_wait_ns.load(std::memory_order_relaxed); }

extern "C" {

int ds4a_test_set_wait_limit(long long limit_ns) {
    if (limit_ns < 0 || limit_ns > 10000000000LL) return DS4A_ERR_ARG;
    g_test_wait_ns.store(limit_ns, std::memory_order_relaxed);
    return DS4A_OK;
}

const char *ds4a_status_str(int status) {
    switch (status) {
        case DS4A_OK: return "ok";
        case DS4A_ERR_ARG: return "invalid argument";
        case DS4A_ERR_CAPACITY: return "output capacity exceeded";
        case DS4A_ERR_UNSUPPORTED: return "unsupported shape";
        case DS4A_ERR_CUDA: return "CUDA error";
        case DS4A_ERR_TIMEOUT: return "device wait timed out";
        case DS4A_ERR_WORKSPACE: return "workspace missing or too small";
        case DS4A_ERR_DEVICE_INDEX: return "row index out of range (device)";
        default: return "unknown status";
    }
}

int ds4a_last_device_error(void *stream) {
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    if (cudaStreamSynchronize(c.stream) != cudaSuccess) return DS4A_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, c.err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DS4A_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(c.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return DS4A_ERR_CUDA;
    }
    return static_cast<int>(v);
}

int ds4a_compress_append(const uint16_t *k, const uint16_t *v, int n_new, int head_dim,
                         const float *score_w, int ratio, long long pos, float *state,
                         uint16_t *comp_k, uint16_t *comp_v, long long cap, void *stream) {
    if (n_new < 0 || pos < 0 || cap < 0 || ratio < 1) return DS4A_ERR_ARG;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0 || ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (n_new == 0) return DS4A_OK;
    if (!k || !v || !score_w || !state || !comp_k || !comp_v) return DS4A_ERR_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(score_w, 4) || !aligned(state, 4) ||
        !aligned(comp_k, 2) || !aligned(comp_v, 2))
        return DS4A_ERR_ARG;
    if ((pos + n_new) / ratio > cap) return DS4A_ERR_CAPACITY;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_compress(k, v, n_new, head_dim, score_w, ratio, pos, state, comp_k,
                                           comp_v, c));
}

int ds4a_compress_append_keys(const uint16_t *k, const uint16_t *v, const uint16_t *k_idx_tok, int n_new,
                              int head_dim, int d_idx, const float *score_w, int ratio, long long pos, float *state,
                              uint16_t *comp_k, uint16_t *comp_v, uint16_t *comp_kidx, long long cap, void *stream) {
    if (n_new < 0 || pos < 0 || cap < 0 || ratio < 1) return DS4A_ERR_ARG;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0 || ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0) return DS4A_ERR_UNSUPPORTED;
    if (n_new == 0) return DS4A_OK;
    if (!k || !v || !k_idx_tok || !score_w || !state || !comp_k || !comp_v || !comp_kidx) return DS4A_ERR_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_idx_tok, 16) || !aligned(score_w, 4) ||
        !aligned(state, 4) || !aligned(comp_k, 2) || !aligned(comp_v, 2) || !aligned(comp_kidx, 2))
        return DS4A_ERR_ARG;
    if ((pos + n_new) / ratio > cap) return DS4A_ERR_CAPACITY;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_compress(k, v, n_new, head_dim, score_w, ratio, pos, state, comp_k, comp_v, c,
                                           k_idx_tok, comp_kidx, d_idx));
}

size_t ds4a_indexer_workspace_bytes(int n_q, long long n_rows, int k) {
    if (n_q < 0 || n_rows < 0) return 0;
    return ds4a::indexer_ws_bytes(n_q, n_rows, k);
}

int ds4a_indexer_topk(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                      int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                      int32_t *out_n, void *ws, size_t ws_bytes, void *stream) {
    if (n_q < 0 || n_rows < 0 || q_pos0 < 0 || ratio < 1 || k < 1) return DS4A_ERR_ARG;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0 || k > 2048 || n_rows > 0x7fffffffLL)
        return DS4A_ERR_UNSUPPORTED;
    if (n_q == 0) return DS4A_OK;
    if (!q_idx || !out_idx || (n_rows > 0 && !k_idx)) return DS4A_ERR_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(out_idx, 4) || !aligned(out_n, 4))
        return DS4A_ERR_ARG;
    if (!ws || !aligned(ws, 16) || ws_bytes < ds4a::indexer_ws_bytes(n_q, n_rows, k)) return DS4A_ERR_WORKSPACE;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_indexer(q_idx, n_q, k_idx, n_rows, d_idx, q_pos0, ratio, k, out_idx,
                                          out_n, ws, c));
}

int ds4a_indexer_topk_compress(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows, int d_idx,
                               long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                               size_t ws_bytes, const uint16_t *k_new, const uint16_t *v_new, int head_dim,
                               const float *score_w, float *state, uint16_t *comp_k, uint16_t *comp_v,
                               long long cap, void *stream) {
    // the checks of ds4a_indexer_topk (n_q = 1) and of ds4a_compress_append (n_new = 1, pos = q_pos)
    if (n_rows < 0 || q_pos < 0 || ratio < 1 || k < 1 || cap < 0) return DS4A_ERR_ARG;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0 || k > 2048 || n_rows > 0x7fffffffLL)
        return DS4A_ERR_UNSUPPORTED;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0 || ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (!q_idx || !out_idx || (n_rows > 0 && !k_idx)) return DS4A_ERR_ARG;
    if (!k_new || !v_new || !score_w || !state || !comp_k || !comp_v) return DS4A_ERR_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(out_idx, 4) || !aligned(out_n, 4))
        return DS4A_ERR_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(score_w, 4) || !aligned(state, 4) ||
        !aligned(comp_k, 2) || !aligned(comp_v, 2))
        return DS4A_ERR_ARG;
    if (!ws || !aligned(ws, 16) || ws_bytes < ds4a::indexer_ws_bytes(1, n_rows, k)) return DS4A_ERR_WORKSPACE;
    if ((q_pos + 1) / ratio > cap) return DS4A_ERR_CAPACITY;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_indexer_compress(q_idx, k_idx, n_rows, d_idx, q_pos, ratio, k, out_idx, out_n, ws,
                                                   k_new, v_new, head_dim, score_w, state, comp_k, comp_v, c));
}

int ds4a_indexer_topk_compress_keys(const uint16_t *q_idx, uint16_t *k_idx, long long n_rows, int d_idx,
                                    long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                                    size_t ws_bytes, const uint16_t *k_new, const uint16_t *v_new,
                                    const uint16_t *k_idx_tok, int head_dim, const float *score_w, float *state,
                                    uint16_t *comp_k, uint16_t *comp_v, long long cap, void *stream) {
    // the checks of ds4a_compress_append_keys (n_new = 1, comp_kidx = k_idx) and of ds4a_indexer_topk (n_q = 1)
    if (n_rows < 0 || q_pos < 0 || ratio < 1 || k < 1 || cap < 0) return DS4A_ERR_ARG;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0 || k > 2048 || n_rows > 0x7fffffffLL)
        return DS4A_ERR_UNSUPPORTED;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0 || ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (!q_idx || !out_idx || !k_idx) return DS4A_ERR_ARG;
    if (!k_new || !v_new || !k_idx_tok || !score_w || !state || !comp_k || !comp_v) return DS4A_ERR_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(out_idx, 4) || !aligned(out_n, 4))
        return DS4A_ERR_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_idx_tok, 16) || !aligned(score_w, 4) ||
        !aligned(state, 4) || !aligned(comp_k, 2) || !aligned(comp_v, 2))
        return DS4A_ERR_ARG;
    if (!ws || !aligned(ws, 16) || ws_bytes < ds4a::indexer_ws_bytes(1, n_rows, k)) return DS4A_ERR_WORKSPACE;
    // the row the token completes is written to comp_k, comp_v and k_idx
    if ((q_pos + 1) / ratio > (cap < n_rows ? cap : n_rows)) return DS4A_ERR_CAPACITY;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_indexer_compress(q_idx, k_idx, n_rows, d_idx, q_pos, ratio, k, out_idx, out_n, ws,
                                                   k_new, v_new, head_dim, score_w, state, comp_k, comp_v, c,
                                                   k_idx_tok));
}

static int check_heads(int H, int D) {
    if (D != 64 && D != 128) return DS4A_ERR_UNSUPPORTED;
    if (H < 8 || H > 64 || H % 8 != 0) return DS4A_ERR_UNSUPPORTED;
    return DS4A_OK;
}

int ds4a_attn_decode(const uint16_t *q, int H, int D, const uint16_t *win_k,
                     const uint16_t *win_v, int n_win, const uint16_t *comp_k,
                     const uint16_t *comp_v, long long n_comp, const int32_t *sel, int n_sel,
                     float scale, uint16_t *out, void *ws, size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    int rc = check_heads(H, D);
    if (rc != DS4A_OK) return rc;
    if (n_win < 1 || n_win > 4096 || n_sel < 0 || n_comp < 0) return DS4A_ERR_ARG;
    if (n_sel > 0x7fffffff - n_win) return DS4A_ERR_UNSUPPORTED;   // n_win + n_sel must fit in int
    if (!q || !win_k || !win_v || !out) return DS4A_ERR_ARG;
    if (n_sel > 0 && (!comp_k || !comp_v)) return DS4A_ERR_ARG;
    if (!sel && n_sel > n_comp) return DS4A_ERR_ARG;
    if (!aligned(q, 4) || !aligned(win_k, 16) || !aligned(win_v, 16) || !aligned(comp_k, 16) ||
        !aligned(comp_v, 16) || !aligned(sel, 4) || !aligned(out, 16))
        return DS4A_ERR_ARG;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_attn_decode(q, H, D, win_k, win_v, n_win, comp_k, comp_v, n_comp, sel,
                                              n_sel, scale, out, c));
}

int ds4a_compress_attn_decode(const uint16_t *k_new, const uint16_t *v_new, const float *score_w, int ratio,
                              long long pos, float *state, uint16_t *comp_k, uint16_t *comp_v, long long cap,
                              const uint16_t *q, int H, int D, const uint16_t *win_k, const uint16_t *win_v,
                              int n_win, float scale, uint16_t *out, void *stream) {
    // the checks of ds4a_compress_append (n_new = 1, head_dim = D) and of ds4a_attn_decode
    // (sel = NULL, n_sel = floor((pos+1)/ratio), n_comp = cap)
    if (pos < 0 || cap < 0 || ratio < 1) return DS4A_ERR_ARG;
    int rc = check_heads(H, D);
    if (rc != DS4A_OK) return rc;
    if (ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (n_win < 1 || n_win > 4096) return DS4A_ERR_ARG;
    if (!k_new || !v_new || !score_w || !state || !comp_k || !comp_v || !q || !win_k || !win_v || !out)
        return DS4A_ERR_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(score_w, 4) || !aligned(state, 4) ||
        !aligned(comp_k, 16) || !aligned(comp_v, 16) || !aligned(q, 4) || !aligned(win_k, 16) ||
        !aligned(win_v, 16) || !aligned(out, 16))
        return DS4A_ERR_ARG;
    if ((pos + 1) / ratio > cap) return DS4A_ERR_CAPACITY;
    if (n_win + (pos + 1) / ratio > 0x7fffffffLL) return DS4A_ERR_UNSUPPORTED;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_compress_attn_decode(k_new, v_new, score_w, ratio, pos, state, q, H, D, win_k,
                                                       win_v, n_win, comp_k, comp_v, scale, out, c));
}

int ds4a_attn_prefill(const uint16_t *q, int T, int H, int D, const uint16_t *raw_k,
                      const uint16_t *raw_v, int n_prior, int window, const uint16_t *comp_k,
                      const uint16_t *comp_v, long long n_comp, const int32_t *sel, int k_stride,
                      long long q_pos0, int ratio, float scale, uint16_t *out, void *ws,
                      size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    int rc = check_heads(H, D);
    if (rc != DS4A_OK) return rc;
    if (T < 0 || window < 1 || window > 4096 || n_prior < 0 || q_pos0 < 0 || ratio < 0 || n_comp < 0)
        return DS4A_ERR_ARG;
    if (n_prior > q_pos0) return DS4A_ERR_ARG;
    const long long need_prior = (window - 1) < q_pos0 ? (window - 1) : q_pos0;
    if (n_prior < need_prior) return DS4A_ERR_ARG;
    if (T == 0) return DS4A_OK;
    if (!q || !raw_k || !raw_v || !out) return DS4A_ERR_ARG;
    if (ratio > 0 && n_comp > 0 && (!comp_k || !comp_v)) return DS4A_ERR_ARG;
    if (sel && k_stride < 1) return DS4A_ERR_ARG;
    if (!aligned(q, 4) || !aligned(raw_k, 16) || !aligned(raw_v, 16) || !aligned(comp_k, 16) ||
        !aligned(comp_v, 16) || !aligned(sel, 4) || !aligned(out, 4))
        return DS4A_ERR_ARG;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_attn_prefill(q, T, H, D, raw_k, raw_v, n_prior, window, comp_k, comp_v,
                                               n_comp, sel, k_stride, q_pos0, ratio, scale, out, c));
}

int ds4a_probe_gather(const uint16_t *table, long long n_table, int D, const int32_t *idx, long long n_idx,
                      unsigned int *sink, void *stream) {
    if (n_table < 0 || n_idx < 0 || D < 8 || D > 256 || D % 8 != 0) return DS4A_ERR_ARG;
    if (n_idx == 0) return DS4A_OK;
    if (!table || !idx || !sink || !aligned(table, 16) || !aligned(idx, 4) || !aligned(sink, 4)) return DS4A_ERR_ARG;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_gather_probe(table, n_table, D, idx, n_idx, sink, c));
}

// ---- batched decode: B independent sessions per call ------------------------------------

size_t ds4a_decode_batched_workspace_bytes(int B, long long cap) {
    if (B < 0 || cap < 0) return 0;
    return static_cast<size_t>(B) * ds4a::indexer_batched_ws_stride(cap);
}

static int check_batch(int B, int W, long long cap, const long long *pos) {
    if (B < 0 || cap < 0 || W < 1 || W > 4096) return DS4A_ERR_ARG;
    if (B > 65535 || cap > 0x7fffffffLL) return DS4A_ERR_UNSUPPORTED;
    if (B > 0 && (!pos || !aligned(pos, 8))) return DS4A_ERR_ARG;
    return DS4A_OK;
}

int ds4a_indexer_topk_compress_batched(int B, const uint16_t *q_idx, const uint16_t *k_idx, long long cap,
                                       int d_idx, const long long *pos, int ratio, int k, int32_t *out_idx,
                                       int32_t *out_n, void *ws, size_t ws_bytes, const uint16_t *ring_k,
                                       const uint16_t *ring_v, int W, int head_dim, const float *score_w,
                                       float *state, uint16_t *comp_k, uint16_t *comp_v, void *stream) {
    int rc = check_batch(B, W, cap, pos);
    if (rc != DS4A_OK) return rc;
    if (ratio < 1 || k < 1) return DS4A_ERR_ARG;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0 || k > 2048) return DS4A_ERR_UNSUPPORTED;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0 || ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (B == 0) return DS4A_OK;
    if (!q_idx || !out_idx || (cap > 0 && !k_idx) || !ring_k || !ring_v || !score_w || !state || !comp_k ||
        !comp_v)
        return DS4A_ERR_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(out_idx, 4) || !aligned(out_n, 4) ||
        !aligned(ring_k, 16) || !aligned(ring_v, 16) || !aligned(score_w, 4) || !aligned(state, 4) ||
        !aligned(comp_k, 2) || !aligned(comp_v, 2))
        return DS4A_ERR_ARG;
    if (!ws || !aligned(ws, 256) || ws_bytes < ds4a_decode_batched_workspace_bytes(B, cap)) return DS4A_ERR_WORKSPACE;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_indexer_compress_batched(B, q_idx, k_idx, cap, d_idx, pos, ratio, k, out_idx, out_n,
                                                           ws, ring_k, ring_v, W, head_dim, score_w, state, comp_k,
                                                           comp_v, c));
}

static int attn_batched_common(int B, const uint16_t *q, int H, int D, const uint16_t *ring_k, const uint16_t *ring_v,
                               int W, const long long *pos, const uint16_t *comp_k, const uint16_t *comp_v,
                               long long cap, int ratio, uint16_t *out) {
    int rc = check_batch(B, W, cap, pos);
    if (rc != DS4A_OK) return rc;
    rc = check_heads(H, D);
    if (rc != DS4A_OK) return rc;
    if (ratio < 0) return DS4A_ERR_ARG;
    if (ratio > 1024) return DS4A_ERR_UNSUPPORTED;
    if (B > 0 && (!q || !ring_k || !ring_v || !out || (ratio > 0 && cap > 0 && (!comp_k || !comp_v))))
        return DS4A_ERR_ARG;
    if (!aligned(q, 4) || !aligned(ring_k, 16) || !aligned(ring_v, 16) || !aligned(comp_k, 16) ||
        !aligned(comp_v, 16) || !aligned(out, 16))
        return DS4A_ERR_ARG;
    if (W + cap > 0x7fffffffLL) return DS4A_ERR_UNSUPPORTED;
    return DS4A_OK;
}

int ds4a_attn_decode_batched(int B, const uint16_t *q, int H, int D, const uint16_t *ring_k, const uint16_t *ring_v,
                             int W, const long long *pos, const uint16_t *comp_k, const uint16_t *comp_v,
                             long long cap, const int32_t *sel, int n_sel, int ratio, float scale, uint16_t *out,
                             void *stream) {
    int rc = attn_batched_common(B, q, H, D, ring_k, ring_v, W, pos, comp_k, comp_v, cap, ratio, out);
    if (rc != DS4A_OK) return rc;
    if (n_sel < 0 || !aligned(sel, 4)) return DS4A_ERR_ARG;
    if (sel && (n_sel > 0x7fffffff - W)) return DS4A_ERR_UNSUPPORTED;
    if (B == 0) return DS4A_OK;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_attn_decode_batched(B, q, H, D, ring_k, ring_v, W, pos, comp_k, comp_v, cap, sel,
                                                      n_sel, ratio, scale, out, nullptr, nullptr, c));
}

int ds4a_compress_attn_decode_batched(int B, const float *score_w, int ratio, float *state, uint16_t *comp_k,
                                      uint16_t *comp_v, long long cap, const uint16_t *q, int H, int D,
                                      const uint16_t *ring_k, const uint16_t *ring_v, int W, const long long *pos,
                                      float scale, uint16_t *out, void *stream) {
    int rc = attn_batched_common(B, q, H, D, ring_k, ring_v, W, pos, comp_k, comp_v, cap, ratio, out);
    if (rc != DS4A_OK) return rc;
    if (ratio < 1) return DS4A_ERR_ARG;
    if (B > 0 && (!score_w || !state || !comp_k || !comp_v)) return DS4A_ERR_ARG;
    if (!aligned(score_w, 4) || !aligned(state, 4)) return DS4A_ERR_ARG;
    if (B == 0) return DS4A_OK;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    return from_cuda(ds4a::launch_attn_decode_batched(B, q, H, D, ring_k, ring_v, W, pos, comp_k, comp_v, cap,
                                                      nullptr, 0, ratio, scale, out, score_w, state, c));
}

// ---- one decode step of one layer from host memory ------------------------------------------

// Every check that the calls ds4a_decode_layer_step makes would make, done before
// anything is enqueued (so that a failing call leaves the device arrays as they were).
static int check_layer(const ds4a_decode_layer_t *L, long long pos) {
    if (!L || pos < 0) return DS4A_ERR_ARG;
    int rc = check_heads(L->H, L->D);
    if (rc != DS4A_OK) return rc;
    if (L->W < 1 || L->W > 4096 || L->ratio < 0 || L->topk < 0 || L->cap < 0) return DS4A_ERR_ARG;
    if (L->ratio > 1024 || L->topk > 2048) return DS4A_ERR_UNSUPPORTED;
    if ((L->topk > 0 && L->ratio == 0) || (L->pooled_keys && L->topk == 0)) return DS4A_ERR_ARG;
    if (!L->ring_k || !L->ring_v || !L->q || !L->out) return DS4A_ERR_ARG;
    if (!aligned(L->ring_k, 16) || !aligned(L->ring_v, 16) || !aligned(L->q, 16) || !aligned(L->out, 16))
        return DS4A_ERR_ARG;
    if (L->ratio > 0) {
        if (!L->score_w || !L->state || !L->comp_k || !L->comp_v) return DS4A_ERR_ARG;
        if (!aligned(L->score_w, 4) || !aligned(L->state, 4) || !aligned(L->comp_k, 16) || !aligned(L->comp_v, 16))
            return DS4A_ERR_ARG;
        if ((pos + 1) / L->ratio > L->cap) return DS4A_ERR_CAPACITY;
        if (L->W + (pos + 1) / L->ratio > 0x7fffffffLL) return DS4A_ERR_UNSUPPORTED;
    }
    if (L->topk > 0) {
        if (L->d_idx < 8 || L->d_idx > 256 || L->d_idx % 8 != 0 || L->cap > 0x7fffffffLL) return DS4A_ERR_UNSUPPORTED;
        if (!L->q_idx || !L->out_idx || (L->cap > 0 && !L->k_idx) || (L->pooled_keys && !L->k_idx_tok))
            return DS4A_ERR_ARG;
        if (!aligned(L->q_idx, 16) || !aligned(L->k_idx, 16) || !aligned(L->k_idx_tok, 16) ||
            !aligned(L->out_idx, 4) || !aligned(L->out_n, 4))
            return DS4A_ERR_ARG;
        if (!L->ws || !aligned(L->ws, 16) || L->ws_bytes < ds4a::indexer_ws_bytes(1, L->cap, L->topk))
            return DS4A_ERR_WORKSPACE;
    }
    return DS4A_OK;
}

// The device-visible address of a page-locked (or registered) host buffer, or nullptr
// for any other pointer.
static const void *device_view(const void *p) {
    if (!p) return nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int ds4a_decode_layer_step(const ds4a_decode_layer_t *L, long long pos, const ds4a_decode_host_inputs_t *in,
                           uint16_t *out_host, void *stream) {
    int rc = check_layer(L, pos);
    if (rc != DS4A_OK) return rc;
    const int H = L->H, D = L->D;
    const long long slot = pos % L->W;
    const int n_win = static_cast<int>(pos + 1 < L->W ? pos + 1 : L->W);
    uint16_t *k_new = L->ring_k + slot * D;
    uint16_t *v_new = L->ring_v + slot * D;
    ds4a::Ctx c;
    rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;

    // the token's inputs, each to its device array
    const unsigned row = static_cast<unsigned>(D) * 2, idx_row = static_cast<unsigned>(L->d_idx) * 2;
    ds4a::IngestArgs ing{};
    auto add = [&](void *dst, const void *src, unsigned n) {
        if (src) ing.seg[ing.n++] = ds4a::IngestSeg{src, dst, n};
    };
    if (in) {
        add(k_new, in->k, row);
        add(v_new, in->v, row);
        add(L->q, in->q, static_cast<unsigned>(H) * row);
        if (L->topk > 0) {
            add(L->q_idx, in->q_idx, idx_row);
            if (L->pooled_keys) add(L->k_idx_tok, in->k_idx_tok, idx_row);
            else if ((pos + 1) % L->ratio == 0)
                add(L->k_idx + ((pos + 1) / L->ratio - 1) * L->d_idx, in->k_idx_row, idx_row);
        }
    }
    // Page-locked inputs: one kernel reads them over the host link and writes the arrays.
    // On an indexer layer the first kernel after it reads its own inputs (the indexer
    // query, the token's K, V and indexer key) from the host buffers and runs beside it;
    // the kernel after that starts once it has finished.  On the other layers the first
    // kernel reads window rows early, so it is launched without programmatic dependence
    // and starts once the input kernel has finished.  Other host memory: one copy each.
    ds4a::IngestArgs views = ing;
    bool mapped = true;
    for (int s = 0; s < ing.n && mapped; ++s) mapped = (views.seg[s].src = device_view(ing.seg[s].src)) != nullptr;
    const uint16_t *q_idx_r = L->q_idx, *k_r = k_new, *v_r = v_new, *ki_tok_r = L->k_idx_tok;
    ds4a::Ctx c_first = c;
    if (ing.n > 0 && mapped) {
        if (ds4a::launch_ingest(views, c) != cudaSuccess) {
            cudaGetLastError();
            return DS4A_ERR_CUDA;
        }
        if (L->topk > 0) {
            auto view = [](const uint16_t *host, const uint16_t *dflt) {
                return host ? static_cast<const uint16_t *>(device_view(host)) : dflt;
            };
            q_idx_r = view(in->q_idx, q_idx_r);
            k_r = view(in->k, k_r);
            v_r = view(in->v, v_r);
            if (L->pooled_keys) ki_tok_r = view(in->k_idx_tok, ki_tok_r);
        } else {
            c_first.pdl = false;
        }
    } else {
        for (int s = 0; s < ing.n; ++s)
            if (cudaMemcpyAsync(ing.seg[s].dst, ing.seg[s].src, ing.seg[s].bytes, cudaMemcpyHostToDevice, c.stream) !=
                cudaSuccess) {
                cudaGetLastError();
                return DS4A_ERR_CUDA;
            }
    }
    // a page-locked output buffer is written by the attention kernel directly
    const void *out_view = device_view(out_host);
    const bool out_direct = out_view != nullptr && aligned(out_view, 16);
    uint16_t *out = out_direct ? static_cast<uint16_t *>(const_cast<void *>(out_view)) : L->out;

    // the step's launches (the device calls' launchers; every check has passed)
    cudaError_t e = cudaSuccess;
    if (L->topk > 0) {
        if (L->pooled_keys) {
            e = ds4a::launch_indexer_compress(q_idx_r, L->k_idx, L->cap, L->d_idx, pos, L->ratio, L->topk, L->out_idx,
                                              L->out_n, L->ws, k_r, v_r, D, L->score_w, L->state, L->comp_k,
                                              L->comp_v, c_first, ki_tok_r);
        } else {
            e = ds4a::launch_indexer_compress(q_idx_r, L->k_idx, L->cap, L->d_idx, pos, L->ratio, L->topk, L->out_idx,
                                              L->out_n, L->ws, k_r, v_r, D, L->score_w, L->state, L->comp_k,
                                              L->comp_v, c_first);
        }
        if (e == cudaSuccess)
            e = ds4a::launch_attn_decode(L->q, H, D, L->ring_k, L->ring_v, n_win, L->comp_k, L->comp_v, L->cap,
                                         L->out_idx, L->topk, L->scale, out, c);
    } else if (L->ratio > 0) {
        e = ds4a::launch_compress_attn_decode(k_new, v_new, L->score_w, L->ratio, pos, L->state, L->q, H, D, L->ring_k,
                                              L->ring_v, n_win, L->comp_k, L->comp_v, L->scale, out, c_first);
    } else {
        e = ds4a::launch_attn_decode(L->q, H, D, L->ring_k, L->ring_v, n_win, nullptr, nullptr, 0, nullptr, 0,
                                     L->scale, out, c_first);
    }
    if (e != cudaSuccess) return from_cuda(e);
    if (out_host) {
        if ((!out_direct && cudaMemcpyAsync(out_host, L->out, static_cast<size_t>(H) * row, cudaMemcpyDeviceToHost,
                                            c.stream) != cudaSuccess) ||
            cudaStreamSynchronize(c.stream) != cudaSuccess) {
            cudaGetLastError();
            return DS4A_ERR_CUDA;
        }
    }
    return DS4A_OK;
}

}  // extern "C"

// ---- indexer entry point that allocates nothing -------------------------------------------
// Some callers cannot give the library a workspace: plugin and callback hosts
// whose enqueue step must not allocate device memory (an allocation there can
// synchronise the device or is simply not allowed by the host), and callers that
// run under a fixed, pre-reserved memory budget.  For them this file keeps the
// one-query indexer's scratch (ticket header + one u32 key per visible row) in a
// statically sized device array that every GPU loading the library holds until
// the process exits.
namespace {

constexpr long long kNoAllocMaxRows = 65536;   // 65536 visible rows: 256 KiB of keys
constexpr size_t kNoAllocHeaderBytes = 256;
constexpr size_t kNoAllocScratchBytes = kNoAllocHeaderBytes + kNoAllocMaxRows * sizeof(uint32_t);

// Zero when the module loads.  The indexer kernel's last CTA puts the completion
// ticket in the header back to zero when it finishes, so no call has to clear it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per device (with that device current);
// `ready` is stored with release order after the address, read with acquire order.
struct NoAllocSlot {
    void *addr = nullptr;
    std::atomic<bool> ready{false};
};
NoAllocSlot g_noalloc[kMaxDevices];

}  // namespace

extern "C" int ds4a_indexer_topk_noalloc(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows,
                                         int d_idx, long long q_pos, int ratio, int k, int32_t *out_idx,
                                         int32_t *out_n, void *stream) {
    if (n_rows < 0 || q_pos < 0 || ratio < 1 || k < 1) return DS4A_ERR_ARG;
    if (d_idx < 8 || d_idx > 256 || d_idx % 8 != 0 || k > 2048) return DS4A_ERR_UNSUPPORTED;
    // the kernel scores (and keeps a key for) the visible rows only
    const long long n_vis = (q_pos + 1) / ratio < n_rows ? (q_pos + 1) / ratio : n_rows;
    if (n_vis > kNoAllocMaxRows) return DS4A_ERR_WORKSPACE;   // beyond the built-in scratch
    if (!q_idx || !out_idx || (n_vis > 0 && !k_idx)) return DS4A_ERR_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(out_idx, 4) || !aligned(out_n, 4))
        return DS4A_ERR_ARG;
    if (ds4a::indexer_ws_bytes(1, n_vis, k) > kNoAllocScratchBytes) return DS4A_ERR_WORKSPACE;
    ds4a::Ctx c;
    int rc = make_ctx(stream, c);
    if (rc != DS4A_OK) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS4A_ERR_CUDA;
    NoAllocSlot &slot = g_noalloc[dev];
    if (!slot.ready.load(std::memory_order_acquire)) {
        // once per device, with that device current: the device address of the array
        std::lock_guard<std::mutex> lock(g_mu);
        if (!slot.ready.load(std::memory_order_relaxed)) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
                cudaGetLastError();
                return DS4A_ERR_CUDA;
            }
            slot.addr = p;
            slot.ready.store(true, std::memory_order_release);
        }
    }
    // rows past n_vis are never read: the call is the same as one over the visible rows
    return from_cuda(ds4a::launch_indexer(q_idx, 1, k_idx, n_vis, d_idx, q_pos, ratio, k, out_idx, out_n,
                                          slot.addr, c));
}
