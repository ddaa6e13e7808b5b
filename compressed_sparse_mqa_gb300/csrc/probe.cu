// probe.cu -- a measurement kernel, not a step of the attention path: the rate at which
// this GPU gathers rows by index from global memory into shared memory.  Prefill
// attention is bound by that data movement (every query gathers its own window and
// kept compressed rows), so the benchmark reports the attention kernel's gathered
// bytes per second against this kernel's rate on the same rows.
//
// Every CTA takes tiles of 128 indices in turn; for a tile its threads copy each row's
// 16-byte chunks with cp.async into one of three shared-memory stages (two tiles in
// flight while the next is issued).  Indices outside the table are skipped and
// recorded as DS4A_ERR_DEVICE_INDEX.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace ds4a {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeRows = 128;    // rows per tile
constexpr int kProbeStages = 3;    // tiles in flight per CTA

__global__ void __launch_bounds__(kProbeThreads) gather_probe_kernel(const uint16_t *table, long long n_table, int D,
                                                                     const int32_t *idx, long long n_idx,
                                                                     unsigned int *err, unsigned int *sink) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ long long s_row[kProbeStages][kProbeRows];   // the rows of the tiles in flight
    pdl_wait();
    pdl_trigger();
    const int chunks = D / 8;                      // 16-byte chunks per row
    const size_t stage_bytes = static_cast<size_t>(kProbeRows) * D * 2;
    const long long n_tiles = (n_idx + kProbeRows - 1) / kProbeRows;
    // a tile's indices are read into shared memory one tile ahead of its copies, so no
    // copy waits on the load of its own index
    auto fetch_rows = [&](long long t, int st) {
        if (threadIdx.x < kProbeRows) {
            const long long r = t * kProbeRows + threadIdx.x;
            long long row = -1;
            if (t < n_tiles && r < n_idx) {
                row = idx[r];
                if (row < 0 || row >= n_table) {
                    record_error(err, DS4A_ERR_DEVICE_INDEX);
                    row = -1;
                }
            }
            s_row[st][threadIdx.x] = row;
        }
    };
    fetch_rows(blockIdx.x, 0);
    int it = 0;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
        const int st = it % kProbeStages;
        __syncthreads();   // s_row[st] is filled; s_row[(it + 1) % stages] is no longer read
        fetch_rows(t + gridDim.x, (it + 1) % kProbeStages);
        unsigned char *dst = smem + st * stage_bytes;
        for (int i = threadIdx.x; i < kProbeRows * chunks; i += kProbeThreads) {
            const long long row = s_row[st][i / chunks];
            if (row >= 0) cp_async16(dst + static_cast<size_t>(i) * 16, table + row * D + (i % chunks) * 8);
        }
        cp_async_commit();
        cp_async_wait<kProbeStages - 1>();
    }
    cp_async_wait<0>();
    __syncthreads();
    // one word of what arrived, so that the copies have an observable effect
    if (threadIdx.x == 0) atomicAdd(sink, *reinterpret_cast<const unsigned int *>(smem));
}

}  // namespace

cudaError_t launch_gather_probe(const uint16_t *table, long long n_table, int D, const int32_t *idx, long long n_idx,
                                unsigned int *sink, const Ctx &c) {
    const size_t smem = kProbeStages * static_cast<size_t>(kProbeRows) * D * 2;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kProbeStages * kProbeRows * 256 * 2));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const long long n_tiles = (n_idx + kProbeRows - 1) / kProbeRows;
    const long long grid = n_tiles < 2LL * c.num_sms ? n_tiles : 2LL * c.num_sms;
    return launch(gather_probe_kernel, dim3(static_cast<unsigned>(grid > 0 ? grid : 1)), dim3(kProbeThreads), smem, c,
                  1, table, n_table, D, idx, n_idx, c.err, sink);
}

}  // namespace ds4a
