// ingest.cu -- the input kernel of ds4a_decode_layer_step: one decode step's inputs,
// read by the GPU from page-locked host memory (mapped into the device's address
// space) and written into the layer's device arrays, in one launch rather than one
// copy-engine transfer per array.  Eight CTAs share every segment's 16-byte chunks
// (2-byte elements where a segment is not 16-byte aligned), so the reads over the
// host link are all in flight together.
#include "ds4a_common.cuh"
#include "ds4a_internal.h"

namespace ds4a {
namespace {

constexpr int kIngestThreads = 256;
constexpr int kIngestCtas = 8;

__global__ void __launch_bounds__(kIngestThreads) ingest_kernel(IngestArgs a) {
    // The kernels ahead (the previous step's) have finished reading what this overwrites.
    // A kernel after this one launched with programmatic dependence may start now: it
    // reads none of these arrays before its own dependency wait.
    pdl_wait();
    pdl_trigger();
    const int tid = blockIdx.x * blockDim.x + threadIdx.x, nth = gridDim.x * blockDim.x;
    for (int s = 0; s < a.n; ++s) {
        const IngestSeg g = a.seg[s];
        const uintptr_t bits = reinterpret_cast<uintptr_t>(g.src) | reinterpret_cast<uintptr_t>(g.dst) | g.bytes;
        if ((bits & 15) == 0) {
            const uint4 *src = static_cast<const uint4 *>(g.src);
            uint4 *dst = static_cast<uint4 *>(g.dst);
            for (unsigned i = tid; i < g.bytes / 16; i += nth) dst[i] = src[i];
        } else {
            const uint16_t *src = static_cast<const uint16_t *>(g.src);
            uint16_t *dst = static_cast<uint16_t *>(g.dst);
            for (unsigned i = tid; i < g.bytes / 2; i += nth) dst[i] = src[i];
        }
    }
}

}  // namespace

cudaError_t launch_ingest(const IngestArgs &a, const Ctx &c) {
    return launch(ingest_kernel, dim3(kIngestCtas), dim3(kIngestThreads), 0, c, 1, a);
}

}  // namespace ds4a
