// pa_copy_segments: several copies in one kernel, the segment list read when the kernel runs.
//
// A decode step's inputs (q and the new K/V rows, "Inference engine: inside
// nano-vLLM", section "Attention in nano-vLLM") are produced on the host in
// the engine this library serves.  A captured CUDA graph has fixed operand
// addresses, so a step either copies its inputs into the graph's staging on
// the host first or reads them where they are.  This kernel does the second:
// it reads a small list of (source, destination, bytes) from page-locked host
// memory (or device memory) at run time, so a graph that begins with it can
// be pointed at a new step's buffers by rewriting the list, and all SMs pull
// the bytes over the CPU-GPU link at once (no host-side copy, no copy-engine
// transfer per buffer).

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_segments_kernel(const pa_copy_segment *segments, int32_t count) {
    // the next kernel of the step may be launched now; it waits for this grid before its reads
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kCopyThreads;
    for (int s = 0; s < count; ++s) {
        const pa_copy_segment seg = segments[s];
        const uint8_t *src = static_cast<const uint8_t *>(seg.src);
        uint8_t *dst = static_cast<uint8_t *>(seg.dst);
        const int64_t bytes = static_cast<int64_t>(seg.bytes);
        int64_t done = 0;
        if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
            const int64_t vecs = bytes >> 4;
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
            // four loads in flight per thread before the stores
            int64_t i = tid;
            for (; i + 3 * nthreads < vecs; i += 4 * nthreads) {
                const uint4 a = s4[i], b = s4[i + nthreads], c = s4[i + 2 * nthreads], d = s4[i + 3 * nthreads];
                d4[i] = a;
                d4[i + nthreads] = b;
                d4[i + 2 * nthreads] = c;
                d4[i + 3 * nthreads] = d;
            }
            for (; i < vecs; i += nthreads) d4[i] = s4[i];
            done = vecs << 4;
        }
        for (int64_t i = done + tid; i < bytes; i += nthreads) dst[i] = src[i];
    }
}

}  // namespace

cudaError_t launch_copy_segments(const pa_copy_segment *segments, int32_t count, int32_t ctas, cudaStream_t stream) {
    if (count == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, copy_segments_kernel, segments, count);
}

}  // namespace pa
