// pa_decode_static_workspace: paged decode for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they run decode: an
// engine that reserved (nearly) all free device memory for its KV pool at
// start-up has no headroom left for a per-call workspace, and a plugin whose
// host framework owns every device allocation has no allocator of its own.
// For them this entry point uses scratch memory that is part of the loaded
// library: a file-scope __device__ array, resident on every GPU the library
// is loaded on until the process exits.  It allocates nothing itself.
//
// The kernels are the ones pa_decode launches; this file only supplies their
// workspace.  Host code cannot use the array's name as a device address, so
// the address is looked up with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and cached.
#include <stdio.h>

#include <mutex>

#include "pa_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

// The split-K partials of one call.  Every call uses the same array.
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set-up on first use).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

namespace pa {
int set_last_error(int code, const char *msg);
}

extern "C" PA_API int pa_decode_static_workspace(
    const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, void *out,
    pa_dtype dtype, int32_t *err_flag, void *stream) {
    // Size check first, on the host: nothing is touched when the shape does not fit.
    const size_t need = pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                  block_size);
    if (need > kStaticScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "pa_decode_static_workspace: this shape needs %zu bytes of scratch but the static scratch holds "
                 "%zu; use pa_decode with a caller workspace",
                 need, kStaticScratchBytes);
        return pa::set_last_error(PA_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "pa_decode_static_workspace: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        return pa::set_last_error(PA_ERR_CUDA, msg);
    }
    return pa_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                     num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out, scratch,
                     kStaticScratchBytes, dtype, err_flag, stream);
}
