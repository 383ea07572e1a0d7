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
// the address is looked up with cudaGetSymbolAddress, with the device current,
// and cached per device together with the unique id of the context it belongs
// to: after a device reset the next call sees a new context and looks the
// address up again.
//
// Under CUDA's default lazy module loading, the array is placed in device
// memory only when its module is first used, i.e. at the first call on a
// device.  A call with batch == 0 is the set-up call: it places the array and
// loads every kernel this entry point can launch, and computes nothing, so a
// caller can take the 8 MiB (and the kernels' code) before it gives the rest
// of the device memory to its KV pool.
#include <cuda.h>
#include <stdio.h>

#include <mutex>

#include "pa_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

// The split-K partials of one call.  Every call uses the same array.
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long *);

struct Slot {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void *ptr;
};

std::mutex g_mu;
Slot g_slot[kMaxDevices] = {};

template <typename F> F driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

// Unique id of the current context (ids are never reused within a process), or 0.
unsigned long long current_context_id() {
    static const CtxGetCurrent get_current = driver_fn<CtxGetCurrent>("cuCtxGetCurrent");
    static const CtxGetId get_id = driver_fn<CtxGetId>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_decode_scratch on the current device (looked up once per context).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // 0 before the device's primary context exists; then the lookup below creates it
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    if (!id || g_slot[dev].ctx_id != id || !g_slot[dev].ptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_slot[dev] = Slot{current_context_id(), p};
    }
    *out = g_slot[dev].ptr;
    return cudaSuccess;
}

}  // namespace

namespace pa {
int set_last_error(int code, const char *msg);
cudaError_t preload_decode_kernels();
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
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess && batch == 0) e = pa::preload_decode_kernels();  // the set-up call
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "pa_decode_static_workspace: set-up of the static scratch failed: %s",
                 cudaGetErrorString(e));
        return pa::set_last_error(PA_ERR_CUDA, msg);
    }
    return pa_decode(q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                     num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, out, scratch,
                     kStaticScratchBytes, dtype, err_flag, stream);
}
