// Slot-mapped store of this step's K/V rows into the paged pool.
//
// Follows store_kvcache of "Inference engine: inside nano-vLLM" (section
// "Attention in nano-vLLM"): token t's K row and V row (num_kv_heads*head_dim
// contiguous elements each) are copied to cache row slot_mapping[t]; slot -1
// is skipped.  The reference launches one program per token; here one warp
// moves one token's K and V rows with 16-byte vector accesses (when the
// pointers and strides allow), every lane holding all its loads in flight
// before it stores, so each SM keeps tens of KB of reads outstanding.

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kUnroll = 4;  // vectors per lane in flight per row

template <typename V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
store_kv_kernel(const V *__restrict__ k, const V *__restrict__ v, int64_t k_stride_v, int64_t v_stride_v,
                V *__restrict__ k_cache, V *__restrict__ v_cache, const int32_t *__restrict__ slot_mapping,
                int32_t num_tokens, int32_t row_v, int64_t num_slots, int32_t *err_flag) {
    // the attention kernel of the same step may be launched now (it waits for this grid)
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int32_t t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= num_tokens) return;
    const V *ks = k + t * k_stride_v;
    const V *vs = v + t * v_stride_v;
    for (int base = 0; base < row_v; base += 32 * kUnroll) {
        // the row loads do not depend on the slot: issue them with the slot load, so a warp
        // waits for one memory round trip before its stores instead of two
        V kr[kUnroll], vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_v) {
                kr[u] = __ldg(ks + i);
                vr[u] = __ldg(vs + i);
            }
        }
        const int64_t slot = slot_mapping[t];
        if (slot == -1) return;
        if (slot < -1 || slot >= num_slots) {
            if (lane == 0 && base == 0) raise_flag(err_flag, PA_FLAG_BAD_SLOT);
            return;
        }
        V *kd = k_cache + slot * row_v;
        V *vd = v_cache + slot * row_v;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_v) {
                kd[i] = kr[u];
                vd[i] = vr[u];
            }
        }
    }
}

template <typename V>
cudaError_t launch_vec(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride, void *k_cache,
                       void *v_cache, const int32_t *slot_mapping, int32_t num_tokens, int32_t row_elems,
                       int64_t num_slots, int32_t *err_flag, cudaStream_t stream) {
    constexpr int per = sizeof(V) / 2;  // 16-bit elements per vector
    const dim3 grid((num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock);
    store_kv_kernel<V><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        static_cast<const V *>(k), static_cast<const V *>(v), k_row_stride / per, v_row_stride / per,
        static_cast<V *>(k_cache), static_cast<V *>(v_cache), slot_mapping, num_tokens, row_elems / per,
        num_slots, err_flag);
    return cudaGetLastError();
}

bool aligned(const void *p, int64_t bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

// The same store into an E4M3 pool with per-tensor scales: each element
// becomes the nearest E4M3 value of x / scale (fp32 division; ties to even;
// saturating at +-448).  A lane converts 8 elements: one 16-byte load, one
// 8-byte store.
template <typename T>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
store_kv_fp8_kernel(const T *__restrict__ k, const T *__restrict__ v, int64_t k_stride, int64_t v_stride,
                    uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                    const int32_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t row, int64_t num_slots,
                    float k_scale, float v_scale, int32_t *err_flag) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int32_t t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= num_tokens) return;
    for (int i = 8 * lane; i < row; i += 32 * 8) {
        // the row loads are issued with the slot load (they do not depend on it)
        const uint4 kr = *reinterpret_cast<const uint4 *>(k + t * k_stride + i);
        const uint4 vr = *reinterpret_cast<const uint4 *>(v + t * v_stride + i);
        const int64_t slot = slot_mapping[t];
        if (slot == -1) return;
        if (slot < -1 || slot >= num_slots) {
            if (lane == 0 && i == 0) raise_flag(err_flag, PA_FLAG_BAD_SLOT);
            return;
        }
        *reinterpret_cast<uint2 *>(k_cache + slot * row + i) = quantize8_e4m3<T>(kr, k_scale);
        *reinterpret_cast<uint2 *>(v_cache + slot * row + i) = quantize8_e4m3<T>(vr, v_scale);
    }
}

}  // namespace

cudaError_t launch_store_kv_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                                void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                                int32_t row_elems, int64_t num_slots, pa_dtype dtype, float k_scale, float v_scale,
                                int32_t *err_flag, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const dim3 grid((num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock);
    if (dtype == PA_BF16)
        store_kv_fp8_kernel<__nv_bfloat16><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), k_row_stride, v_row_stride,
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), slot_mapping, num_tokens, row_elems,
            num_slots, k_scale, v_scale, err_flag);
    else
        store_kv_fp8_kernel<__half><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
            static_cast<const __half *>(k), static_cast<const __half *>(v), k_row_stride, v_row_stride,
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), slot_mapping, num_tokens, row_elems,
            num_slots, k_scale, v_scale, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_store_kv(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                            void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                            int32_t row_elems, int64_t num_slots, int32_t *err_flag, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    // widest access every row start allows
    for (int bytes = 16; bytes >= 2; bytes /= 2) {
        const int per = bytes / 2;
        const bool ok = aligned(k, bytes) && aligned(v, bytes) && aligned(k_cache, bytes) &&
                        aligned(v_cache, bytes) && k_row_stride % per == 0 && v_row_stride % per == 0 &&
                        row_elems % per == 0;
        if (!ok) continue;
        switch (bytes) {
            case 16: return launch_vec<uint4>(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping,
                                              num_tokens, row_elems, num_slots, err_flag, stream);
            case 8: return launch_vec<uint2>(k, v, k_row_stride, v_row_stride, k_cache, v_cache, slot_mapping,
                                             num_tokens, row_elems, num_slots, err_flag, stream);
            case 4: return launch_vec<uint32_t>(k, v, k_row_stride, v_row_stride, k_cache, v_cache,
                                                slot_mapping, num_tokens, row_elems, num_slots, err_flag, stream);
            default: return launch_vec<uint16_t>(k, v, k_row_stride, v_row_stride, k_cache, v_cache,
                                                 slot_mapping, num_tokens, row_elems, num_slots, err_flag, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
