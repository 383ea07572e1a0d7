// Shared device helpers for the paged-KV kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_api.h"

namespace pa {

// ---------------------------------------------------------------- dtypes

template <typename T> struct Dt;
template <> struct Dt<__half> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ __half from_float(float a) { return __float2half_rn(a); }
};
template <> struct Dt<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ __nv_bfloat16 from_float(float a) { return __float2bfloat16_rn(a); }
};

// Eight 16-bit elements (one 16-byte vector) as eight E4M3 codes, element i in
// byte i: the nearest E4M3 value of x / scale (IEEE fp32 division, ties to
// even, saturating at +-448, NaN stays NaN).
template <typename T> __device__ __forceinline__ uint2 quantize8_e4m3(const uint4 raw, float scale) {
    const T *x = reinterpret_cast<const T *>(&raw);
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t bytes = 0;
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const float2 f = make_float2(static_cast<float>(x[4 * h + e]) / scale,
                                         static_cast<float>(x[4 * h + e + 1]) / scale);
            const __nv_fp8x2_storage_t pair = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
            bytes |= static_cast<uint32_t>(pair) << (8 * e);
        }
        w[h] = bytes;
    }
    return make_uint2(w[0], w[1]);
}

// ------------------------------------------------------------ error flag

__device__ __forceinline__ void raise_flag(int32_t *err_flag, int bits) {
    if (err_flag) atomicOr(err_flag, bits);
}

// ---------------------------------------------------------------- memory

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async global->shared copy; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------- warp-level matrices

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}

// D(16x8, f32) += A(16x16) * B(16x8), A row-major fragment, B column fragment.
template <typename T> struct Mma;
template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                     "{%8,%9}, {%0,%1,%2,%3};\n"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
};
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                     "{%8,%9}, {%0,%1,%2,%3};\n"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ float warp_max_xor(float v, int lane_mask) {
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, lane_mask));
}

}  // namespace pa

// Host-side launchers (defined in the .cu files, called by pa_api.cu).
namespace pa {
cudaError_t launch_store_kv(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                            void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                            int32_t row_elems, int64_t num_slots, int32_t *err_flag, cudaStream_t stream);

cudaError_t launch_store_kv_fp8(const void *k, const void *v, int64_t k_row_stride, int64_t v_row_stride,
                                void *k_cache, void *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                                int32_t row_elems, int64_t num_slots, pa_dtype dtype, float k_scale, float v_scale,
                                int32_t *err_flag, cudaStream_t stream);

struct DecodePlan {
    int stages;         // ring depth of the partition kernel (2 or 3)
    int partition;      // tokens per split-K partition (multiple of the tile)
    int max_parts;      // partitions per sequence at the maximum context
    // shared prefixes (pa_decode_options groups; all 0 without)
    int pre_partition;  // tokens per prefix partition
    int pre_parts;      // prefix partitions at the longest shared prefix
    int seqs_per_cta;   // member sequences one prefix CTA serves
    int group_ctas;     // prefix CTAs per group and (kv head, prefix partition)
    int64_t prefix_ctas;  // num_groups * group_ctas
    int slots;          // workspace partials per (sequence, q head): pre_parts + max_parts
    size_t ws_bytes;    // workspace bytes
};
// The E4M3 pool of the fp8 calls: K = code * k_scale, V = code * v_scale.
struct Fp8Scales {
    float k_scale, v_scale;
};
// fp8: the plan of the E4M3 partition kernel (its own ring and occupancy).
// opt (nullable): the caller's overrides of the partition size and the ring depth.
DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t max_blocks_per_seq, int32_t block_size, bool fp8 = false,
                       const pa_decode_options *opt = nullptr);
// The store fused into pa_store_decode (the new rows of one decode step).
struct FusedStore {
    const void *k;
    const void *v;
    int64_t k_row_stride;  // elements between sequences' rows
    int64_t v_row_stride;
    const int32_t *slot_mapping;
};
cudaError_t launch_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t num_blocks, int32_t block_size, float scale, void *out, void *workspace,
                          const DecodePlan &plan, pa_dtype dtype, int32_t *err_flag, cudaStream_t stream,
                          const FusedStore *fused = nullptr, const Fp8Scales *fp8 = nullptr,
                          const pa_decode_options *opt = nullptr);
cudaError_t launch_sample(const void *logits, int64_t row_stride, int32_t batch, int32_t vocab, pa_dtype dtype,
                          const float *temperatures, const float *noise, uint64_t seed, uint64_t offset,
                          int32_t *tokens, int32_t *err_flag, cudaStream_t stream);
cudaError_t launch_prefill(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs,
                           int32_t total_q, int32_t max_seqlen_q, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_blocks, int32_t block_size, float scale, void *out, pa_dtype dtype,
                           int32_t *err_flag, int32_t sms, cudaStream_t stream, const char **why);
cudaError_t launch_copy_segments(const pa_copy_segment *segments, int32_t count, int32_t ctas, cudaStream_t stream);
// The two streams of a pa_sm_split (sm_split.cu): fork makes both wait for `from`'s work so
// far, join makes `to` wait for everything issued on both.
cudaStream_t split_stream(const pa_sm_split *s, int i);
int split_sms(const pa_sm_split *s, int i);
int split_device(const pa_sm_split *s);
cudaError_t split_fork(const pa_sm_split *s, cudaStream_t from);
cudaError_t split_join(const pa_sm_split *s, cudaStream_t to);
}  // namespace pa
