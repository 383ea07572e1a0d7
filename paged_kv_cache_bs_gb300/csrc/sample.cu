// Temperature sampling by the exponential race ("From nano-vLLM to vLLM:
// Scheduler, Paged KV Cache, Prefill/Decode, Tensor Parallelism, and
// Sampling", section 17): for each row, a = logits / T, p = softmax(a),
// token = argmax_i p_i / max(E_i, 1e-10) with E_i ~ Exp(1).  The kernel takes
// the decision in the race's log form, argmax_i a_i - log(max(E_i, 1e-10))
// with a_i = logits_i * (1 / T),
// which section 17.5 of the same page shows to select the same token (the
// softmax denominator is common to all i), so one pass over the logits
// suffices and no softmax is formed.  Only near-ties can resolve differently
// from the fp32 ratio form.
//
// Each row is split over a cluster of 8 CTAs (256 threads each); every CTA
// finds the winner of its slice, and the cluster's first CTA compares the
// eight winners through distributed shared memory and writes the token -- no
// workspace and no second kernel.  The noise is read from the caller's
// buffer, or drawn in-kernel from Philox4x32-10, so that nothing but the
// logits has to come from memory.
#include <cooperative_groups.h>
#include <math.h>

#include "pa_common.cuh"

namespace cg = cooperative_groups;

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;  // CTAs per row
constexpr float kMinNoise = 1e-10f;

struct SampleArgs {
    const void *logits;
    int64_t row_stride;  // elements
    int32_t vocab;
    const float *temperatures;
    const float *noise;  // nullable
    uint32_t seed_lo, seed_hi, off_lo, off_hi;
    int32_t *tokens;
    int32_t *err_flag;
};

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds, each two 32x32 -> 64-bit products of
// counter words with the round multipliers, the high halves xored with the
// other counter words and the round key.  The round keys (the key advanced by
// the Weyl increments between rounds) depend only on the seed, so a thread
// derives them once.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
    __device__ __forceinline__ PhiloxKeys(uint32_t s0, uint32_t s1) {
#pragma unroll
        for (int r = 0; r < 10; ++r) {
            k0[r] = s0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
            k1[r] = s1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
        }
    }
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys &k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.k0[r], lo1, hi0 ^ c.w ^ k.k1[r], lo0);
    }
    return c;
}

// Hardware base-2 logarithm (MUFU): absolute error about 2^-22.
__device__ __forceinline__ float lg2_hw(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// An Exp(1) sample from 24 random bits, in units of 1/ln 2 (E' = E / ln 2, E = -ln u):
// u = ((x >> 8) + 1) 2^-24 in (0, 1], E' = -log2(u).  Near u = 1, where E is small
// and decides the race's winners, -ln(1 - v) = v + v^2/2 + v^3/3 + v^4/4 + v^5/5 +
// ... with v = 1 - u exact (relative error below 3e-7 for v < 1/16, rounding
// included); elsewhere E >= 0.0645 and the hardware logarithm is within 2e-6.  Both
// forms are computed and one is selected (no divergent branch).  The race only
// compares log E_i + const, so the common factor 1/ln 2 does not change the winner.
__device__ __forceinline__ float exp1_scaled(uint32_t x) {
    const float u = static_cast<float>((x >> 8) + 1u) * 0x1p-24f;
    const float v = 1.f - u;
    const float series = v * fmaf(v, fmaf(v, fmaf(v, fmaf(v, 0.2f, 0.25f), 0.33333334f), 0.5f), 1.f) *
                         1.4426950408889634f;
    const float hw = -lg2_hw(u);
    return v < 0.0625f ? series : hw;
}

// Eight consecutive logits (from a 16-byte aligned address): loaded raw, widened to floats.
template <typename T> struct Vec8;
template <> struct Vec8<float> {
    struct Raw {
        float4 a, b;
    };
    static __device__ __forceinline__ Raw load(const float *p) {
        return Raw{*reinterpret_cast<const float4 *>(p), *reinterpret_cast<const float4 *>(p + 4)};
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&v)[8]) {
        v[0] = r.a.x, v[1] = r.a.y, v[2] = r.a.z, v[3] = r.a.w, v[4] = r.b.x, v[5] = r.b.y, v[6] = r.b.z, v[7] = r.b.w;
    }
    static __device__ __forceinline__ float one(const float *p) { return *p; }
};
template <> struct Vec8<__nv_bfloat16> {
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint4 *>(p); }
    static __device__ __forceinline__ void unpack(const Raw &a, float (&v)[8]) {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ float one(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
};
template <> struct Vec8<__half> {
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const __half *p) { return *reinterpret_cast<const uint4 *>(p); }
    static __device__ __forceinline__ void unpack(const Raw &a, float (&v)[8]) {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[j] & 0xFFFFu)));
            v[2 * j + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[j] >> 16)));
        }
    }
    static __device__ __forceinline__ float one(const __half *p) { return __half2float(*p); }
};

// Larger score wins, then the smaller index.
__device__ __forceinline__ bool better(float s1, int i1, float s2, int i2) {
    return i1 >= 0 && (i2 < 0 || s1 > s2 || (s1 == s2 && i1 < i2));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
    __shared__ float red_v[kWarps];
    __shared__ int red_i[kWarps];
    __shared__ float win_v;
    __shared__ int win_i;
    cg::cluster_group cluster = cg::this_cluster();
    const int part = static_cast<int>(cluster.block_rank());
    asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the logits come from the previous kernel
    const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float temp = a.temperatures[b];
    const bool valid_t = temp > 1e-10f && isfinite(temp);  // the pages' sampler has no greedy path
    const T *row = static_cast<const T *>(a.logits) + b * a.row_stride;
    const int V = a.vocab;
    // this CTA's slice of the row, in 8-element groups when the row is 16-byte aligned
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int ngroups = vec ? V / 8 : 0;
    const int g_per = (ngroups + kCluster - 1) / kCluster;
    const int g0 = min(ngroups, part * g_per), g1 = min(ngroups, g0 + g_per);
    const int tail0 = 8 * ngroups, tail_per = (V - tail0 + kCluster - 1) / kCluster;
    const int t0 = min(V, tail0 + part * tail_per), t1 = min(V, t0 + tail_per);

    // Scores in base 2: a_i log2(e) - log2(max(E_i, 1e-10)), the race's ln form times log2(e) > 0
    // (same winner).  The in-kernel draws are E_i / ln 2, clamped at 1e-10 / ln 2: a common shift.
    float best = -INFINITY;  // -inf never wins: a row with no finite score keeps index -1
    int best_i = -1;
    const float inv_t2 = 1.4426950408889634f / temp;
    auto visit = [&](int i, float x, float e, float min_noise) {
        const float sc = x * inv_t2 - lg2_hw(fmaxf(e, min_noise));
        if (sc > best) {  // a thread visits its indices in increasing order: ties keep the first
            best = sc;
            best_i = i;
        }
    };
    constexpr float kMinScaledNoise = kMinNoise * 1.4426950408889634f;
    const float *noise = a.noise ? a.noise + static_cast<int64_t>(b) * V : nullptr;
    if (valid_t) {
        const PhiloxKeys keys(a.seed_lo, a.seed_hi);
        const float min_noise = noise ? kMinNoise : kMinScaledNoise;
        for (int g = g0 + tid; g < g1; g += kThreads) {
            float v[8], e[8];
            Vec8<T>::unpack(Vec8<T>::load(row + 8 * g), v);
            if (noise) {
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = noise[8 * g + j];
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 r = philox4x32_10(make_uint4(2 * g + h, b, a.off_lo, a.off_hi), keys);
                    e[4 * h] = exp1_scaled(r.x);
                    e[4 * h + 1] = exp1_scaled(r.y);
                    e[4 * h + 2] = exp1_scaled(r.z);
                    e[4 * h + 3] = exp1_scaled(r.w);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) visit(8 * g + j, v[j], e[j], min_noise);
        }
        for (int i = t0 + tid; i < t1; i += kThreads) {
            float e;
            if (noise) {
                e = noise[i];
            } else {
                const uint4 r = philox4x32_10(make_uint4(i >> 2, b, a.off_lo, a.off_hi), keys);
                const int q = i & 3;
                e = exp1_scaled(q == 0 ? r.x : q == 1 ? r.y : q == 2 ? r.z : r.w);
            }
            visit(i, Vec8<T>::one(row + i), e, min_noise);
        }
    }
    // CTA winner
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (better(v2, i2, best, best_i)) {
            best = v2;
            best_i = i2;
        }
    }
    if (lane == 0) {
        red_v[warp] = best;
        red_i[warp] = best_i;
    }
    __syncthreads();
    if (tid == 0) {
        float bv = red_v[0];
        int bi = red_i[0];
        for (int w = 1; w < kWarps; ++w)
            if (better(red_v[w], red_i[w], bv, bi)) {
                bv = red_v[w];
                bi = red_i[w];
            }
        win_v = bv;
        win_i = bi;
    }
    // row winner: the first CTA of the cluster reads the others' winners from their shared memory
    cluster.sync();
    if (part == 0 && tid == 0) {
        float bv = win_v;
        int bi = win_i;
        for (int r = 1; r < kCluster; ++r) {
            const float rv = *cluster.map_shared_rank(&win_v, r);
            const int ri = *cluster.map_shared_rank(&win_i, r);
            if (better(rv, ri, bv, bi)) {
                bv = rv;
                bi = ri;
            }
        }
        a.tokens[b] = valid_t ? bi : -1;  // -1 also when no logit is finite
        if (!valid_t) raise_flag(a.err_flag, PA_FLAG_BAD_VALUE);
    }
    cluster.sync();  // the others' shared memory stays until it has been read
}

}  // namespace

cudaError_t launch_sample(const void *logits, int64_t row_stride, int32_t batch, int32_t vocab, pa_dtype dtype,
                          const float *temperatures, const float *noise, uint64_t seed, uint64_t offset,
                          int32_t *tokens, int32_t *err_flag, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    SampleArgs a;
    a.logits = logits;
    a.row_stride = row_stride;
    a.vocab = vocab;
    a.temperatures = temperatures;
    a.noise = noise;
    a.seed_lo = static_cast<uint32_t>(seed);
    a.seed_hi = static_cast<uint32_t>(seed >> 32);
    a.off_lo = static_cast<uint32_t>(offset);
    a.off_hi = static_cast<uint32_t>(offset >> 32);
    a.tokens = tokens;
    a.err_flag = err_flag;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCluster, batch);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    switch (dtype) {
        case PA_F32: return cudaLaunchKernelEx(&cfg, sample_kernel<float>, a);
        case PA_BF16: return cudaLaunchKernelEx(&cfg, sample_kernel<__nv_bfloat16>, a);
        default: return cudaLaunchKernelEx(&cfg, sample_kernel<__half>, a);
    }
}

}  // namespace pa
