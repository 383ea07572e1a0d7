// Paged GQA decode attention, split over context partitions.
//
// What is computed is the decode branch of the attention layer in
// "Inference engine: inside nano-vLLM" (flash_attn_with_kvcache with
// cache_seqlens and block_table): each sequence's single query attends over
// its context, position j read from cache row
// block_table[j / bs] * bs + j % bs ("nano-vLLM Part 2", section 2.2).
//
// Design (GB300): decode is HBM-bound, so everything serves the K/V stream.
//   * One CTA per (partition, kv head, sequence).  The G query heads of the
//     group share every K/V tile, so each cache byte is read once.
//   * Pages are gathered through the block table into a 3-stage shared-memory
//     ring with 16-byte cp.async (rows of one kv head are D*2 bytes, strided
//     by H_kv*D*2 in the pool), XOR-swizzled so the warp-matrix loads below
//     are bank-conflict free.
//   * Each warp owns 16 tokens of a 64-token tile.  S^T = K Q^T and
//     O^T += V^T P^T are m16n8k16 warp MMAs with the G (<= 8) heads in the
//     N dimension: the contraction is tiny, the point is only to keep the
//     per-byte instruction count far below the issue budget an HBM-rate
//     stream leaves (about 90 warp instructions per 512 bytes per SM).
//   * Softmax is online, in fp32, in the log2 domain; row maxima are reduced
//     with warp shuffles.  P is rounded to the input dtype for the PV MMA
//     while the normaliser sums the fp32 values.
//   * Warps merge through shared memory at the end of the partition; a
//     sequence with one partition writes its output directly, otherwise the
//     (max, sum, unnormalised O) partials go to the workspace and a second
//     kernel merges them by log-sum-exp; it is launched as a programmatic
//     dependent of the first, so its launch overlaps the partition kernel.
#include <math.h>
#include <stdlib.h>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 64;      // tokens per pipeline stage, 16 per warp
constexpr int kStages = 3;
constexpr int kMaxTablePages = 257;  // block-table entries one partition may touch
constexpr int kMaxPartition = 2048;
constexpr int kMinPartition = 128;
constexpr int kTargetCtas = 16 * 152;  // ragged batches: enough waves to absorb the length spread
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const void *q;
    int64_t q_row_stride;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    int32_t max_blocks;
    const int32_t *context_lens;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t num_blocks;
    int32_t log2_bs;
    float scale_log2;
    void *out;
    float *ws_o;     // [B][H_q][max_parts][D]  unnormalised partial outputs
    float2 *ws_ml;   // [B][H_q][max_parts]     (running max, running sum), log2 domain
    int32_t partition;
    int32_t max_parts;
    int32_t *err_flag;
};

template <int D> struct Shape {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kChunks = D / 8;  // 16-byte chunks per row
    static constexpr int kTileBytes = kTile * kRowBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
    static constexpr int kKSteps = D / 16;
    static constexpr int kRowsPerPass = kThreads / kChunks;
    static constexpr int kPasses = kTile / kRowsPerPass;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kMergeBytes = kWarps * 8 * (D + 2) * 4;
    static constexpr int kSmemBytes =
        (kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes) + kMaxTablePages * 4;
};

// Context length of sequence b, or 0 (flagged) when it is out of range.
__device__ __forceinline__ int context_len(const DecodeArgs &a, int b) {
    const int L = a.context_lens[b];
    const int64_t cap = static_cast<int64_t>(a.max_blocks) << a.log2_bs;
    return (L < 0 || L > cap) ? -1 : L;
}

__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
    return row * row_bytes + ((chunk ^ (row & 7)) << 4);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) decode_partition_kernel(const DecodeArgs a) {
    using S = Shape<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + (S::kRingBytes > S::kMergeBytes ? S::kRingBytes
                                                                                         : S::kMergeBytes));

    const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Launched as a programmatic dependent of the previous kernel on the stream (the store
    // of this step): wait for it to finish before reading the cache, and let the merge
    // kernel be launched right away (it waits for this grid itself).
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    int L = context_len(a, b);
    if (L < 0) {
        if (p == 0 && tid == 0) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
        L = 0;
    }
    const int start = p * a.partition;
    T *out = static_cast<T *>(a.out);
    if (start >= L) {
        if (p == 0)  // empty context (e.g. a padding row): zero output, no page read
            for (int i = tid; i < a.group * D; i += kThreads)
                out[(static_cast<int64_t>(b) * a.num_q_heads + g * a.group + i / D) * D + i % D] =
                    Dt<T>::from_float(0.f);
        return;
    }
    const int end = min(L, start + a.partition);
    const int nparts = (L + a.partition - 1) / a.partition;
    const int ntiles = (end - start + kTile - 1) / kTile;
    const int bs_mask = (1 << a.log2_bs) - 1;

    // block-table slice of this partition, validated once
    const int first_page = start >> a.log2_bs;
    const int npages = ((end - 1) >> a.log2_bs) - first_page + 1;
    for (int i = tid; i < npages; i += kThreads) {
        int pg = a.block_tables[static_cast<int64_t>(b) * a.max_blocks + first_page + i];
        if (pg < 0 || pg >= a.num_blocks) {
            raise_flag(a.err_flag, PA_FLAG_BAD_BLOCK);
            pg = -1;  // read as zeros
        }
        bt_s[i] = pg;
    }

    // query fragments (B operand of S^T = K Q^T): head lane/4 of the group
    uint32_t qb[S::kKSteps][2];
    {
        const int hq = lane >> 2;
        const int dq = (lane & 3) * 2;
        const T *qrow = static_cast<const T *>(a.q) + static_cast<int64_t>(b) * a.q_row_stride +
                        static_cast<int64_t>(g * a.group + hq) * D;
#pragma unroll
        for (int ks = 0; ks < S::kKSteps; ++ks) {
            if (hq < a.group) {
                qb[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + dq);
                qb[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + dq);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
    }
    __syncthreads();  // bt_s ready

    const T *kc = static_cast<const T *>(a.k_cache);
    const T *vc = static_cast<const T *>(a.v_cache);
    const int chunk = tid % S::kChunks;
    const int row0 = tid / S::kChunks;
    const int64_t head_off = static_cast<int64_t>(g) * D + chunk * 8;
    const int64_t row_elems = static_cast<int64_t>(a.num_kv_heads) * D;

    auto load_tile = [&](int t, int stage) {
        const uint32_t kb = smem_u32(smem + stage * S::kStageBytes);
        const uint32_t vb = kb + S::kTileBytes;
        const int tile_start = start + t * kTile;
#pragma unroll
        for (int i = 0; i < S::kPasses; ++i) {
            const int r = row0 + i * S::kRowsPerPass;
            const int j = tile_start + r;
            const uint32_t so = swz(r, chunk, S::kRowBytes);
            const T *ks = kc, *vs = vc;
            uint32_t nbytes = 0;
            if (j < end) {
                const int pg = bt_s[(j >> a.log2_bs) - first_page];
                if (pg >= 0) {
                    const int64_t off = ((static_cast<int64_t>(pg) << a.log2_bs) + (j & bs_mask)) * row_elems +
                                        head_off;
                    ks = kc + off;
                    vs = vc + off;
                    nbytes = 16;
                }
            }
            cp_async_16(kb + so, ks, nbytes);
            cp_async_16(vb + so, vs, nbytes);
        }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < ntiles) load_tile(s, s);
        cp_async_commit();
    }

    float o[S::kKSteps][4];
#pragma unroll
    for (int mt = 0; mt < S::kKSteps; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*(lane%4) and +1
    const int wrow = warp * 16;

    for (int t = 0; t < ntiles; ++t) {
        cp_async_wait<kStages - 2>();
        __syncthreads();  // tile t visible to all; stage of tile t-1 free for reuse
        {
            const int nt = t + kStages - 1;
            if (nt < ntiles) load_tile(nt, nt % kStages);
            cp_async_commit();
        }
        const uint32_t kb = smem_u32(smem + (t % kStages) * S::kStageBytes);
        const uint32_t vb = kb + S::kTileBytes;

        // S^T (16 tokens x 8 heads) = K (16 x D) . Q^T (D x 8)
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int r = wrow + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int csel = lane >> 4;
#pragma unroll
            for (int ks = 0; ks < S::kKSteps; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(kb + swz(r, ks * 2 + csel, S::kRowBytes), a0, a1, a2, a3);
                Mma<T>::run(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
        }
        // lane holds tokens j0 (sc[0], sc[1]) and j0 + 8 (sc[2], sc[3]) for heads 2*(lane%4), +1
        const int j0 = start + t * kTile + wrow + (lane >> 2);
        const bool v0 = j0 < end, v1 = j0 + 8 < end;
        const float s0 = v0 ? sc[0] * a.scale_log2 : -INFINITY;
        const float s1 = v0 ? sc[1] * a.scale_log2 : -INFINITY;
        const float s2 = v1 ? sc[2] * a.scale_log2 : -INFINITY;
        const float s3 = v1 ? sc[3] * a.scale_log2 : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
        mx0 = warp_max_xor(mx0, 4);
        mx1 = warp_max_xor(mx1, 4);
        mx0 = warp_max_xor(mx0, 8);
        mx1 = warp_max_xor(mx1, 8);
        mx0 = warp_max_xor(mx0, 16);
        mx1 = warp_max_xor(mx1, 16);
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;  // all masked so far: keep exp2 finite
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float c0 = exp2f(m0 - mu0), c1 = exp2f(m1 - mu1);
        const float p0 = exp2f(s0 - mu0), p1 = exp2f(s1 - mu1);
        const float p2 = exp2f(s2 - mu0), p3 = exp2f(s3 - mu1);
        l0 = l0 * c0 + (p0 + p2);
        l1 = l1 * c1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int mt = 0; mt < S::kKSteps; ++mt) {
            o[mt][0] *= c0;
            o[mt][1] *= c1;
            o[mt][2] *= c0;
            o[mt][3] *= c1;
        }
        // P^T as the B operand (16 tokens x 8 heads): transpose the two 8x8 halves
        const uint32_t pb0 = movmatrix_trans(Dt<T>::pack(p0, p1));
        const uint32_t pb1 = movmatrix_trans(Dt<T>::pack(p2, p3));
        // O^T (D x 8) += V^T (D x 16 tokens) . P^T (16 x 8)
        {
            const int i = lane >> 3;
            const int r = wrow + (lane & 7) + (i >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < S::kKSteps; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(vb + swz(r, mt * 2 + (i & 1), S::kRowBytes), a0, a1, a2, a3);
                Mma<T>::run(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // ring no longer needed: reuse it to merge the warps

    l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);

    float *mo = reinterpret_cast<float *>(smem);               // [warp][head 8][D]
    float *mm = mo + kWarps * 8 * D;                           // [warp][head 8]
    float *ml = mm + kWarps * 8;                               // [warp][head 8]
    {
        const int h0 = (lane & 3) * 2;
        const int dr = lane >> 2;
        float *w = mo + warp * 8 * D;
#pragma unroll
        for (int mt = 0; mt < S::kKSteps; ++mt) {
            w[h0 * D + mt * 16 + dr] = o[mt][0];
            w[(h0 + 1) * D + mt * 16 + dr] = o[mt][1];
            w[h0 * D + mt * 16 + dr + 8] = o[mt][2];
            w[(h0 + 1) * D + mt * 16 + dr + 8] = o[mt][3];
        }
        if (lane < 4) {
            mm[warp * 8 + h0] = m0;
            mm[warp * 8 + h0 + 1] = m1;
            ml[warp * 8 + h0] = l0;
            ml[warp * 8 + h0 + 1] = l1;
        }
    }
    __syncthreads();

    for (int i = tid; i < a.group * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * 8 + h]);
        float acc = 0.f, sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = exp2f(mm[w * 8 + h] - M);  // a warp with no token has max -inf: weight 0
            acc += mo[(w * 8 + h) * D + d] * wt;
            sum += ml[w * 8 + h] * wt;
        }
        const int hq = g * a.group + h;
        if (nparts == 1) {
            out[(static_cast<int64_t>(b) * a.num_q_heads + hq) * D + d] = Dt<T>::from_float(acc / sum);
        } else {
            const int64_t idx = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.max_parts + p;
            a.ws_o[idx * D + d] = acc;
            if (d == 0) a.ws_ml[idx] = make_float2(M, sum);
        }
    }
}

// Log-sum-exp merge of the partitions of sequences that have more than one.
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a) {
    const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    // launched early (programmatic dependent launch): wait until the partition grid has
    // finished and its partials are visible
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int L = max(context_len(a, b), 0);
    const int np = (L + a.partition - 1) / a.partition;
    if (np <= 1) return;
    const int64_t base = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.max_parts;
    float M = -INFINITY;
    for (int p = 0; p < np; ++p) M = fmaxf(M, a.ws_ml[base + p].x);
    float acc = 0.f, sum = 0.f;
    for (int p = 0; p < np; ++p) {
        const float2 ml = a.ws_ml[base + p];
        const float wt = exp2f(ml.x - M);
        sum += ml.y * wt;
        acc += a.ws_o[(base + p) * D + d] * wt;
    }
    static_cast<T *>(a.out)[(static_cast<int64_t>(b) * a.num_q_heads + hq) * D + d] =
        Dt<T>::from_float(acc / sum);
}

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

}  // namespace

// Resident decode CTAs the current device holds at once (2 per SM).
static int resident_ctas() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2 * 148;
    if (!cached[dev]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
        cached[dev] = 2 * sms;
    }
    return cached[dev];
}

DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t max_blocks_per_seq, int32_t block_size) {
    DecodePlan pl{};
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int64_t pairs = static_cast<int64_t>(batch) * num_kv_heads;
    const int64_t slots = resident_ctas();
    const int64_t tiles = (cap + kTile - 1) / kTile;
    int64_t part;
    if (pairs >= 2 * slots) {
        part = tiles * kTile;  // (sequence, kv head) pairs alone fill two waves: no split
    } else if (2 * pairs <= slots) {
        // few (sequence, kv head) pairs: one wave of equal partitions, each CTA streaming as
        // long as possible (the per-CTA start-up cost is paid once per SM slot)
        const int64_t per = slots / pairs > 1 ? slots / pairs : 1;
        part = ((tiles + per - 1) / per) * kTile;
    } else {
        // ragged batches: enough smaller partitions for the scheduler to even out lengths
        part = kMaxPartition;
        while (part > kMinPartition && pairs * ((cap + part - 1) / part) < kTargetCtas) part /= 2;
    }
    if (const char *env = getenv("PA_DECODE_PARTITION")) {  // tuning override
        const int v = atoi(env);
        if (v >= kTile && v % kTile == 0 && v <= (1 << 20)) part = v;
    }
    while (part / block_size > kMaxTablePages - 1) part = (part / 2 + kTile - 1) / kTile * kTile;  // table slice fits
    if (part < kTile) part = kTile;
    pl.partition = static_cast<int>(part);
    pl.max_parts = static_cast<int>(cap > 0 ? (cap + part - 1) / part : 1);
    const size_t n = static_cast<size_t>(batch) * num_q_heads * pl.max_parts;
    const size_t ml_bytes = (n * sizeof(float2) + 255) / 256 * 256;
    pl.ws_bytes = ml_bytes + n * head_dim * sizeof(float);
    return pl;
}

cudaError_t launch_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t num_blocks, int32_t block_size, float scale, void *out, void *workspace,
                          const DecodePlan &plan, pa_dtype dtype, int32_t *err_flag, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    DecodeArgs a;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_q_heads / num_kv_heads;
    a.num_blocks = num_blocks;
    a.log2_bs = ilog2(block_size);
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    const size_t n = static_cast<size_t>(batch) * num_q_heads * plan.max_parts;
    const size_t ml_bytes = (n * sizeof(float2) + 255) / 256 * 256;
    a.ws_ml = static_cast<float2 *>(workspace);
    a.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ml_bytes);
    a.partition = plan.partition;
    a.max_parts = plan.max_parts;
    a.err_flag = err_flag;

    using S128 = Shape<128>;
    using S64 = Shape<64>;
    cudaError_t e;
    auto run = [&](auto kern_part, auto kern_comb, int smem, int d) -> cudaError_t {
        // opt in to more than 48 KB of dynamic shared memory (a per-device function attribute)
        cudaError_t err = cudaFuncSetAttribute(kern_part, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        kern_part<<<dim3(a.max_parts, a.num_kv_heads, batch), kThreads, smem, stream>>>(a);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        if (a.max_parts > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(a.num_q_heads, batch);
            cfg.blockDim = dim3(d);
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&cfg, kern_comb, a);
        }
        return err;
    };
    if (dtype == PA_BF16) {
        e = head_dim == 128 ? run(decode_partition_kernel<__nv_bfloat16, 128>, decode_combine_kernel<__nv_bfloat16, 128>,
                                  S128::kSmemBytes, 128)
                            : run(decode_partition_kernel<__nv_bfloat16, 64>, decode_combine_kernel<__nv_bfloat16, 64>,
                                  S64::kSmemBytes, 64);
    } else {
        e = head_dim == 128 ? run(decode_partition_kernel<__half, 128>, decode_combine_kernel<__half, 128>,
                                  S128::kSmemBytes, 128)
                            : run(decode_partition_kernel<__half, 64>, decode_combine_kernel<__half, 64>,
                                  S64::kSmemBytes, 64);
    }
    return e;
}

}  // namespace pa
