// Chunked prefill over a paged prefix on the 5th-generation tensor cores.
//
// What is computed is the prefill branch of the attention layer in
// "Inference engine: inside nano-vLLM" (flash_attn_varlen_func with
// cu_seqlens_q / cu_seqlens_k and a block table): sequence i owns
// Lq = cu_q[i+1]-cu_q[i] query rows and a context of Lk = cu_k[i+1]-cu_k[i]
// tokens, the first P = Lk - Lq of them a cached prefix; query r attends over
// context positions 0..P+r ("nano-vLLM Part 2", sections 2.5 and 4.1).  With
// a block table every context position is read from the pool (prefix and the
// rows pa_store_kv wrote this step, as the pages' layer does with
// k, v = k_cache, v_cache); without one, keys are the packed k/v rows.
//
// One CTA = 128 query rows of one query head (TMEM lane r = query row r).
//   * Q (once) and each 128-key K/V tile arrive by TMA with the 128-byte
//     swizzle the MMA descriptors expect; K/V tiles are double-buffered and
//     fetched page by page through the block table (one box per page when a
//     page is shorter than the tile).
//   * S = Q K^T: 128x128x16 tcgen05.mma steps, fp32 accumulator in TMEM.
//   * Softmax: each thread owns one row; it loads its S row from TMEM, masks
//     (causal, bottom-right aligned, and past the context), and exponentiates
//     in the log2 domain against a running maximum that is only moved when a
//     tile's maximum exceeds it by more than 2^8, so the TMEM accumulator O
//     is rescaled rarely; P goes to shared memory as bf16/fp16 in the swizzled
//     K-major layout.
//   * O += P V: tcgen05.mma with V as an N-major (D-contiguous) operand,
//     accumulating in TMEM.
//   * Every mbarrier wait is bounded; a wait that gives up flags
//     PA_FLAG_TIMEOUT, drains what this CTA has in flight (bounded again),
//     frees TMEM and returns.
#include <math.h>

#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 128;
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefillMaps {
    CUtensorMap q;  // [total_q rows, H_q*D cols]
    CUtensorMap k;  // pool [N*bs rows, H_kv*D cols] (or packed [total_q, H_kv*D])
    CUtensorMap v;
};

struct PrefillArgs {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;  // null: keys are the packed k/v rows
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t log2_bs;
    int32_t box_rows;  // rows per K/V TMA box: min(block_size, 128)
    int32_t num_q_heads;
    int32_t group;
    int32_t total_q;
    int32_t qtiles;
    float scale_log2;
    void *out;
    int32_t *err_flag;
};

template <int D> struct PShape {
    static constexpr int kHalfBytes = 128 * 128;          // 128 rows x 64 columns (128 B) of a tile
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // Q, K or V tile of 128 rows
    static constexpr int kPBytes = 2 * kHalfBytes;           // 128 rows x 128 keys
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kTileBytes;                // stage s: K then V
    static constexpr int kOffP = kOffKV + 4 * kTileBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kSmem = kOffBar + 64 + 1024;       // barriers, TMEM slot, alignment slack
    static constexpr uint32_t kTmemCols = 256;               // S: 128 columns, O: D columns
};

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillMaps maps,
                                                              const PrefillArgs a) {
    using S = PShape<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1024-byte aligned for the 128-byte swizzle atoms
    uint8_t *sgen = smem_raw + (sb - raw);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int seq = blockIdx.z, h = blockIdx.y;
    const int qt = a.qtiles - 1 - static_cast<int>(blockIdx.x);  // later (heavier) tiles start first

    const int q_start = a.cu_q[seq], q_end = a.cu_q[seq + 1];
    const int Lq = q_end - q_start, Lk = a.cu_k[seq + 1] - a.cu_k[seq];
    const int P = Lk - Lq;
    const bool paged = a.block_tables != nullptr;
    const bool bad = Lq < 0 || P < 0 || q_start < 0 || q_end > a.total_q || (!paged && P != 0) ||
                     (paged && static_cast<int64_t>(Lk) > (static_cast<int64_t>(a.max_blocks) << a.log2_bs));
    if (bad) {
        if (tid == 0 && blockIdx.x == 0 && h == 0) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
        return;
    }
    if (tid == 0 && blockIdx.x == 0 && h == 0 && Lq > a.qtiles * kBM) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
    const int q0 = qt * kBM;
    if (q0 >= Lq) return;

    const int g = h / a.group;
    const int hi = min(Lk, P + q0 + kBM);  // keys [0, hi) are visible to some row of this tile
    const int nkt = (hi + kBN - 1) / kBN;

    const uint32_t sQ = sb + S::kOffQ;
    const uint32_t sP = sb + S::kOffP;
    const uint32_t bar_full = sb + S::kOffBar;  // + 8 * stage
    const uint32_t bar_q = bar_full + 16, bar_s = bar_full + 24, bar_o = bar_full + 32;
    const uint32_t tmem_slot = bar_full + 40;
    __shared__ int s_abort;

    if (tid == 0) {
        tc::mbar_init(bar_full, 1);
        tc::mbar_init(bar_full + 8, 1);
        tc::mbar_init(bar_q, 1);
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        tc::mbar_fence_init();
        tc::prefetch_tmap(&maps.q);
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.v);
        s_abort = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, S::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + S::kOffBar + 40);
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;

    auto sK = [&](int st) { return sb + S::kOffKV + st * 2 * S::kTileBytes; };
    auto sV = [&](int st) { return sK(st) + S::kTileBytes; };

    // ---- producer: one K/V tile through the block table (thread 0 only)
    auto load_kv = [&](int kt, int st) {
        const uint32_t bar = bar_full + 8 * st;
        const int j0 = kt * kBN;
        const int x = g * D;
        if (!paged) {
            tc::mbar_arrive_expect_tx(bar, 2 * S::kTileBytes);
            for (int hf = 0; hf < S::kHalves; ++hf) {
                tc::tma_load_2d(sK(st) + hf * S::kHalfBytes, &maps.k, x + hf * 64, q_start + j0, bar);
                tc::tma_load_2d(sV(st) + hf * S::kHalfBytes, &maps.v, x + hf * 64, q_start + j0, bar);
            }
            return;
        }
        const int rows = a.box_rows;
        const int npg = kBN / rows;
        const int pages_in_ctx = (Lk + (1 << a.log2_bs) - 1) >> a.log2_bs;
        int n = 0;
        for (int p = 0; p < npg; ++p)
            if (((j0 + p * rows) >> a.log2_bs) < pages_in_ctx) ++n;
        tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * rows * 128 * S::kHalves * 2));
        for (int p = 0; p < npg; ++p) {
            const int jp = j0 + p * rows;
            const int lp = jp >> a.log2_bs;
            if (lp >= pages_in_ctx) break;
            int page = a.block_tables[static_cast<int64_t>(seq) * a.max_blocks + lp];
            if (page < 0 || page >= a.num_blocks) {
                raise_flag(a.err_flag, PA_FLAG_BAD_BLOCK);
                page = 0;  // stay inside the pool; the sequence's output is then unspecified
            }
            const int y = (page << a.log2_bs) + (jp & ((1 << a.log2_bs) - 1));
            for (int hf = 0; hf < S::kHalves; ++hf) {
                tc::tma_load_2d(sK(st) + hf * S::kHalfBytes + p * rows * 128, &maps.k, x + hf * 64, y, bar);
                tc::tma_load_2d(sV(st) + hf * S::kHalfBytes + p * rows * 128, &maps.v, x + hf * 64, y, bar);
            }
        }
    };

    // in-flight bookkeeping for the bounded-wait exit path (thread 0)
    int loads_issued = 0;  // K/V tiles whose TMA was issued
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar_q, S::kTileBytes);
        for (int hf = 0; hf < S::kHalves; ++hf)
            tc::tma_load_2d(sQ + hf * S::kHalfBytes, &maps.q, h * D + hf * 64, q_start + q0, bar_q);
        load_kv(0, 0);
        loads_issued = 1;
        if (nkt > 1) {
            load_kv(1, 1);
            loads_issued = 2;
        }
    }

    constexpr uint32_t kIdS = tc::idesc_f16(kBM, kBN, IsBf16<T>::value, false);
    constexpr uint32_t kIdO = tc::idesc_f16(kBM, D, IsBf16<T>::value, true);

    const int row = tid;                 // TMEM lane and query row within the tile
    const int limit = P + q0 + row;      // last visible context position of this row
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    int waited_tiles = 0, s_commits = 0, o_commits = 0;

    for (int kt = 0; kt < nkt; ++kt) {
        const int st = kt & 1;
        const uint32_t full_phase = (kt >> 1) & 1;
        const int j0 = kt * kBN;
        const int valid = min(kBN, Lk - j0);
        if (tid == 0) {
            ok = tc::mbar_wait(bar_full + 8 * st, full_phase, kWaitCycles);
            if (kt == 0) ok = ok && tc::mbar_wait(bar_q, 0, kWaitCycles);
        }
        if (valid < kBN) {
            // rows past the context may hold anything (NaN included): zero them so P*V stays finite
            if (tid != 0) ok = tc::mbar_wait(bar_full + 8 * st, full_phase, kWaitCycles);
            const int nchunks = (kBN - valid) * 8 * S::kHalves;
            uint4 *vz = reinterpret_cast<uint4 *>(sgen + (sV(st) - sb));
            for (int c = tid; c < nchunks; c += kThreads) {
                const int hf = c / ((kBN - valid) * 8);
                const int rem = c % ((kBN - valid) * 8);
                vz[(hf * S::kHalfBytes + (valid + rem / 8) * 128) / 16 + rem % 8] = make_uint4(0, 0, 0, 0);
            }
            tc::fence_async_smem();
        }
        if (__syncthreads_or(!ok)) goto abort;
        waited_tiles = kt + 1;

        // ---- S = Q K^T
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks / 4) * S::kHalfBytes + (ks % 4) * 32;
                tc::umma_f16(tS, tc::smem_desc_sw128(sQ + off, 16, 1024), tc::smem_desc_sw128(sK(st) + off, 16, 1024),
                             kIdS, ks > 0);
            }
            tc::umma_commit(bar_s);
        }
        s_commits = kt + 1;
        ok = tc::mbar_wait(bar_s, kt & 1, kWaitCycles);
        tc::fence_after_sync();
        if (__syncthreads_or(!ok)) goto abort;

        // ---- softmax, part 1: the row of S, masked and scaled, and its maximum
        uint32_t sr[4][32];
        float mx = -INFINITY;
        const bool need_mask = (j0 + kBN - 1 > P + q0) || (j0 + kBN > Lk);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            tc::tmem_ld32(tS + lane_base + 32 * c, sr[c]);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = j0 + 32 * c + e;
                float s = __uint_as_float(sr[c][e]) * a.scale_log2;
                if (need_mask && (j > limit || j >= Lk)) s = -INFINITY;
                sr[c][e] = __float_as_uint(s);
                mx = fmaxf(mx, s);
            }
        }

        // ---- PV of the previous tile must be done: O is stable, P and its K/V stage are free
        if (kt > 0) {
            ok = tc::mbar_wait(bar_o, (kt - 1) & 1, kWaitCycles);
            tc::fence_after_sync();
        }
        if (tid == 0 && ok && kt >= 1 && kt + 1 < nkt) {
            load_kv(kt + 1, st ^ 1);
            loads_issued = kt + 2;
        }

        // ---- softmax, part 2: running maximum, rare rescale of O, P to shared memory
        const float m_new = fmaxf(m_used, mx);
        const bool rescale = kt > 0 && m_new > m_used + kRescaleThreshold;
        if (kt == 0) {
            m_used = m_new;
        } else if (__any_sync(0xffffffffu, rescale)) {
            const float alpha = rescale ? exp2f(m_used - m_new) : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(tO + lane_base + 32 * c, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tc::tmem_st32(tO + lane_base + 32 * c, o);
            }
            l_sum *= alpha;
            if (rescale) m_used = m_new;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {  // 8 keys = one 16-byte chunk
                uint32_t w[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float p0 = exp2f(__uint_as_float(sr[c][q8 * 8 + 2 * e2]) - m_used);
                    const float p1 = exp2f(__uint_as_float(sr[c][q8 * 8 + 2 * e2 + 1]) - m_used);
                    l_sum += p0 + p1;
                    w[e2] = Dt<T>::pack(p0, p1);
                }
                const int chunk = c * 4 + q8;  // 0..15 along the keys
                const int hf = chunk >> 3, cc = chunk & 7;
                const uint32_t addr = sP + hf * S::kHalfBytes + row * 128 + ((cc ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        if (__syncthreads_or(!ok)) goto abort;

        // ---- O += P V
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks) {
                const uint32_t aoff = (ks / 4) * S::kHalfBytes + (ks % 4) * 32;
                tc::umma_f16(tO, tc::smem_desc_sw128(sP + aoff, 16, 1024),
                             tc::smem_desc_sw128(sV(st) + ks * 16 * 128, S::kHalfBytes, 1024), kIdO,
                             (kt > 0 || ks > 0) ? 1u : 0u);
            }
            tc::umma_commit(bar_o);
        }
        o_commits = kt + 1;
    }

    // ---- epilogue: O / l -> out
    ok = tc::mbar_wait(bar_o, (nkt - 1) & 1, kWaitCycles);
    tc::fence_after_sync();
    if (__syncthreads_or(!ok)) goto abort;
    {
        const int qrow = q0 + row;
        const float inv_l = 1.f / l_sum;
        T *dst = static_cast<T *>(a.out) + (static_cast<int64_t>(q_start + qrow) * a.num_q_heads + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::tmem_ld32(tO + lane_base + 32 * c, o);
            if (qrow < Lq) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    uint4 v;
                    v.x = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 0]) * inv_l, __uint_as_float(o[q8 * 8 + 1]) * inv_l);
                    v.y = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 2]) * inv_l, __uint_as_float(o[q8 * 8 + 3]) * inv_l);
                    v.z = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 4]) * inv_l, __uint_as_float(o[q8 * 8 + 5]) * inv_l);
                    v.w = Dt<T>::pack(__uint_as_float(o[q8 * 8 + 6]) * inv_l, __uint_as_float(o[q8 * 8 + 7]) * inv_l);
                    *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * q8) = v;
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, S::kTmemCols);
    }
    return;

abort:
    // A wait gave up: flag it, let what this CTA started finish (bounded), free TMEM.
    if (tid == 0) {
        if (atomicExch(&s_abort, 1) == 0) raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
        for (int t = waited_tiles; t < loads_issued; ++t)
            tc::mbar_wait(bar_full + 8 * (t & 1), (t >> 1) & 1, kWaitCycles);
        if (s_commits > 0) tc::mbar_wait(bar_s, (s_commits - 1) & 1, kWaitCycles);
        if (o_commits > 0) tc::mbar_wait(bar_o, (o_commits - 1) & 1, kWaitCycles);
        tc::mbar_wait(bar_q, 0, kWaitCycles);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, S::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// 2-D map over a row-major [rows, cols] 16-bit matrix with (64 x box_rows) boxes, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, pa_dtype dt, int64_t cols, int64_t rows, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(m, dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

template <typename T, int D>
cudaError_t run(const PrefillMaps &maps, const PrefillArgs &a, int num_seqs, cudaStream_t stream) {
    using S = PShape<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    prefill_kernel<T, D><<<dim3(a.qtiles, a.num_q_heads, num_seqs), kThreads, S::kSmem, stream>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const void *q, const void *k, const void *v, const void *k_cache, const void *v_cache,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs,
                           int32_t total_q, int32_t max_seqlen_q, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_blocks, int32_t block_size, float scale, void *out, pa_dtype dtype,
                           int32_t *err_flag, cudaStream_t stream, const char **why) {
    *why = nullptr;
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return cudaSuccess;
    PrefillMaps maps;
    const int64_t kv_cols = static_cast<int64_t>(num_kv_heads) * head_dim;
    bool ok = make_map(&maps.q, q, dtype, static_cast<int64_t>(num_q_heads) * head_dim, total_q, kBM);
    int box_rows = kBN;
    if (block_tables) {
        box_rows = block_size < kBN ? block_size : kBN;
        const int64_t rows = static_cast<int64_t>(num_blocks) * block_size;
        ok = ok && make_map(&maps.k, k_cache, dtype, kv_cols, rows, box_rows) &&
             make_map(&maps.v, v_cache, dtype, kv_cols, rows, box_rows);
    } else {
        ok = ok && make_map(&maps.k, k, dtype, kv_cols, total_q, kBN) && make_map(&maps.v, v, dtype, kv_cols, total_q, kBN);
    }
    if (!ok) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or tensor too large)";
        return cudaErrorInvalidValue;
    }
    PrefillArgs a;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.log2_bs = ilog2(block_size);
    a.box_rows = box_rows;
    a.num_q_heads = num_q_heads;
    a.group = num_q_heads / num_kv_heads;
    a.total_q = total_q;
    a.qtiles = (max_seqlen_q + kBM - 1) / kBM;
    a.scale_log2 = scale * kLog2e;
    a.out = out;
    a.err_flag = err_flag;
    if (dtype == PA_BF16)
        return head_dim == 128 ? run<__nv_bfloat16, 128>(maps, a, num_seqs, stream)
                               : run<__nv_bfloat16, 64>(maps, a, num_seqs, stream);
    return head_dim == 128 ? run<__half, 128>(maps, a, num_seqs, stream) : run<__half, 64>(maps, a, num_seqs, stream);
}

}  // namespace pa
