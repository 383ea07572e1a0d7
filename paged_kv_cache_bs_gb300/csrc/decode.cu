// Paged GQA decode attention, split over context partitions.
//
// What is computed is the decode branch of the attention layer in
// "Inference engine: inside nano-vLLM" (flash_attn_with_kvcache with
// cache_seqlens and block_table): each sequence's single query attends over
// its context, position j read from cache row
// block_table[j / bs] * bs + j % bs ("nano-vLLM Part 2", section 2.2).
//
// Design (GB300): decode is HBM-bound, so everything serves the K/V stream,
// and the instructions spent per cache byte are kept low enough that one SM
// can pull its share of the HBM bandwidth (and more, when L2 serves pages that
// several sequences share).
//   * One CTA per (partition, kv head, sequence).  The G query heads of the
//     group share every K/V tile, so each cache byte is read once.
//   * A producer warp (one thread) fetches each 64-token K and V tile with
//     TMA, one box per page (or per 64 rows of a longer page) and per 128-byte
//     column slice of the kv head's row, into a ring with the 128-byte swizzle,
//     so the warp-matrix loads below are bank-conflict free: 3 stages with two
//     CTAs per SM, or, when pages are shorter than a tile (several boxes per
//     tile), 2 stages with three CTAs per SM.  Full / empty mbarriers hand
//     stages over; every wait is bounded.  The grid is sized from the
//     occupancy the device reports for the chosen ring.
//   * Each of 4 consumer warps owns 16 tokens of a tile.  It loads its K and
//     V fragments into registers and releases the stage at once, then
//     computes S^T = K Q^T and O^T += V^T P^T as m16n8k16 warp MMAs with the
//     G (<= 8) heads in the N dimension: the contraction is tiny, the tensor
//     cores only keep the per-byte instruction count low.
//   * Softmax is online, in fp32, in the log2 domain, with a lazily moved
//     maximum: the reference maximum changes (and O is rescaled) only when a
//     score exceeds it by more than 2^8, so most tiles need no warp reduction.
//     P is rounded to the input dtype for the PV MMA while the normaliser sums
//     the fp32 values.
//   * Warps merge through shared memory at the end of the partition; a
//     sequence with one partition writes its output directly, otherwise the
//     (max, sum, unnormalised O) partials go to the workspace and a second
//     kernel merges them by log-sum-exp, eight partitions per memory round
//     trip; both kernels are launched as programmatic dependents, so each
//     launch overlaps the kernel before it.
#include <math.h>

#include <algorithm>

#include <type_traits>

#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTile = 64;      // tokens per pipeline stage, 16 per consumer warp
// Ring depth: 3 stages with 2 CTAs per SM, or 2 stages with 3 CTAs per SM
// (more producers issuing when pages are short and a tile takes many boxes).
// An E4M3 pool halves the tile, so its kernel keeps 3 stages with 3 CTAs per SM.
template <int ST, bool F8 = false> constexpr int ctas_per_sm() { return (ST == 2 || F8) ? 3 : 2; }
constexpr int kF8Stages = 3;
constexpr int kMaxTablePages = 257;  // block-table entries one partition may touch
constexpr int kMaxPartition = 2048;
constexpr int kMinPartition = 128;
// Ragged batches: enough waves to absorb the length spread.  Measured on the Qwen3-0.6B-like
// workload (64 sequences, context U[128, 4096]): 4 waves (1024-token partitions) beat 8 (512)
// by 1.4 % on the bf16 pool and by 9 % on the E4M3 pool, whose CTAs stream half the bytes.
constexpr int kTargetWaves = 4;
// Tokens per partition of a shared prefix (one CTA per group chunk, kv head and partition):
// measured on the Qwen3-8B-like shared-prefix decode, one 512-token partition per prefix
// (149.5 us) beats two of 256 (155.6 us) and four of 128.
constexpr int kPrefixPartition = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

struct DecodeArgs {
    const void *q;
    int64_t q_row_stride;
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
    float *ws_o;     // [B][H_q][slots][D]  unnormalised partial outputs
    float2 *ws_ml;   // [B][H_q][slots]     (reference max, sum), log2 domain
    int32_t partition;
    int32_t max_parts;
    int32_t *err_flag;
    // fused store (null slot_mapping: none): sequence b's new K/V rows go to cache row slot_mapping[b]
    const int32_t *slot_mapping;
    const void *k_new;
    const void *v_new;
    int64_t k_new_stride, v_new_stride;  // elements between sequences' rows
    void *k_cache_w;
    void *v_cache_w;
    float k_scale, v_scale;  // E4M3 pool: K = code * k_scale, V = code * v_scale (1 for 16-bit pools)
    int32_t batch;
    // shared prefixes: the first prefix_ctas z indices of the grid are prefix CTAs (0: none)
    int32_t prefix_ctas;
    int32_t group_ctas;      // prefix CTAs per group: ceil(largest group / seqs_per_cta)
    int32_t seqs_per_cta;    // members one prefix CTA serves: 32 query rows / group
    const int32_t *group_offsets;
    const int32_t *group_seqs;
    const int32_t *prefix_lens;  // [batch], or null
    int32_t pre_partition;   // tokens per prefix partition
    int32_t pre_parts;       // workspace slots of prefix partials, before the private partitions'
    int32_t slots;           // workspace slots per (sequence, q head): pre_parts + max_parts
    // 1: wait for the previous kernel before reading the cache.  0 (the sequences' grid after the
    // prefix grid): that grid already waited before letting this one launch, and each CTA waits
    // for it (griddepcontrol.wait) before it reads the prefix partials and before it exits
    int32_t wait_at_start;
    // null, or three addresses {q, k_new, v_new} read when the kernels run, in place of the
    // fields above (a captured graph pointed at a new step's buffers between replays)
    const void *const *operands;
};

// Shared memory: the ring (each tile = D/64 slices of 64 rows x 128 bytes,
// every slice 1024-byte aligned for the swizzle), then the block-table slice,
// the mbarriers and the abort word.  After the loop the ring holds the warps'
// partial outputs for the merge.
template <int D, int ST, bool F8 = false> struct Shape {
    static constexpr int kStages = ST;
    static constexpr int kRowBytes = F8 ? D : 2 * D;  // one kv head's row
    static constexpr int kSlices = kRowBytes / 128;
    static constexpr int kSliceBytes = kTile * 128;
    static constexpr int kTileBytes = kSlices * kSliceBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
    static constexpr int kKSteps = D / 16;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kMergeBytes = kConsumerWarps * 8 * (D + 2) * 4;
    static constexpr int kBodyBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kTableOff = kBodyBytes;
    static constexpr int kBarOff = kTableOff + (kMaxTablePages * 4 + 7) / 8 * 8;
    static constexpr int kAbortOff = kBarOff + 2 * kStages * 8;
    static constexpr int kSmemBytes = kAbortOff + 16 + 1024;  // + slack to align the base to 1024
};

// Context length of sequence b, or -1 (to be flagged) when it is out of range.
__device__ __forceinline__ int context_len(const DecodeArgs &a, int b) {
    const int L = a.context_lens[b];
    const int64_t cap = static_cast<int64_t>(a.max_blocks) << a.log2_bs;
    return (L < 0 || L > cap) ? -1 : L;
}

// Fused store, by the producer warp of the CTA that holds the last partition of
// sequence b for kv head g: this head's slices of the new K and V rows go to
// cache row slot_mapping[b] (quantised to E4M3 codes for an F8 pool), which
// must be the slot of position L-1 (the token stored this step is the last one
// of the context), else the row is flagged and not written.  No other CTA
// reads that slice, and the proxy fence makes the plain stores visible to the
// TMA loads this warp issues next.
template <typename T, int D, bool F8>
__device__ __forceinline__ void store_new_row(const DecodeArgs &a, const void *k_new, const void *v_new, int b, int g,
                                              int L, int lane) {
    constexpr int kChunks = D / 8;  // 8-element (16-byte) chunks of one head's new row
    const bool is_v = lane >= kChunks;
    const int ci = is_v ? lane - kChunks : lane;
    // The slot, the page of position L-1 and this lane's chunk of the new row do not depend on
    // one another: they are loaded together, one memory round trip before the checks (the row
    // of a padding sequence, slot -1, is read and dropped).
    const int j = L - 1;
    const int slot = a.slot_mapping[b];
    const int pg = a.block_tables[static_cast<int64_t>(b) * a.max_blocks + (j >> a.log2_bs)];
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 2 * kChunks)
        raw = *reinterpret_cast<const uint4 *>(static_cast<const T *>(is_v ? v_new : k_new) +
                                               b * (is_v ? a.v_new_stride : a.k_new_stride) + g * D + ci * 8);
    if (slot == -1) return;
    const int64_t expect =
        (pg < 0 || pg >= a.num_blocks) ? -2 : (static_cast<int64_t>(pg) << a.log2_bs) + (j & ((1 << a.log2_bs) - 1));
    if (slot != expect) {
        if (lane == 0 && g == 0) raise_flag(a.err_flag, PA_FLAG_BAD_SLOT);
        return;
    }
    if (lane < 2 * kChunks) {
        const int64_t e = (static_cast<int64_t>(slot) * a.num_kv_heads + g) * D + ci * 8;  // pool element
        if constexpr (F8)
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(is_v ? a.v_cache_w : a.k_cache_w) + e) =
                quantize8_e4m3<T>(raw, is_v ? a.v_scale : a.k_scale);
        else
            *reinterpret_cast<uint4 *>(static_cast<T *>(is_v ? a.v_cache_w : a.k_cache_w) + e) = raw;
        asm volatile("fence.proxy.async.global;\n" ::: "memory");
    }
    __syncwarp();
}

// Byte offset of 16-byte chunk c (0 .. D/8-1) of tile row r in the swizzled layout.  A tile is
// kept as groups of 2^lbr rows (one TMA box: a page, or 64 rows of a longer page); inside a group
// the row's 128-byte slices follow one another, each 2^lbr rows of 128 bytes (with one slice per
// row this is plain row order).
template <int kSlices>
__device__ __forceinline__ uint32_t tile_off(int r, int c, int lbr) {
    const int rows = 1 << lbr;
    return (r >> lbr) * (rows * 128 * kSlices) + (c >> 3) * (rows * 128) + (r & (rows - 1)) * 128 +
           (((c & 7) ^ (r & 7)) << 4);
}

// Two E4M3 codes (low byte first) as an fp16 pair (low half first): exact,
// every E4M3 value is an fp16 value.  e4m3x2_lo converts bytes 0-1 of the
// word, e4m3x2_hi bytes 2-3 (the half is picked by the register move, no shift).
__device__ __forceinline__ uint32_t e4m3x2_lo(uint32_t codes) {
    uint32_t out;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(out) : "r"(codes));
    return out;
}
__device__ __forceinline__ uint32_t e4m3x2_hi(uint32_t codes) {
    uint32_t out;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(out) : "r"(codes));
    return out;
}

// One consumer lane's share of the online softmax of two query columns (N indices
// 2*(lane%4) and +1 of the warp's m16n8 tiles): the unnormalised O^T fragments, the
// running maxima m, the exponent references mu (m, or 0 while m = -inf) and the sums l.
template <int D> struct Acc {
    float o[D / 16][4];
    float m0, m1, l0, l1, mu0, mu1;
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = mu0 = mu1 = 0.f;
    }
};

// K and V fragments of 16 tokens of a stage (F8: V kept as byte-permuted codes).
template <int D, bool F8> struct Frags {
    uint32_t kf[D / 16][4];
    uint32_t vf[F8 ? D / 32 : D / 16][4];
};

// F8: the pool holds E4M3 codes (one byte per element, D = 128).  K and V are
// widened to fp16 in registers (exactly: every E4M3 value is an fp16 value)
// and the warp MMAs run in fp16, q converted once.  ldmatrix moves 16-bit
// units, i.e. pairs of codes, so the fragments use the contraction index in a
// fixed permutation, applied alike to both operands: for S^T = K Q^T, k-step
// ks and lane quad j = lane % 4 hold d = 16 ks + 4j + {0, 1} (fragment k = 2j,
// 2j+1) and 16 ks + 4j + {2, 3} (k = 2j + 8, 2j + 9); for O^T = V^T P^T, the
// transposed load gives each lane two tokens of two neighbouring d, one byte
// permutation splits them by d, and row m = lane / 4 of block mt holds
// d = 16 mt + 2m, row m + 8 holds d = 16 mt + 2m + 1.  V stays in codes until
// its MMA (fewer live registers).
template <int D, int kSlices, bool F8>
__device__ __forceinline__ void load_frags(Frags<D, F8> &f, uint32_t kb, uint32_t vb, int wrow, int lane, int lbr) {
    const int rk = wrow + (lane & 7) + ((lane >> 3) & 1) * 8, ck = lane >> 4;
    if constexpr (F8) {
        // one x4 load covers two 16-byte d chunks of the warp's 16 tokens
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4(kb + tile_off<kSlices>(rk, kp * 2 + ck, lbr), r0, r1, r2, r3);
            f.kf[2 * kp][0] = e4m3x2_lo(r0);
            f.kf[2 * kp][1] = e4m3x2_lo(r1);
            f.kf[2 * kp][2] = e4m3x2_hi(r0);
            f.kf[2 * kp][3] = e4m3x2_hi(r1);
            f.kf[2 * kp + 1][0] = e4m3x2_lo(r2);
            f.kf[2 * kp + 1][1] = e4m3x2_lo(r3);
            f.kf[2 * kp + 1][2] = e4m3x2_hi(r2);
            f.kf[2 * kp + 1][3] = e4m3x2_hi(r3);
            ldmatrix_x4_trans(vb + tile_off<kSlices>(rk, kp * 2 + ck, lbr), r0, r1, r2, r3);
            // bytes (token 2j, d 2m), (2j, 2m+1), (2j+1, 2m), (2j+1, 2m+1) -> split by d:
            // bytes 0-1 are tokens 2j, 2j+1 of d 2m, bytes 2-3 those of d 2m+1
            f.vf[kp][0] = __byte_perm(r0, 0, 0x3120);
            f.vf[kp][1] = __byte_perm(r1, 0, 0x3120);
            f.vf[kp][2] = __byte_perm(r2, 0, 0x3120);
            f.vf[kp][3] = __byte_perm(r3, 0, 0x3120);
        }
    } else {
        const int rv = wrow + (lane & 7) + (lane >> 4) * 8, cv = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
            ldmatrix_x4(kb + tile_off<kSlices>(rk, ks * 2 + ck, lbr), f.kf[ks][0], f.kf[ks][1], f.kf[ks][2], f.kf[ks][3]);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
            ldmatrix_x4_trans(vb + tile_off<kSlices>(rv, mt * 2 + cv, lbr), f.vf[mt][0], f.vf[mt][1], f.vf[mt][2],
                              f.vf[mt][3]);
    }
}

// The online-softmax step over 16 tokens whose first is context position `tok`: S^T = K Q^T,
// P = exp2(S - mu), O^T += V^T P^T.  Token j counts for column 0 (1) of this lane when
// j < lim0 (lim1); V rows at or past `end` may hold anything (NaN) and are zeroed.
template <typename MT, int D, bool F8>
__device__ __forceinline__ void attend16(Frags<D, F8> &f, Acc<D> &s, const uint32_t (&qb)[D / 16][2], float scale_log2,
                                         int tok, int end, int lim0, int lim1, int lane) {
    constexpr int kKSteps = D / 16;
    // S^T (16 tokens x 8 columns) = K (16 x D) . Q^T (D x 8), independent chains
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kKSteps; ks += 2) {
        Mma<MT>::run(sa, f.kf[ks][0], f.kf[ks][1], f.kf[ks][2], f.kf[ks][3], qb[ks][0], qb[ks][1]);
        Mma<MT>::run(sb, f.kf[ks + 1][0], f.kf[ks + 1][1], f.kf[ks + 1][2], f.kf[ks + 1][3], qb[ks + 1][0],
                     qb[ks + 1][1]);
    }
    // lane holds tokens lane/4 (s0, s1) and lane/4 + 8 (s2, s3) for columns 2*(lane%4), +1
    float s0 = (sa[0] + sb[0]) * scale_log2, s1 = (sa[1] + sb[1]) * scale_log2;
    float s2 = (sa[2] + sb[2]) * scale_log2, s3 = (sa[3] + sb[3]) * scale_log2;
    if (tok + 16 > min(lim0, lim1)) {  // some of these tokens are past a column's context
        const int j0 = tok + (lane >> 2);
        if (j0 >= lim0) s0 = -INFINITY;
        if (j0 >= lim1) s1 = -INFINITY;
        if (j0 + 8 >= lim0) s2 = -INFINITY;
        if (j0 + 8 >= lim1) s3 = -INFINITY;
    }
    if (tok + 16 > end) {
        // V rows past the end: zero them in the fragments, whose tokens are 2*(lane%4) + {0, 1}
        // (regs 0, 1) and + 8 (regs 2, 3)
        const int jt = tok + (lane & 3) * 2;
        if constexpr (F8) {  // codes: bytes 0, 2 are token 2j (+8 in regs 1, 3), bytes 1, 3 token 2j+1
            const uint32_t lo = (jt < end ? 0x00FF00FFu : 0u) | (jt + 1 < end ? 0xFF00FF00u : 0u);
            const uint32_t hi = (jt + 8 < end ? 0x00FF00FFu : 0u) | (jt + 9 < end ? 0xFF00FF00u : 0u);
#pragma unroll
            for (int kp = 0; kp < kKSteps / 2; ++kp) {
                f.vf[kp][0] &= lo;
                f.vf[kp][1] &= hi;
                f.vf[kp][2] &= lo;
                f.vf[kp][3] &= hi;
            }
        } else {
            const uint32_t lo = (jt < end ? 0xFFFFu : 0u) | (jt + 1 < end ? 0xFFFF0000u : 0u);
            const uint32_t hi = (jt + 8 < end ? 0xFFFFu : 0u) | (jt + 9 < end ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < kKSteps; ++mt) {
                f.vf[mt][0] &= lo;
                f.vf[mt][1] &= lo;
                f.vf[mt][2] &= hi;
                f.vf[mt][3] &= hi;
            }
        }
    }
    // move the reference maximum only when a score exceeds it by more than 2^8
    const bool grow = fmaxf(s0, s2) > s.m0 + kRescaleThreshold || fmaxf(s1, s3) > s.m1 + kRescaleThreshold;
    if (__any_sync(0xffffffffu, grow)) {
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
        mx0 = warp_max_xor(mx0, 4);
        mx1 = warp_max_xor(mx1, 4);
        mx0 = warp_max_xor(mx0, 8);
        mx1 = warp_max_xor(mx1, 8);
        mx0 = warp_max_xor(mx0, 16);
        mx1 = warp_max_xor(mx1, 16);
        const float mn0 = fmaxf(s.m0, mx0), mn1 = fmaxf(s.m1, mx1);
        const float nu0 = mn0 == -INFINITY ? 0.f : mn0;  // all masked so far: keep exp2 finite
        const float nu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float c0 = tc::ex2_approx(s.mu0 - nu0), c1 = tc::ex2_approx(s.mu1 - nu1);
        s.l0 *= c0;
        s.l1 *= c1;
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) {
            s.o[mt][0] *= c0;
            s.o[mt][1] *= c1;
            s.o[mt][2] *= c0;
            s.o[mt][3] *= c1;
        }
        s.m0 = mn0;
        s.m1 = mn1;
        s.mu0 = nu0;
        s.mu1 = nu1;
    }
    const float p0 = tc::ex2_approx(s0 - s.mu0), p1 = tc::ex2_approx(s1 - s.mu1);
    const float p2 = tc::ex2_approx(s2 - s.mu0), p3 = tc::ex2_approx(s3 - s.mu1);
    s.l0 += p0 + p2;
    s.l1 += p1 + p3;
    // P^T as the B operand (16 tokens x 8 columns): transpose the two 8x8 halves
    const uint32_t pb0 = movmatrix_trans(Dt<MT>::pack(p0, p1));
    const uint32_t pb1 = movmatrix_trans(Dt<MT>::pack(p2, p3));
    // O^T (D x 8) += V^T (D x 16 tokens) . P^T (16 x 8)
    if constexpr (F8) {
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) {
            const uint32_t pa = f.vf[mt >> 1][(mt & 1) * 2], pc = f.vf[mt >> 1][(mt & 1) * 2 + 1];
            Mma<MT>::run(s.o[mt], e4m3x2_lo(pa), e4m3x2_hi(pa), e4m3x2_lo(pc), e4m3x2_hi(pc), pb0, pb1);
        }
    } else {
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt)
            Mma<MT>::run(s.o[mt], f.vf[mt][0], f.vf[mt][1], f.vf[mt][2], f.vf[mt][3], pb0, pb1);
    }
}

// The producer thread's loop: each 64-token tile of context positions [start, end) into the
// ring, one TMA box per page (or per 64 rows of a longer page) and kv-head row slice.  bt_s
// holds the physical pages of logical pages first_page, first_page + 1, ...  Returns the tiles
// started (a wait that gave up stops the loop, flagged).
template <int D, int ST, bool F8>
__device__ __forceinline__ int produce_tiles(const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                             const CUtensorMap *tm_k_tail, const CUtensorMap *tm_v_tail,
                                             const DecodeArgs &a, int g, int start, int end, int first_page,
                                             const int32_t *bt_s, uint32_t ring, uint32_t bars,
                                             volatile int *abort_s) {
    using S = Shape<D, ST, F8>;
    constexpr int kStages = ST;
    const int ntiles = (end - start + kTile - 1) / kTile;
    const int box_rows = min(1 << a.log2_bs, kTile);
    const int bs_mask = (1 << a.log2_bs) - 1;
    int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages;
        if (t >= kStages &&
            !tc::mbar_wait_or_abort(bars + 8 * (kStages + s), ((t / kStages) - 1) & 1, kWaitCycles, abort_s)) {
            raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
            break;
        }
        const int tile_start = start + t * kTile;
        const int valid = min(kTile, end - tile_start);
        const uint32_t full = bars + 8 * s;
        const uint32_t kdst = ring + s * S::kStageBytes;
        const uint32_t vdst = kdst + S::kTileBytes;
        if (valid < kTile && box_rows == kTile) {
            // the context ends inside this tile of one page: fetch it in 16-row boxes up to the
            // end instead of a whole 64-row box (rows past the end are masked either way)
            constexpr int kTailRows = 16;
            const int nsub = (valid + kTailRows - 1) / kTailRows;
            tc::mbar_arrive_expect_tx(full, nsub * kTailRows * S::kRowBytes * 2);
            const int y0 = (bt_s[(tile_start >> a.log2_bs) - first_page] << a.log2_bs) + (tile_start & bs_mask);
            for (int i = 0; i < nsub; ++i) {
#pragma unroll
                for (int h = 0; h < S::kSlices; ++h) {
                    const int x = g * D + h * (F8 ? 128 : 64);  // elements: 128 bytes per slice
                    const uint32_t off = h * (kTile * 128) + i * kTailRows * 128;
                    tc::tma_load_2d(kdst + off, tm_k_tail, x, y0 + i * kTailRows, full);
                    tc::tma_load_2d(vdst + off, tm_v_tail, x, y0 + i * kTailRows, full);
                }
            }
            issued = t + 1;
            continue;
        }
        const int nbox = (valid + box_rows - 1) / box_rows;
        tc::mbar_arrive_expect_tx(full, nbox * box_rows * S::kRowBytes * 2);
        for (int i = 0; i < nbox; ++i) {
            const int j = tile_start + i * box_rows;
            const int y = (bt_s[(j >> a.log2_bs) - first_page] << a.log2_bs) + (j & bs_mask);
            const uint32_t box_off = i * box_rows * 128 * S::kSlices;
            if constexpr (S::kSlices == 1) {
                const int x = g * D;  // elements: one 128-byte slice holds the kv head's row
                tc::tma_load_2d(kdst + box_off, tm_k, x, y, full);
                tc::tma_load_2d(vdst + box_off, tm_v, x, y, full);
            } else {
                // both 128-byte slices of the kv head's rows in one 3-D box, slice by slice
                tc::tma_load_3d(kdst + box_off, tm_k, 0, y, g * S::kSlices, full);
                tc::tma_load_3d(vdst + box_off, tm_v, 0, y, g * S::kSlices, full);
            }
        }
        issued = t + 1;
    }
    return issued;
}

// After a wait gave up: let every load this CTA started land before the CTA leaves.
template <int ST> __device__ __forceinline__ void drain(uint32_t bars, int issued) {
    for (int s = 0; s < ST && s < issued; ++s) {
        const int t_last = s + ST * ((issued - 1 - s) / ST);
        tc::mbar_wait(bars + 8 * s, (t_last / ST) & 1, kWaitCycles);
    }
}

// Loads the block-table entries of logical pages [first_page, first_page + span) of
// `table` (a sequence's row) into registers, one memory round trip for the CTA of NT threads.
template <int NT> constexpr int per_thread() { return (kMaxTablePages + NT - 1) / NT; }
constexpr int kPerThread = per_thread<kThreads>();
template <int NT>
__device__ __forceinline__ void prefetch_table(int (&pg)[per_thread<NT>()], const int32_t *table, int first_page,
                                               int span, int tid) {
#pragma unroll
    for (int k = 0; k < per_thread<NT>(); ++k) {
        const int i = tid + k * NT;
        pg[k] = i < span ? table[first_page + i] : 0;
    }
}

// Stores the first npages prefetched entries into the shared slice, a bad id flagged and
// read as page 0.
template <int NT>
__device__ __forceinline__ void publish_table(const int (&pg)[per_thread<NT>()], int32_t *bt_s, int npages,
                                              const DecodeArgs &a, int tid) {
#pragma unroll
    for (int k = 0; k < per_thread<NT>(); ++k) {
        const int i = tid + k * NT;
        if (i < npages) {
            int p = pg[k];
            if (p < 0 || p >= a.num_blocks) {
                raise_flag(a.err_flag, PA_FLAG_BAD_BLOCK);
                p = 0;
            }
            bt_s[i] = p;
        }
    }
}

// Tokens at the start of sequence b's context that its group's prefix CTAs read (0: not
// grouped), clamped to what the workspace holds; a length that is no whole number of pages
// or not below the context is flagged (the descriptor is the caller's).
__device__ __forceinline__ int shared_prefix(const DecodeArgs &a, int b, int L, bool flag) {
    if (!a.prefix_lens) return 0;
    const int P = a.prefix_lens[b];
    if (P <= 0) return 0;
    if (flag && ((P & ((1 << a.log2_bs) - 1)) || P >= L)) raise_flag(a.err_flag, PA_FLAG_BAD_GROUP);
    return min(P, min(a.pre_parts * a.pre_partition, a.max_blocks << a.log2_bs));
}

// Partials of sequence b's output (per q head): its prefix partitions, then its private
// partitions [p_lo, p_hi) (slots pre_parts + p).  Every kernel that writes or merges them
// derives the same numbers from the same inputs.
struct PartialSet {
    int npre, p_lo, p_hi;
    __device__ __forceinline__ int count() const { return npre + p_hi - p_lo; }
    __device__ __forceinline__ int slot(int i, int pre_parts) const {
        return i < npre ? i : pre_parts + p_lo + (i - npre);
    }
};
__device__ __forceinline__ PartialSet partial_set(const DecodeArgs &a, int b) {
    const int L = max(context_len(a, b), 0);
    const int P = shared_prefix(a, b, L, false);
    const int ps = min(P, L);
    PartialSet r;
    r.npre = P > 0 ? (P + a.pre_partition - 1) / a.pre_partition : 0;
    r.p_lo = ps / a.partition;
    r.p_hi = ps < L ? (L + a.partition - 1) / a.partition : r.p_lo;
    return r;
}

// The shared-prefix kernel: one CTA per (group chunk, kv head, prefix partition) streams the
// group's shared pages once for up to 32 query rows -- the G heads of up to 32 / G member
// sequences -- and writes each row's softmax partial to the workspace.  Row r is head r % G of
// the chunk's member r / G.  Rows come in four groups of 8 (the N dimension of the MMAs); two
// consumer warps own each row group and split every 64-token tile between them (32 tokens
// each), then merge their states through shared memory.
// Sequence of member mi of a prefix chunk whose members start at group_seqs[m0] (nm of them),
// or -1 past the chunk or for an index outside the batch.
__device__ __forceinline__ int group_member(const DecodeArgs &a, int m0, int nm, int mi) {
    if (mi >= nm) return -1;
    const int b = a.group_seqs[m0 + mi];
    return (b >= 0 && b < a.batch) ? b : -1;
}

// Consumer warps of the shared-prefix kernel: 4 (one per row group, walking every 16-token slice
// of a tile) or 8 (two per row group, half a tile each, merged at the end).  Measured on the
// Qwen3-8B-like shared-prefix decode: 4 warps with a 2-stage ring, one partition per prefix,
// 149.5 us per step; 8 warps 154.4 us; 3 stages 151.6 us.
constexpr int kPrefixConsumerWarps = 4;
constexpr int kPrefixStages = 2;  // ring depth
constexpr int kPrefixProducerWarp = kPrefixConsumerWarps;
constexpr int kPrefixThreads = (kPrefixConsumerWarps + 1) * 32;
constexpr int kPrefixRows = 32;  // query rows of one prefix CTA

template <typename T, int D, int ST>
__global__ void __launch_bounds__(kPrefixThreads, ctas_per_sm<kPrefixStages>())
    decode_prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_k_tail, const __grid_constant__ CUtensorMap tm_v_tail,
                         const DecodeArgs a) {
    using S = Shape<D, ST, false>;
    constexpr int kStages = ST;
    constexpr int kPerT = per_thread<kPrefixThreads>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + S::kTableOff);
    const uint32_t ring = smem_u32(smem);
    const uint32_t bars = smem_u32(smem + S::kBarOff);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + S::kAbortOff);
    const int pp = blockIdx.x, g = blockIdx.y;
    const int gi = blockIdx.z / a.group_ctas, chunk = blockIdx.z % a.group_ctas;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the previous kernel on the stream (this step's store) first; the sequences' grid may
    // launch once every prefix CTA is past this point
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    const int off0 = a.group_offsets[gi], off1 = a.group_offsets[gi + 1];
    if (off0 < 0 || off1 > a.batch || off0 > off1) {  // group_seqs has room for batch entries
        if (tid == 0 && pp == 0 && g == 0 && chunk == 0) raise_flag(a.err_flag, PA_FLAG_BAD_GROUP);
        return;
    }
    const void *q_src = a.operands ? a.operands[0] : a.q;  // the step's q (see DecodeArgs::operands)
    if (reinterpret_cast<uintptr_t>(q_src) & 15) {  // flagged by the sequences' grid as well
        if (tid == 0) raise_flag(a.err_flag, PA_FLAG_BAD_VALUE);
        return;
    }
    const int m0 = off0 + chunk * a.seqs_per_cta;
    const int nm = min(a.seqs_per_cta, off1 - m0);  // members of this chunk
    if (nm <= 0) return;
    const int leader = a.group_seqs[off0];
    if (leader < 0 || leader >= a.batch) {
        if (tid == 0 && pp == 0 && g == 0) raise_flag(a.err_flag, PA_FLAG_BAD_GROUP);
        return;
    }
    const int start = pp * a.pre_partition;
    const int first_page = start >> a.log2_bs;
    const int span = min(a.max_blocks, ((start + a.pre_partition - 1) >> a.log2_bs) + 1) - first_page;
    int pg_pre[kPerT];
    prefetch_table<kPrefixThreads>(pg_pre, a.block_tables + static_cast<int64_t>(leader) * a.max_blocks, first_page,
                                   span, tid);
    const int Ll = max(context_len(a, leader), 0);
    const int P = shared_prefix(a, leader, Ll, false);
    const int end = min(start + a.pre_partition, P);
    if (start >= end) return;
    const int npages = ((end - 1) >> a.log2_bs) - first_page + 1;

    publish_table<kPrefixThreads>(pg_pre, bt_s, npages, a, tid);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(bars + 8 * s, 1);
            tc::mbar_init(bars + 8 * (kStages + s), kPrefixConsumerWarps);
        }
        *abort_s = 0;
        tc::mbar_fence_init();
    }
    if (warp == kPrefixProducerWarp && lane == 0) {
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    __syncthreads();  // table slice, barriers ready

    Acc<D> acc;
    acc.init();
    int issued = 0;
    const int ntiles = (end - start + kTile - 1) / kTile;
    // this warp's row group rg and tile half hh; this lane's two columns (rows rc0, rc0 + 1) and
    // its B-operand row rq: member sequences and their context limits (loaded while the first
    // tile is in flight)
    const int G = a.group;
    constexpr int kSplit = kPrefixConsumerWarps / 4;         // warps sharing a row group
    constexpr int kSubPerWarp = (kTile / 16) / kSplit;        // 16-token slices per warp and tile
    const int rg = warp / kSplit, hh = warp % kSplit;
    const int rc0 = 8 * rg + 2 * (lane & 3), rq = 8 * rg + (lane >> 2);
    int b0 = -1, b1 = -1;
    if (warp == kPrefixProducerWarp) {
        if (lane == 0)
            issued = produce_tiles<D, ST, false>(&tm_k, &tm_v, &tm_k_tail, &tm_v_tail, a, g, start, end, first_page,
                                                 bt_s, ring, bars, abort_s);
    } else {
        b0 = group_member(a, m0, nm, rc0 / G);
        b1 = group_member(a, m0, nm, (rc0 + 1) / G);
        const int bq = group_member(a, m0, nm, rq / G);
        const int lim0 = b0 >= 0 ? min(P, max(context_len(a, b0), 0)) : 0;
        const int lim1 = b1 >= 0 ? min(P, max(context_len(a, b1), 0)) : 0;
        // query fragments (B operand of S^T = K Q^T): row rq's head
        uint32_t qb[D / 16][2];
        const int dq = (lane & 3) * 2;
        const T *qrow = bq >= 0 ? static_cast<const T *>(q_src) + static_cast<int64_t>(bq) * a.q_row_stride +
                                      static_cast<int64_t>(g * G + rq % G) * D
                                : nullptr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            if (qrow) {
                qb[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + dq);
                qb[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + dq);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
        const int lbr = min(a.log2_bs, 6);
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % kStages;
            const bool ok = tc::mbar_wait_or_abort(bars + 8 * s, (t / kStages) & 1, kWaitCycles, abort_s);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
                break;
            }
            const uint32_t kb = ring + s * S::kStageBytes;
            const uint32_t vb = kb + S::kTileBytes;
            const int tile_start = start + t * kTile;
#pragma unroll 1
            for (int u = kSubPerWarp * hh; u < kSubPerWarp * (hh + 1); ++u) {
                if (tile_start + 16 * u >= end) break;
                Frags<D, false> f;
                load_frags<D, S::kSlices, false>(f, kb, vb, 16 * u, lane, lbr);
                attend16<T, D, false>(f, acc, qb, a.scale_log2, tile_start + 16 * u, end, lim0, lim1, lane);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bars + 8 * (kStages + s));  // stage free for the next tile
        }
    }
    // the caller's descriptor: every member of the chunk shares the leader's pages of this
    // partition (checked once, by the first kv head's CTAs), reads the same prefix and has
    // tokens after it
    if (g == 0) {
        for (int i = tid; i < nm * npages; i += kPrefixThreads) {
            const int b = a.group_seqs[m0 + i / npages];
            if (b < 0 || b >= a.batch ||
                a.block_tables[static_cast<int64_t>(b) * a.max_blocks + first_page + i % npages] != bt_s[i % npages])
                raise_flag(a.err_flag, PA_FLAG_BAD_GROUP);
        }
        if (pp == 0 && tid < nm) {
            const int b = a.group_seqs[m0 + tid];
            if (b < 0 || b >= a.batch || a.prefix_lens[b] != a.prefix_lens[leader] || context_len(a, b) <= P)
                raise_flag(a.err_flag, PA_FLAG_BAD_GROUP);
        }
    }
    __syncthreads();
    if (*abort_s) {
        if (warp == kPrefixProducerWarp && lane == 0) drain<ST>(bars, issued);
        return;
    }
    // the two warps of a row group hold the same columns in the same lanes: the second warp
    // hands its state over through shared memory (the ring is free), the first merges and writes
    constexpr int kStateFloats = (D / 16) * 4 + 4;  // O fragments, then (m0, m1, l0, l1)
    float *xs = reinterpret_cast<float *>(smem) + (rg * 32 + lane) * kStateFloats;
    if (warp < kPrefixConsumerWarps) {
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 4);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 4);
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 8);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 8);
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 16);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 16);
        if (kSplit == 2 && hh == 1) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) xs[mt * 4 + e] = acc.o[mt][e];
            xs[(D / 16) * 4 + 0] = acc.m0 == -INFINITY ? -INFINITY : acc.mu0;
            xs[(D / 16) * 4 + 1] = acc.m1 == -INFINITY ? -INFINITY : acc.mu1;
            xs[(D / 16) * 4 + 2] = acc.l0;
            xs[(D / 16) * 4 + 3] = acc.l1;
        }
    }
    __syncthreads();
    if (warp >= kPrefixConsumerWarps || hh == 1) return;
    const int dr = lane >> 2;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int b = c ? b1 : b0;
        if (b < 0) continue;
        const float ma = (c ? acc.m1 : acc.m0) == -INFINITY ? -INFINITY : (c ? acc.mu1 : acc.mu0);
        const float mb = kSplit == 2 ? xs[(D / 16) * 4 + c] : -INFINITY;
        const float M = fmaxf(ma, mb);
        const float wa = M == -INFINITY ? 0.f : exp2f(ma - M), wb = M == -INFINITY ? 0.f : exp2f(mb - M);
        const int hq = g * G + (rc0 + c) % G;
        const int64_t idx = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.slots + pp;
        float *o = a.ws_o + idx * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const float x0 = kSplit == 2 ? xs[mt * 4 + c] * wb : 0.f, x1 = kSplit == 2 ? xs[mt * 4 + c + 2] * wb : 0.f;
            o[mt * 16 + dr] = acc.o[mt][c] * wa + x0;
            o[mt * 16 + dr + 8] = acc.o[mt][c + 2] * wa + x1;
        }
        if (dr == 0)
            a.ws_ml[idx] = make_float2(M, (c ? acc.l1 : acc.l0) * wa + (kSplit == 2 ? xs[(D / 16) * 4 + 2 + c] * wb : 0.f));
    }
}

template <typename T, int D, int ST, bool F8>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<ST, F8>())
    decode_partition_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_k_tail,
                            const __grid_constant__ CUtensorMap tm_v_tail, const DecodeArgs a) {
    using S = Shape<D, ST, F8>;
    using MT = typename std::conditional<F8, __half, T>::type;  // MMA operand type
    constexpr int kStages = ST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Launched as a programmatic dependent of the previous kernel on the stream (the store
    // of this step, or the shared-prefix grid): wait for it to finish before reading the cache
    // (after a shared-prefix grid the wait comes later, see wait_at_start), then let the next
    // kernel be launched right away (it waits for this grid itself).
    if (a.wait_at_start) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + S::kTableOff);
    const uint32_t ring = smem_u32(smem);
    const uint32_t bars = smem_u32(smem + S::kBarOff);  // full[s] at 8s, empty[s] at 8(kStages + s)
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + S::kAbortOff);

    const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the step's q and new rows: the call's, or the addresses the operands array holds now
    // (loaded with the length and the table below, one round trip)
    const void *q_src = a.q, *k_src = a.k_new, *v_src = a.v_new;
    if (a.operands) {
        q_src = a.operands[0];
        if (a.slot_mapping) {
            k_src = a.operands[1];
            v_src = a.operands[2];
        }
        // every access below is a 4- or 16-byte vector: an unaligned address is flagged and the
        // CTA leaves (the same decision in every thread, before any barrier)
        if ((reinterpret_cast<uintptr_t>(q_src) | reinterpret_cast<uintptr_t>(k_src) |
             reinterpret_cast<uintptr_t>(v_src)) & 15) {
            if (tid == 0) raise_flag(a.err_flag, PA_FLAG_BAD_VALUE);
            if (!a.wait_at_start) asm volatile("griddepcontrol.wait;\n" ::: "memory");
            return;
        }
    }

    // The block-table entries this partition can touch are loaded together with the context
    // length (one memory round trip before the first TMA instead of two); entries past the
    // context are loaded (they lie inside the table's row) but never used.
    const int part_start = p * a.partition;
    const int first_page = part_start >> a.log2_bs;
    const int span = min(a.max_blocks, ((part_start + a.partition - 1) >> a.log2_bs) + 1) - first_page;
    int pg_pre[kPerThread];
    prefetch_table<kThreads>(pg_pre, a.block_tables + static_cast<int64_t>(b) * a.max_blocks, first_page, span, tid);
    int L = context_len(a, b);
    if (L < 0) {
        if (p == 0 && tid == 0) raise_flag(a.err_flag, PA_FLAG_BAD_LENGTH);
        L = 0;
    }
    // a shared prefix [0, ps) is read by the group's prefix CTAs: this partition covers the
    // rest of [part_start, part_start + partition)
    const int P = shared_prefix(a, b, L, p == 0 && g == 0 && tid == 0);
    const int ps = min(P, L);
    const int start = max(part_start, ps);
    T *out = static_cast<T *>(a.out);
    if (start >= min(part_start + a.partition, L)) {
        if (p == 0 && L == 0) {  // empty context (e.g. a padding row): zero output, no page read
            for (int i = tid; i < a.group * D; i += kThreads)
                out[(static_cast<int64_t>(b) * a.num_q_heads + g * a.group + i / D) * D + i % D] =
                    Dt<T>::from_float(0.f);
        }
        // a new token needs a context position outside the shared prefix
        if (a.slot_mapping && g == 0 && tid == 0 && (L == 0 ? p == 0 : (L - 1) / a.partition == p) &&
            a.slot_mapping[b] != -1)
            raise_flag(a.err_flag, PA_FLAG_BAD_SLOT);
        if (!a.wait_at_start) asm volatile("griddepcontrol.wait;\n" ::: "memory");
        return;
    }
    const int end = min(L, part_start + a.partition);
    // this sequence's partials: its prefix partitions (the prefix grid's), then its private
    // partitions; with one private partition this CTA writes the output, folding in the
    // prefix partials, else the merge kernel merges them all
    const int npre = P > 0 ? (P + a.pre_partition - 1) / a.pre_partition : 0;
    const bool direct = (L + a.partition - 1) / a.partition - ps / a.partition == 1;
    const int ntiles = (end - start + kTile - 1) / kTile;

    // block-table slice of this partition, validated once (a bad id is flagged and read as page 0)
    const int npages = ((end - 1) >> a.log2_bs) - first_page + 1;  // <= span
    publish_table<kThreads>(pg_pre, bt_s, npages, a, tid);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(bars + 8 * s, 1);
            tc::mbar_init(bars + 8 * (kStages + s), kConsumerWarps);
        }
        *abort_s = 0;
        tc::mbar_fence_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }

    // query fragments (B operand of S^T = K Q^T): head lane/4 of the group
    uint32_t qb[S::kKSteps][2];
    if constexpr (F8) {  // fp16, contraction index d = 16 ks + 4j + {0..3} (see the F8 note above)
        const int hq = lane >> 2, j = lane & 3;
        const T *qrow = static_cast<const T *>(q_src) + static_cast<int64_t>(b) * a.q_row_stride +
                        static_cast<int64_t>(g * a.group + hq) * D;
#pragma unroll
        for (int ks = 0; ks < S::kKSteps; ++ks) {
            if (hq < a.group && warp < kConsumerWarps) {
                const T *qd = qrow + ks * 16 + 4 * j;
                qb[ks][0] = Dt<__half>::pack(static_cast<float>(qd[0]), static_cast<float>(qd[1]));
                qb[ks][1] = Dt<__half>::pack(static_cast<float>(qd[2]), static_cast<float>(qd[3]));
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
    } else {
        const int hq = lane >> 2;
        const int dq = (lane & 3) * 2;
        const T *qrow = static_cast<const T *>(q_src) + static_cast<int64_t>(b) * a.q_row_stride +
                        static_cast<int64_t>(g * a.group + hq) * D;
#pragma unroll
        for (int ks = 0; ks < S::kKSteps; ++ks) {
            if (hq < a.group && warp < kConsumerWarps) {
                qb[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + dq);
                qb[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + dq);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
    }
    __syncthreads();  // table slice, barriers ready

    Acc<D> acc;
    acc.init();
    int issued = 0;  // tiles the producer started

    if (warp == kProducerWarp) {
        if (a.slot_mapping && end == L) store_new_row<T, D, F8>(a, k_src, v_src, b, g, L, lane);
        if (lane == 0)
            issued = produce_tiles<D, ST, F8>(&tm_k, &tm_v, &tm_k_tail, &tm_v_tail, a, g, start, end, first_page, bt_s,
                                              ring, bars, abort_s);
    } else {
        const int lbr = min(a.log2_bs, 6);  // log2 of the rows of one TMA box (at most the 64-row tile)
        const int wrow = warp * 16;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % kStages;
            const bool ok = tc::mbar_wait_or_abort(bars + 8 * s, (t / kStages) & 1, kWaitCycles, abort_s);
            if (!__all_sync(0xffffffffu, ok)) {  // leave together: the warp-wide instructions below
                if (lane == 0) raise_flag(a.err_flag, PA_FLAG_TIMEOUT);
                break;
            }
            const uint32_t kb = ring + s * S::kStageBytes;
            const uint32_t vb = kb + S::kTileBytes;
            Frags<D, F8> f;
            load_frags<D, S::kSlices, F8>(f, kb, vb, wrow, lane, lbr);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bars + 8 * (kStages + s));  // stage free for the next tile
            attend16<MT, D, F8>(f, acc, qb, a.scale_log2, start + t * kTile + wrow, end, end, end, lane);
        }
    }
    __syncthreads();
    if (*abort_s) {
        // a wait gave up (flagged above): let every load this CTA started land, then leave
        if (warp == kProducerWarp && lane == 0) drain<ST>(bars, issued);
        if (!a.wait_at_start) asm volatile("griddepcontrol.wait;\n" ::: "memory");
        return;
    }

    // merge the consumer warps (the ring is free: every load has landed and been read)
    float *mo = reinterpret_cast<float *>(smem);    // [warp][head 8][D]
    float *mm = mo + kConsumerWarps * 8 * D;        // [warp][head 8]  reference max
    float *ml = mm + kConsumerWarps * 8;            // [warp][head 8]  sum
    if (warp < kConsumerWarps) {
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 4);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 4);
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 8);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 8);
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, 16);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, 16);
        const int h0 = (lane & 3) * 2;
        const int dr = lane >> 2;
        // the two d of this lane's O^T fragment rows (see the F8 permutation above)
        const int d_lo = F8 ? 2 * dr : dr, d_hi = F8 ? 2 * dr + 1 : dr + 8;
        float *w = mo + warp * 8 * D;
#pragma unroll
        for (int mt = 0; mt < S::kKSteps; ++mt) {
            w[h0 * D + mt * 16 + d_lo] = acc.o[mt][0];
            w[(h0 + 1) * D + mt * 16 + d_lo] = acc.o[mt][1];
            w[h0 * D + mt * 16 + d_hi] = acc.o[mt][2];
            w[(h0 + 1) * D + mt * 16 + d_hi] = acc.o[mt][3];
        }
        if (lane < 4) {  // a warp whose tokens were all masked has m = -inf and sum 0: weight 0 below
            mm[warp * 8 + h0] = acc.m0 == -INFINITY ? -INFINITY : acc.mu0;
            mm[warp * 8 + h0 + 1] = acc.m1 == -INFINITY ? -INFINITY : acc.mu1;
            ml[warp * 8 + h0] = acc.l0;
            ml[warp * 8 + h0 + 1] = acc.l1;
        }
    }
    __syncthreads();
    // the prefix partials are complete once the prefix grid has finished
    if (direct && npre > 0) asm volatile("griddepcontrol.wait;\n" ::: "memory");

    for (int i = tid; i < a.group * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + h]);
        float accv = 0.f, sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = exp2f(mm[w * 8 + h] - M);  // a warp with no token has max -inf: weight 0
            accv += mo[(w * 8 + h) * D + d] * wt;
            sum += ml[w * 8 + h] * wt;
        }
        if constexpr (F8) accv *= a.v_scale;
        const int hq = g * a.group + h;
        if (direct && npre > 0) {  // fold in the prefix partitions' partials, loaded together
            const int64_t base = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.slots;
            for (int k0 = 0; k0 < npre; k0 += 4) {
                float2 pml[4];
                float po[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    pml[j] = k0 + j < npre ? __ldcg(a.ws_ml + base + k0 + j) : make_float2(-INFINITY, 0.f);
                    po[j] = k0 + j < npre ? __ldcg(a.ws_o + (base + k0 + j) * D + d) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float Mn = fmaxf(M, pml[j].x);
                    if (Mn == -INFINITY) continue;
                    const float cold = exp2f(M - Mn), cnew = exp2f(pml[j].x - Mn);
                    accv = accv * cold + po[j] * cnew;
                    sum = sum * cold + pml[j].y * cnew;
                    M = Mn;
                }
            }
        }
        if (direct) {
            out[(static_cast<int64_t>(b) * a.num_q_heads + hq) * D + d] = Dt<T>::from_float(accv / sum);
        } else {
            const int64_t idx = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.slots + a.pre_parts + p;
            a.ws_o[idx * D + d] = accv;
            if (d == 0) a.ws_ml[idx] = make_float2(M, sum);
        }
    }
    if (!a.wait_at_start) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Log-sum-exp merge of the partials of sequences whose context spans several private partitions:
// the prefix partitions' partials (slots [0, prefix partitions)) and the private partitions'
// (slot pre_parts + p for partition p).  One block per (q head, sequence), one thread per d; the
// partials are loaded eight at a time and folded in with an online maximum: one memory round
// trip per eight partials.  (A wider layout -- float4 chunks of several heads per thread, fewer
// blocks -- measured slower: its larger blocks, resident early beside the partition grid's last
// wave, slowed that wave.)
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a) {
    constexpr int kBatch = 8;
    const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    // context_lens and prefix_lens are inputs of the call: this grid launches only after every
    // partition CTA has passed its own wait on the previous kernel, so they may be read before
    // the wait
    const PartialSet ps = partial_set(a, b);
    const int npriv = ps.p_hi - ps.p_lo, n = ps.count();
    if (npriv == 1 || n == 0) return;  // written by its only private partition (prefix partials folded in)
    // launched early (programmatic dependent launch): wait until the partition grid has
    // finished and its partials are visible
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int64_t base = (static_cast<int64_t>(b) * a.num_q_heads + hq) * a.slots;
    float M = -INFINITY, acc = 0.f, sum = 0.f;
    for (int i0 = 0; i0 < n; i0 += kBatch) {
        float2 ml[kBatch];
        float o[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (i0 + j < n) {
                const int64_t slot = base + ps.slot(i0 + j, a.pre_parts);
                ml[j] = a.ws_ml[slot];
                o[j] = a.ws_o[slot * D + d];
            } else {
                ml[j] = make_float2(-INFINITY, 0.f);
                o[j] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const float Mn = fmaxf(M, ml[j].x);
            if (Mn == -INFINITY) continue;  // padding
            const float cold = exp2f(M - Mn), cnew = exp2f(ml[j].x - Mn);
            acc = acc * cold + o[j] * cnew;
            sum = sum * cold + ml[j].y * cnew;
            M = Mn;
        }
    }
    static_cast<T *>(a.out)[(static_cast<int64_t>(b) * a.num_q_heads + hq) * D + d] = Dt<T>::from_float(acc / sum);
}

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

}  // namespace

// Opt the partition kernel in to its shared memory (a per-device function attribute) and ask
// for the largest shared-memory carveout, so that ctas_per_sm<ST>() CTAs fit on an SM.
template <typename T, int D, int ST, bool F8 = false> cudaError_t prepare_partition_kernel() {
    cudaError_t e = cudaFuncSetAttribute(decode_partition_kernel<T, D, ST, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Shape<D, ST, F8>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_partition_kernel<T, D, ST, F8>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// The shared-prefix kernel's shared-memory opt-in.
template <typename T, int D> cudaError_t prepare_prefix_kernel() {
    cudaError_t e = cudaFuncSetAttribute(decode_prefix_kernel<T, D, kPrefixStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Shape<D, kPrefixStages>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_prefix_kernel<T, D, kPrefixStages>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

template <int D, int ST, bool F8 = false> int occupancy() {
    int occ = 0;
    if (prepare_partition_kernel<__nv_bfloat16, D, ST, F8>() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_partition_kernel<__nv_bfloat16, D, ST, F8>,
                                                      kThreads, Shape<D, ST, F8>::kSmemBytes) != cudaSuccess ||
        occ < 1)
        occ = 1;
    return occ < ctas_per_sm<ST, F8>() ? occ : ctas_per_sm<ST, F8>();
}

// Resident partition CTAs the current device holds at once for this kernel variant:
// 16-bit pool with 2 or 3 stages and head dim 64 or 128, or the E4M3 pool (head dim 128).
static int resident_ctas(int stages, int head_dim, bool fp8) {
    static int cached[64][3][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2 * 148;
    const int vi = fp8 ? 2 : stages == 2 ? 0 : 1, hi = head_dim == 64 ? 0 : 1;
    if (!cached[dev][vi][hi]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
        const int occ = vi == 2 ? occupancy<128, kF8Stages, true>()
                        : vi == 1 ? (hi ? occupancy<128, 3>() : occupancy<64, 3>())
                                  : (hi ? occupancy<128, 2>() : occupancy<64, 2>());
        cached[dev][vi][hi] = occ * sms;
    }
    return cached[dev][vi][hi];
}

// Ring depth for a block size.  Pages shorter than a tile make every tile several TMA boxes;
// three CTAs per SM (2 stages each) then keep more producers issuing (measured: block size 16,
// 3-4 % faster without shared pages, 13 % with them), while for longer pages the deeper ring
// is slightly ahead.
static int stages_for(int32_t block_size) { return block_size < kTile ? 2 : 3; }

// Loads every partition and merge kernel of the 16-bit pools into the current context (CUDA loads
// kernels lazily, at first use, by default), so that later launches load no code.
cudaError_t preload_decode_kernels() {
    cudaFuncAttributes fa;
    const void *kernels[] = {
        reinterpret_cast<const void *>(decode_partition_kernel<__nv_bfloat16, 128, 3, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__nv_bfloat16, 128, 2, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__nv_bfloat16, 64, 3, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__nv_bfloat16, 64, 2, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__half, 128, 3, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__half, 128, 2, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__half, 64, 3, false>),
        reinterpret_cast<const void *>(decode_partition_kernel<__half, 64, 2, false>),
        reinterpret_cast<const void *>(decode_combine_kernel<__nv_bfloat16, 128>),
        reinterpret_cast<const void *>(decode_combine_kernel<__nv_bfloat16, 64>),
        reinterpret_cast<const void *>(decode_combine_kernel<__half, 128>),
        reinterpret_cast<const void *>(decode_combine_kernel<__half, 64>),
    };
    for (const void *k : kernels) {
        const cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t max_blocks_per_seq, int32_t block_size, bool fp8, const pa_decode_options *opt) {
    DecodePlan pl{};
    pl.stages = fp8 ? kF8Stages : (opt && opt->stages) ? opt->stages : stages_for(block_size);
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int64_t pairs = static_cast<int64_t>(batch) * num_kv_heads;
    const int64_t slots = resident_ctas(pl.stages, head_dim, fp8);
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
        while (part > kMinPartition && pairs * ((cap + part - 1) / part) < kTargetWaves * slots) part /= 2;
    }
    if (opt && opt->partition) part = opt->partition;  // caller's override (validated by the C ABI)
    while (part / block_size > kMaxTablePages - 1) part = (part / 2 + kTile - 1) / kTile * kTile;  // table slice fits
    if (part < kTile) part = kTile;
    pl.partition = static_cast<int>(part);
    pl.max_parts = static_cast<int>(cap > 0 ? (cap + part - 1) / part : 1);
    // shared prefixes: one CTA per (group chunk, kv head, prefix partition) in front of the grid
    if (opt && opt->num_groups > 0) {
        const int64_t lim = (kMaxTablePages - 1) * static_cast<int64_t>(block_size);
        int64_t pre = opt->prefix_partition ? opt->prefix_partition
                                            : std::min<int64_t>((opt->max_prefix_len + kTile - 1) / kTile * kTile,
                                                                kPrefixPartition);
        while (pre > lim) pre = (pre / 2 + kTile - 1) / kTile * kTile;
        pl.pre_partition = static_cast<int>(std::max<int64_t>(pre, kTile));
        pl.pre_parts = (opt->max_prefix_len + pl.pre_partition - 1) / pl.pre_partition;
            pl.seqs_per_cta = kPrefixRows / (num_q_heads / num_kv_heads);
        pl.group_ctas = (opt->max_group_size + pl.seqs_per_cta - 1) / pl.seqs_per_cta;
        pl.prefix_ctas = static_cast<int64_t>(opt->num_groups) * pl.group_ctas;
    } else {
        pl.pre_partition = kTile;
        pl.pre_parts = pl.seqs_per_cta = pl.group_ctas = 0;
        pl.prefix_ctas = 0;
    }
    pl.slots = pl.pre_parts + pl.max_parts;
    const size_t n = static_cast<size_t>(batch) * num_q_heads * pl.slots;
    const size_t ml_bytes = (n * sizeof(float2) + 255) / 256 * 256;
    pl.ws_bytes = ml_bytes + n * head_dim * sizeof(float);
    return pl;
}

cudaError_t launch_decode(const void *q, int64_t q_row_stride, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t num_blocks, int32_t block_size, float scale, void *out, void *workspace,
                          const DecodePlan &plan, pa_dtype dtype, int32_t *err_flag, cudaStream_t stream,
                          const FusedStore *fused, const Fp8Scales *fp8, const pa_decode_options *opt) {
    if (batch == 0) return cudaSuccess;
    DecodeArgs a;
    a.q = q;
    a.q_row_stride = q_row_stride;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_q_heads / num_kv_heads;
    a.num_blocks = num_blocks;
    a.log2_bs = ilog2(block_size);
    a.scale_log2 = scale * kLog2e * (fp8 ? fp8->k_scale : 1.f);
    a.k_scale = fp8 ? fp8->k_scale : 1.f;
    a.v_scale = fp8 ? fp8->v_scale : 1.f;
    a.out = out;
    const size_t n = static_cast<size_t>(batch) * num_q_heads * plan.slots;
    const size_t ml_bytes = (n * sizeof(float2) + 255) / 256 * 256;
    a.ws_ml = static_cast<float2 *>(workspace);
    a.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ml_bytes);
    a.partition = plan.partition;
    a.max_parts = plan.max_parts;
    a.batch = batch;
    const bool groups = plan.prefix_ctas > 0 && opt;
    a.prefix_ctas = groups ? static_cast<int32_t>(plan.prefix_ctas) : 0;
    a.group_ctas = plan.group_ctas;
    a.seqs_per_cta = plan.seqs_per_cta;
    a.group_offsets = groups ? opt->group_offsets : nullptr;
    a.group_seqs = groups ? opt->group_seqs : nullptr;
    a.prefix_lens = groups ? opt->prefix_lens : nullptr;
    a.pre_partition = plan.pre_partition;
    a.pre_parts = groups ? plan.pre_parts : 0;
    a.slots = plan.slots;
    a.wait_at_start = 1;
    a.err_flag = err_flag;
    a.slot_mapping = fused ? fused->slot_mapping : nullptr;
    a.k_new = fused ? fused->k : nullptr;
    a.v_new = fused ? fused->v : nullptr;
    a.k_new_stride = fused ? fused->k_row_stride : 0;
    a.v_new_stride = fused ? fused->v_row_stride : 0;
    a.k_cache_w = const_cast<void *>(k_cache);
    a.v_cache_w = const_cast<void *>(v_cache);
    a.operands = opt ? opt->operands : nullptr;

    // the pool as [num_blocks * block_size rows, H_kv * D columns]; one box = min(block_size, 64)
    // rows (a box never crosses a page) of one kv head's row: 128 bytes (E4M3 codes, or 16-bit at
    // D = 64) by a 2-D map, or both 128-byte halves of a 16-bit D = 128 row by a 3-D map
    CUtensorMap tm_k, tm_v;
    const int64_t rows = static_cast<int64_t>(num_blocks) * block_size;
    const int64_t cols = static_cast<int64_t>(num_kv_heads) * head_dim;
    const int box_rows = block_size < kTile ? block_size : kTile;
    const pa_dtype pool = fp8 ? PA_E4M3 : dtype;
    const bool two_slices = !fp8 && head_dim == 128;
    const bool maps_ok =
        two_slices ? make_tmap_row_slices(&tm_k, k_cache, pool, cols, rows, box_rows, 2) &&
                         make_tmap_row_slices(&tm_v, v_cache, pool, cols, rows, box_rows, 2)
                   : make_tmap_rows(&tm_k, k_cache, pool, cols, rows, box_rows) &&
                         make_tmap_rows(&tm_v, v_cache, pool, cols, rows, box_rows);
    // the tail of a context inside a 64-row tile of a long page is fetched in 16-row boxes (2-D maps,
    // one 128-byte slice each); with pages shorter than a tile the boxes are already a page long
    CUtensorMap tm_k_tail = tm_k, tm_v_tail = tm_v;
    const bool tails_ok = box_rows != kTile || (make_tmap_rows(&tm_k_tail, k_cache, pool, cols, rows, 16) &&
                                                make_tmap_rows(&tm_v_tail, v_cache, pool, cols, rows, 16));
    if (!maps_ok || !tails_ok) return cudaErrorInvalidValue;

    auto run = [&](auto kern_part, auto kern_comb, auto prepare, int smem, int d, auto kern_pre, auto prepare_pre,
                   int smem_pre) -> cudaError_t {
        cudaError_t err = prepare();
        if (err != cudaSuccess) return err;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (a.prefix_ctas > 0) {
            // the shared-prefix CTAs first, then the sequences' CTAs as its programmatic dependent
            err = prepare_pre();
            if (err != cudaSuccess) return err;
            cfg.gridDim = dim3(a.pre_parts, a.num_kv_heads, a.prefix_ctas);
            cfg.blockDim = dim3(kPrefixThreads);
            cfg.dynamicSmemBytes = smem_pre;
            err = cudaLaunchKernelEx(&cfg, kern_pre, tm_k, tm_v, tm_k_tail, tm_v_tail, a);
            if (err != cudaSuccess) return err;
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            a.wait_at_start = 0;
        }
        cfg.gridDim = dim3(a.max_parts, a.num_kv_heads, batch);
        err = cudaLaunchKernelEx(&cfg, kern_part, tm_k, tm_v, tm_k_tail, tm_v_tail, a);
        if (err != cudaSuccess) return err;
        if (a.max_parts > 1) {
            cfg.gridDim = dim3(a.num_q_heads, batch);
            cfg.blockDim = dim3(d);
            cfg.dynamicSmemBytes = 0;
            err = cudaLaunchKernelEx(&cfg, kern_comb, a);
        }
        return err;
    };
#define PA_DECODE_RUN(T, D, ST)                                                                                  \
    run(decode_partition_kernel<T, D, ST, false>, decode_combine_kernel<T, D>,                                 \
        prepare_partition_kernel<T, D, ST, false>, Shape<D, ST>::kSmemBytes, D,                                 \
        decode_prefix_kernel<T, D, kPrefixStages>, prepare_prefix_kernel<T, D>,                                 \
        Shape<D, kPrefixStages>::kSmemBytes)
#define PA_DECODE_RUN_F8(T)  /* no shared-prefix grid over an E4M3 pool */                                    \
    run(decode_partition_kernel<T, 128, kF8Stages, true>, decode_combine_kernel<T, 128>,                       \
        prepare_partition_kernel<T, 128, kF8Stages, true>, Shape<128, kF8Stages, true>::kSmemBytes, 128,       \
        decode_prefix_kernel<T, 128, kPrefixStages>, prepare_prefix_kernel<T, 128>,                             \
        Shape<128, kPrefixStages>::kSmemBytes)
    const bool bf = dtype == PA_BF16, d128 = head_dim == 128, deep = plan.stages == 3;
    cudaError_t e;
    if (fp8)  // head_dim 128, checked by the caller
        e = bf ? PA_DECODE_RUN_F8(__nv_bfloat16) : PA_DECODE_RUN_F8(__half);
    else if (bf)
        e = d128 ? (deep ? PA_DECODE_RUN(__nv_bfloat16, 128, 3) : PA_DECODE_RUN(__nv_bfloat16, 128, 2))
                 : (deep ? PA_DECODE_RUN(__nv_bfloat16, 64, 3) : PA_DECODE_RUN(__nv_bfloat16, 64, 2));
    else
        e = d128 ? (deep ? PA_DECODE_RUN(__half, 128, 3) : PA_DECODE_RUN(__half, 128, 2))
                 : (deep ? PA_DECODE_RUN(__half, 64, 3) : PA_DECODE_RUN(__half, 64, 2));
#undef PA_DECODE_RUN
#undef PA_DECODE_RUN_F8
    return e;
}

}  // namespace pa
