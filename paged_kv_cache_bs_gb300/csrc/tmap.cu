// Host side of the TMA loads: tensor maps over row-major 16-bit (or E4M3) matrices
// (the paged pool viewed as [num_blocks*block_size rows, H_kv*D columns], or a
// packed [tokens, heads*D] array), encoded through the driver entry point that
// the runtime hands out, so the library links against libcudart only.
#include <string.h>

#include "tc_common.cuh"

namespace pa {
namespace {

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

// The last few maps this thread encoded: a decode step re-encodes the same two
// pool maps every layer and every step.
struct MapKey {
    const void *base;
    int64_t cols, rows;
    int box_rows;
    int box_slices;  // 0: the 2-D map
    pa_dtype dt;
};
constexpr int kCacheSlots = 16;
thread_local MapKey t_keys[kCacheSlots];
thread_local CUtensorMap t_maps[kCacheSlots];
thread_local int t_next = 0;

}  // namespace

namespace {

bool cached(CUtensorMap *m, const MapKey &key) {
    for (int i = 0; i < kCacheSlots; ++i) {
        const MapKey &k = t_keys[i];
        if (k.base == key.base && k.cols == key.cols && k.rows == key.rows && k.box_rows == key.box_rows &&
            k.box_slices == key.box_slices && k.dt == key.dt) {
            memcpy(m, &t_maps[i], sizeof(CUtensorMap));
            return true;
        }
    }
    return false;
}

void remember(const CUtensorMap *m, const MapKey &key) {
    const int slot = t_next;
    t_next = (t_next + 1) % kCacheSlots;
    t_keys[slot] = key;
    memcpy(&t_maps[slot], m, sizeof(CUtensorMap));
}

CUtensorMapDataType tma_type(pa_dtype dt) {
    return dt == PA_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                         : dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

}  // namespace

bool make_tmap_rows(CUtensorMap *m, const void *base, pa_dtype dt, int64_t cols, int64_t rows, int box_rows) {
    const MapKey key{base, cols, rows, box_rows, 0, dt};
    if (cached(m, key)) return true;
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    // one box row is 128 bytes (the swizzle span): 64 16-bit elements or 128 E4M3 codes
    const bool f8 = dt == PA_E4M3;
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * (f8 ? 1 : 2))};
    const cuuint32_t box[2] = {f8 ? 128u : 64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(m, tma_type(dt), 2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    remember(m, key);
    return true;
}

bool make_tmap_row_slices(CUtensorMap *m, const void *base, pa_dtype dt, int64_t cols, int64_t rows, int box_rows,
                          int box_slices) {
    const MapKey key{base, cols, rows, box_rows, box_slices, dt};
    if (cached(m, key)) return true;
    EncodeTiled enc = encoder();
    if (!enc || dt == PA_E4M3 || cols % 64) return false;
    // dims: 64 elements of a 128-byte slice, the rows, the slices of a row
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2), 128u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_slices)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(m, tma_type(dt), 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    remember(m, key);
    return true;
}

}  // namespace pa
