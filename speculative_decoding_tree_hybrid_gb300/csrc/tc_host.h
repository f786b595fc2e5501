// Host-side TMA tensor maps shared by the tensor-core kernels (head
// dimension 128, bf16, 128-byte swizzle: a box row is one 64-dim half of a
// key, query or value row).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace hta {
namespace tch {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [heads][rows][d=128] bf16 (one (b, kv head) per z), boxes of box_rows rows x 64 dims
inline bool encode_kv(CUtensorMap *map, const void *base, int64_t rows, int64_t heads, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)heads};
    const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)(rows > 0 ? rows : 1) * 128 * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [B][T][Hq][d=128] bf16 as a 4-D map; a box is 64 dims x G heads x nt
// tree nodes of one sequence (box row t_local * G + g), zero past T
inline bool encode_q(CUtensorMap *map, const void *base, int B, int T, int Hq, int G, int nt) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {128, (cuuint64_t)Hq, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {128 * 2, (cuuint64_t)Hq * 128 * 2, (cuuint64_t)T * Hq * 128 * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)nt, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tch
}  // namespace hta
