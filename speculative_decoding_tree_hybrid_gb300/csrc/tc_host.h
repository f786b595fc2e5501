// Host-side TMA tensor maps shared by the tensor-core kernels (head
// dimension 128, bf16, 128-byte swizzle: a box row is one 64-dim half of a
// key, query or value row).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hta_internal.cuh"

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

// K/V of any layout as a 4-D map, boxes of box_rows rows x 64 dims:
// head-major [outer][Hkv][rows][128] as (d, rows, Hkv, outer), token-major
// [outer][rows][Hkv][128] as (d, Hkv, rows, outer)
inline bool encode_kv4(CUtensorMap *map, const void *base, bool nhd, int64_t rows, int64_t Hkv, int64_t outer,
                       int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t r = (cuuint64_t)(rows > 0 ? rows : 1), h = (cuuint64_t)Hkv, o = (cuuint64_t)(outer > 0 ? outer : 1);
    const cuuint64_t dims_hnd[4] = {128, r, h, o}, dims_nhd[4] = {128, h, r, o};
    const cuuint64_t str_hnd[3] = {128 * 2, r * 128 * 2, h * r * 128 * 2};
    const cuuint64_t str_nhd[3] = {128 * 2, h * 128 * 2, r * h * 128 * 2};
    const cuuint32_t box_hnd[4] = {64, (cuuint32_t)box_rows, 1, 1}, box_nhd[4] = {64, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), nhd ? dims_nhd : dims_hnd,
              nhd ? str_nhd : str_hnd, nhd ? box_nhd : box_hnd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four K/V maps of an attention launch: 3-D maps over (b, kv head) for
// the contiguous head-major layout, 4-D maps for every other one (boxes of
// min(page_size, tile) rows for a paged cache). The tree maps are encoded
// only when the launch reads the tree.
inline bool encode_kv_maps(const AttnParams &p, int64_t heads, int tile, CUtensorMap *kc, CUtensorMap *vc,
                           CUtensorMap *ks, CUtensorMap *vs) {
    if (!p.kv_generic) {
        if (!encode_kv(kc, p.k_cache, p.Lmax, heads, tile) || !encode_kv(vc, p.v_cache, p.Lmax, heads, tile))
            return false;
        return !p.include_tree ||
               (encode_kv(ks, p.k_spec, p.T, heads, tile) && encode_kv(vs, p.v_spec, p.T, heads, tile));
    }
    const bool nhd = p.kv_nhd != 0, paged = p.page_size > 0;
    const int64_t rows = paged ? p.page_size : p.Lmax, outer = paged ? p.num_pages : p.B;
    const int box = paged && p.page_size < tile ? p.page_size : tile;
    if (!encode_kv4(kc, p.k_cache, nhd, rows, p.Hkv, outer, box) ||
        !encode_kv4(vc, p.v_cache, nhd, rows, p.Hkv, outer, box))
        return false;
    return !p.include_tree || (encode_kv4(ks, p.k_spec, nhd, p.T, p.Hkv, p.B, tile) &&
                               encode_kv4(vs, p.v_spec, nhd, p.T, p.Hkv, p.B, tile));
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
