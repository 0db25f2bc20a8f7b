// tmap.h -- host-side TMA tensor-map encoding for the paged cache and q.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry-point lookup (no
// link against libcuda).  Null if the driver does not provide it.
inline EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// A paged cache [NB, 16, Hkv, D] bf16 viewed as (D, Hkv, 16, NB): one box is 64
// columns x 1 head x the 16 slots of one page (2 KiB, 128-byte swizzle), so a
// page of one head lands as 16 rows of 128 bytes per 64-column half.
inline bool encode_cache_map(CUtensorMap* map, const void* base, int head_dim, int num_kv_heads, int64_t num_blocks,
                             CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_kv_heads), 16,
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2,
                                   static_cast<cuuint64_t>(16) * num_kv_heads * head_dim * 2};
    const cuuint32_t box[4] = {64, 1, 16, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [T, Hq, D] bf16 viewed as (D, Hq, T): one box is 64 columns x G heads x
// tokens_per_box tokens (rows ordered token-major, head-minor).
inline bool encode_q_map(CUtensorMap* map, const void* base, int head_dim, int num_q_heads, int64_t num_tokens,
                         int group, int tokens_per_box) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens_per_box)};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa
