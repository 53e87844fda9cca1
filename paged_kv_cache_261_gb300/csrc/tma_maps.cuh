// Host-side construction of the TMA tensor maps the tensor-core kernels use.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 4-D map over a [num_blocks, block_size, num_kv_heads, 128] 16-bit cache, listed
// innermost first as (dim, kv head, token in block, block). One box = 64 dims x
// 1 kv head x block_size tokens: in shared memory block_size rows of 128 bytes,
// 128-byte swizzled. Coordinates past num_blocks read as zeros.
inline bool make_kv_cache_map(CUtensorMap *m, const void *base, int64_t num_blocks, int block_size,
                              int num_kv_heads, CUtensorMapDataType dt) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t D = 128, es = 2;
    cuuint64_t dims[4] = {D, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {D * es, (cuuint64_t)num_kv_heads * D * es,
                             (cuuint64_t)block_size * num_kv_heads * D * es};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)block_size, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa
