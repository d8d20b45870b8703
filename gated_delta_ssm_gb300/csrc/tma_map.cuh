// tma_map.cuh -- host-side encoding of the tensor maps the bulk tensor copies
// use (conv.cu, prefill_tc.cu). The driver's encoder is fetched through the
// runtime's entry-point query once per process, so nothing links the driver
// library directly.
#pragma once

#include <cuda.h>   // CUtensorMap and its enums
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn tensor_map_encoder()
{
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The [B][T][n_channels] view of token rows `row_stride` elements apart, copied
// in boxes of box_ch channels x box_rows rows of one sequence; rows before the
// sequence start or past its end read as zeros. False when the rows cannot be
// taken by tensor copies (base not 16-byte aligned, rows not a multiple of
// 16 bytes apart, or no encoder).
inline bool encode_rows_map(CUtensorMap *map, const void *x, bool bf16, int64_t n_channels,
                            int64_t row_stride, int64_t T, int64_t B, uint32_t box_ch,
                            uint32_t box_rows)
{
    const size_t es = bf16 ? 2 : 4;
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc || reinterpret_cast<uintptr_t>(x) % 16 != 0 || (row_stride * es) % 16 != 0)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)n_channels, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride * es, (cuuint64_t)row_stride * es * T};
    if (strides[1] >= (1ull << 40))
        return false;
    const cuuint32_t box[3] = {box_ch, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
               const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One 3-D tile copy into shared memory, completing on an mbarrier that was told
// to expect `bytes` (issued by one thread).
__device__ __forceinline__ void tile_copy_3d(const CUtensorMap *map, uint32_t dst, uint32_t mbar,
                                             uint32_t bytes, int c0, int t, int b)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(mbar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(t), "r"(b),
                    "r"(mbar)
                 : "memory");
}

}  // namespace gdn
