// tmap.cu — TMA tensor maps over row-major bf16 matrices (the activation and
// shared-expert operands of the prefill GEMM, the shared-expert tiles of the
// fused decode kernel).  The encoder is the driver's cuTensorMapEncodeTiled,
// reached through the runtime's entry-point query (no link against libcuda).
#include <cudaTypedefs.h>

#include "ds4g_internal.cuh"

namespace ds4g {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool encoder() {
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    return true;
}

bool tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    if (!encoder()) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_bf16_rowtile(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t tile_rows,
                       uint32_t tile_chunks) {
    if (!encoder() || cols % 64) return false;
    // dimensions (fastest first): 64 columns of a chunk, rows, 64-column chunks
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, tile_rows, tile_chunks};
    const cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ds4g
