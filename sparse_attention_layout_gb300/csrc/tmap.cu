// Host-side TMA descriptor encoding through the driver entry point (no link
// dependency on libcuda: the runtime hands out the driver function).
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace bsp {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

int make_tmap_2d(CUtensorMap* map, const void* base, int is_bf16, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, int swizzle_bytes) {
    auto fn = encode_fn();
    if (!fn) return BSP_ERR_CUDA;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    else if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    else if (swizzle_bytes == 0) sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSP_OK : BSP_ERR_UNSUPPORTED;
}

int make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return BSP_ERR_CUDA;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSP_OK : BSP_ERR_UNSUPPORTED;
}

int make_tmap_3d(CUtensorMap* map, const void* base, int is_bf16, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t box0, uint32_t box1, int swizzle_bytes) {
    auto fn = encode_fn();
    if (!fn) return BSP_ERR_CUDA;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : (swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                                : (swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                                                       : CU_TENSOR_MAP_SWIZZLE_NONE)),
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSP_OK : BSP_ERR_UNSUPPORTED;
}

int make_tmap_panels(CUtensorMap* map, const void* base, int is_bf16, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_panels) {
    auto fn = encode_fn();
    if (!fn) return BSP_ERR_CUDA;
    if (cols % 64 != 0) return BSP_ERR_UNSUPPORTED;
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_panels};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSP_OK : BSP_ERR_UNSUPPORTED;
}

}  // namespace bsp
