// tc_host.cu -- host helpers of the tensor-core kernels: TMA descriptors and
// device properties.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_host.h"

namespace lora {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    // Resolved once per process through the runtime, so the library needs no
    // link-time dependency on the driver library.
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace

bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                       uint32_t box_rows, bool swizzle128)
{
    auto fn = encode_fn();
    if (fn == nullptr || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows)
{
    auto fn = encode_fn();
    if (fn == nullptr || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_blocks(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                           uint32_t box_blocks)
{
    auto fn = encode_fn();
    if (fn == nullptr || rows == 0 || cols == 0 || cols % 64 != 0) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_blocks};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_wmaps(WMaps *maps, const void *base, uint64_t cols, uint64_t rows)
{
    return make_tmap_bf16_2d(&maps->m16, base, cols, rows, 64, 16, true) &&
           make_tmap_bf16_2d(&maps->m32, base, cols, rows, 64, 32, true) &&
           make_tmap_bf16_2d(&maps->m64, base, cols, rows, 64, 64, true);
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace lora
