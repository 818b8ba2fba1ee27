// tma.cu -- host side of the tensor-memory-access copies: encoding 2-D tiled
// tensor maps through the driver entry point cuTensorMapEncodeTiled.
#include <cudaTypedefs.h>

#include <mutex>

#include "rz_kernels.h"

namespace rz {

namespace {
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

cudaError_t encode_tensor_map_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                                 uint64_t row_stride, uint32_t box_inner, uint32_t box_rows)
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return cudaErrorNotSupported;
    CUtensorMapDataType type;
    switch (elem_bytes) {
    case 1: type = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
    case 2: type = CU_TENSOR_MAP_DATA_TYPE_UINT16; break;
    case 4: type = CU_TENSOR_MAP_DATA_TYPE_UINT32; break;
    default: return cudaErrorInvalidValue;
    }
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace rz
