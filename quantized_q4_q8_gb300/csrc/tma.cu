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

static PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

cudaError_t encode_tensor_map(CUtensorMap *map, const void *base, int elem_bytes, int rank, const uint64_t *dims,
                              const uint64_t *strides, const uint32_t *box)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    CUtensorMapDataType type;
    switch (elem_bytes) {
    case 1: type = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
    case 2: type = CU_TENSOR_MAP_DATA_TYPE_UINT16; break;
    case 4: type = CU_TENSOR_MAP_DATA_TYPE_UINT32; break;
    default: return cudaErrorInvalidValue;
    }
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    const CUresult r = enc(map, type, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tensor_map_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                                 uint64_t row_stride, uint32_t box_inner, uint32_t box_rows)
{
    const uint64_t dims[2] = {inner, rows};
    const uint64_t strides[1] = {row_stride};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_tensor_map(map, base, elem_bytes, 2, dims, strides, box);
}

}  // namespace rz
