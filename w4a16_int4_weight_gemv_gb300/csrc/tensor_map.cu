// Host side: tensor maps (TMA descriptors) of the packed weight matrix.
//
// The packed weights are a row-major [N][K/8] matrix of 32-bit words (eight
// 4-bit codes each, K contiguous).  A box is box_rows rows x 32 words (128
// bytes, 256 k per row), written to shared memory in the 128-byte swizzled
// layout (16-byte chunk j of row r lands at chunk j ^ (r % 8)), so that eight
// consecutive rows reading the same logical chunk hit eight different bank
// groups.  The warp-MMA kernel loads 16-row boxes, the tensor-core kernel
// 128-row boxes.
//
// cuTensorMapEncodeTiled is a driver function; it is looked up once through
// the runtime's entry-point query, so the library links no driver library.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace w4a16 {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool encode_weight_map(CUtensorMap* map, const void* wq, int N, int K, unsigned box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};  // bytes between rows
    const cuuint32_t box[2] = {kWeightBoxWords, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(wq), dims, strides, box,
              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace w4a16
