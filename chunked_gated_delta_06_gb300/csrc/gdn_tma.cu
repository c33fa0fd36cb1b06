// gdn_tma.cu -- TMA tensor-map encoding (host).
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "gdn_tma.h"

namespace gdn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // resolved once; the pointer never changes afterwards
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace

bool encode_rows_bf16(CUtensorMap *map, const void *base, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box2,
                      uint64_t inner) {
    auto fn = encode_fn();
    if (!fn || !base) return false;
    cuuint64_t dims[3] = {inner, d1 > 0 ? d1 : 1, d2 > 0 ? d2 : 1};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {64, 1, box2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gdn
