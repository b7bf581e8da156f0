// Tiled TMA descriptors (see gdn_tmap.h).
#include "gdn_tmap.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace gdn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;  // benign race: same value
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides, const uint32_t *box)
{
    return encode_tiled_swizzled(map, type, rank, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_tiled_swizzled(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                           const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                           CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides[i];
    }
    return encode(map, type, static_cast<cuuint32_t>(rank), const_cast<void *>(base), d, s, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn
