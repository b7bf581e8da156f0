// Host-side construction of tiled TMA descriptors (CUtensorMap) through the
// driver entry point cuTensorMapEncodeTiled, fetched once per process.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdn {

// A row-major tensor of `rank` dimensions (dims[0] innermost, in elements),
// strides[i] = byte distance between consecutive indices of dimension i + 1,
// copied in boxes of box[0] x ... elements (no swizzle, no interleave, zero
// fill out of bounds).  Returns false if the driver rejects the description.
bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides, const uint32_t *box);
// The same with a shared-memory swizzle (the box's inner extent at most the swizzle span).
bool encode_tiled_swizzled(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                           const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                           CUtensorMapSwizzle swizzle);

}  // namespace gdn
