// TMA tensor-map encoding shared by the tensor-core kernels' launchers.
#pragma once

#include <cuda.h>

namespace ret {

bool tmap_available();
// Tiled map, no interleave, out-of-bounds elements read as zero.
bool tmap_encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                 const cuuint64_t *dims, const cuuint64_t *strides_bytes, const cuuint32_t *box,
                 CUtensorMapSwizzle swz);

}  // namespace ret
