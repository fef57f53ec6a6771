// Host helper: TMA tensor-map encoding through the driver entry point
// (looked up once through the runtime, so the library needs no -lcuda).
#include <cudaTypedefs.h>

#include "tmap.h"

namespace ret {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}
}  // namespace

bool tmap_available() { return encode_fn() != nullptr; }

bool tmap_encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                 const cuuint64_t *dims, const cuuint64_t *strides_bytes, const cuuint32_t *box,
                 CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, rank, const_cast<void *>(base), dims, strides_bytes, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ret
