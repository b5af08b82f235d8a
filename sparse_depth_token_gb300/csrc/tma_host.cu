// Host-side creation of TMA tensor maps (bf16, 128-byte swizzle, zero fill
// outside the tensor). The driver entry point is looked up once through the
// runtime, so the library needs no link-time dependency on libcuda.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace xmod {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}

bool tma_available() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

bool tma_map_bf16(CUtensorMap* m, const void* base, int rank, const int64_t* dims,
                  const int64_t* strides_bytes, const int* box) {
  if (!tma_available() || rank < 2 || rank > 3) return false;
  cuuint64_t d[3];
  cuuint64_t st[2];
  cuuint32_t bx[3];
  cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = (cuuint64_t)strides_bytes[i];
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d,
                  st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace xmod
