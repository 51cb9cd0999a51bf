// TMA tensor-map encoding through the runtime's driver entry point (no libcuda link).
#include <cudaTypedefs.h>

#include <mutex>

#include "launch.h"

namespace bskv {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_lookup_err = cudaSuccess;
}  // namespace

bskv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides_bytes,
                         const uint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    g_lookup_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_lookup_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    set_error("cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(g_lookup_err));
    return BSKV_ERR_CUDA;
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  const CUresult r = g_encode(map, dt, cuuint32_t(rank), const_cast<void*>(base), d, s, b, e,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
    return BSKV_ERR_INVALID_ARG;
  }
  return BSKV_OK;
}

}  // namespace bskv
