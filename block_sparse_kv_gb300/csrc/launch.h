// Host-side helpers shared by the kernel launchers of libbskv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace bskv {

bskv_status cuda_check(cudaError_t e, const char* what);
bskv_status status_args(dev::StatusArgs* out);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda link).
// dims/strides are innermost first; strides_bytes has rank-1 entries (dim 1 upward).
bskv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides_bytes,
                         const uint32_t* box, CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int32_t meta_word(const bskv_plan* p, int h) { return p->meta[size_t(h)]; }

}  // namespace bskv
