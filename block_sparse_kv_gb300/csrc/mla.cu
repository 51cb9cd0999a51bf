// Sparse MLA FP8 decode on the 5th-generation tensor cores (tcgen05 + TMEM).
#include "common.cuh"
#include "internal.h"
#include "launch.h"

using namespace bskv;

extern "C" bskv_status bskv_run_mla_sparse(const bskv_plan* plan, const void* query,
                                           const void* kv_rows, int64_t num_rows,
                                           const int32_t* indices, float bmm1_scale,
                                           float bmm2_scale, void* out, float* lse,
                                           void* float_ws, size_t float_ws_bytes, void* stream) {
  (void)plan; (void)query; (void)kv_rows; (void)num_rows; (void)indices; (void)bmm1_scale;
  (void)bmm2_scale; (void)out; (void)lse; (void)float_ws; (void)float_ws_bytes; (void)stream;
  set_error("run_mla_sparse: not built yet");
  return BSKV_ERR_UNSUPPORTED;
}
