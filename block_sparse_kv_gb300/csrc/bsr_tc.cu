// BSR block-sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {

bskv_status launch_bsr_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                               const void* k, const int64_t* ks, const void* v,
                               const int64_t* vs, void* out, const int64_t* os, float* lse,
                               float sm_scale, cudaStream_t st) {
  (void)plan; (void)q; (void)qs; (void)k; (void)ks; (void)v; (void)vs; (void)out; (void)os;
  (void)lse; (void)sm_scale; (void)st;
  set_error("run_bsr: tensor-core BSR kernel not built yet");
  return BSKV_ERR_UNSUPPORTED;
}

}  // namespace bskv
