// Device status word, error text and small host utilities of libbskv.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {

namespace {
thread_local char g_err[1024] = {0};

// Per device: [0] first error a kernel recorded, [1] testing hook "force timeout".
__device__ int g_status_words[2];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {nullptr};
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

const char* dtype_name(int32_t dt) {
  switch (dt) {
    case BSKV_FP16: return "fp16";
    case BSKV_BF16: return "bf16";
    case BSKV_FP32: return "fp32";
    case BSKV_E4M3: return "e4m3";
    case BSKV_INT32: return "int32";
    case BSKV_INT64: return "int64";
    default: return "unknown";
  }
}

bskv_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return BSKV_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return BSKV_ERR_CUDA;
}

// Device address of the status words of the current device (looked up once per device).
bskv_status status_args(dev::StatusArgs* out) {
  int d = 0;
  if (bskv_status s = cuda_check(cudaGetDevice(&d), "cudaGetDevice")) return s;
  if (d < 0 || d >= kMaxDevices) { set_error("device ordinal %d too large", d); return BSKV_ERR_UNSUPPORTED; }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[d]) {
    void* p = nullptr;
    if (bskv_status s = cuda_check(cudaGetSymbolAddress(&p, g_status_words), "cudaGetSymbolAddress"))
      return s;
    g_status_ptr[d] = static_cast<int*>(p);
  }
  out->status = g_status_ptr[d];
  out->force = g_status_ptr[d] + 1;
  return BSKV_OK;
}

}  // namespace bskv

using namespace bskv;

extern "C" int32_t bskv_version(void) { return 100; }

extern "C" const char* bskv_last_error_message(void) { return g_err; }

extern "C" bskv_status bskv_get_device_status(int32_t* status, int32_t reset) {
  if (!status) { set_error("get_device_status: NULL"); return BSKV_ERR_INVALID_ARG; }
  int v = 0;
  if (bskv_status s = cuda_check(cudaMemcpyFromSymbol(&v, g_status_words, sizeof(int), 0),
                                 "cudaMemcpyFromSymbol"))
    return s;
  *status = v;
  if (reset) {
    const int zero = 0;
    if (bskv_status s = cuda_check(cudaMemcpyToSymbol(g_status_words, &zero, sizeof(int), 0),
                                   "cudaMemcpyToSymbol"))
      return s;
  }
  return BSKV_OK;
}

extern "C" bskv_status bskv_set_debug_force_timeout(int32_t on) {
  const int v = on ? 1 : 0;
  return cuda_check(cudaMemcpyToSymbol(g_status_words, &v, sizeof(int), sizeof(int)),
                    "cudaMemcpyToSymbol");
}

extern "C" bskv_status bskv_plan_upload(bskv_plan* plan, void* int_ws, size_t int_ws_bytes,
                                        void* stream) {
  BSKV_NVTX_RANGE("bskv_plan_upload");
  if (!plan) { set_error("plan_upload: NULL plan"); return BSKV_ERR_INVALID_ARG; }
  const size_t meta_bytes = plan->meta.size() * sizeof(int32_t);
  const size_t cnt_off = merge_counter_offset(plan->meta.size());
  const size_t cnt_bytes = plan->counter_words * sizeof(int32_t);
  const size_t need = cnt_off + cnt_bytes;
  if (!int_ws || int_ws_bytes < need) {
    set_error("plan_upload: int workspace of %zu bytes, %zu needed", int_ws_bytes, need);
    return BSKV_ERR_WORKSPACE_TOO_SMALL;
  }
  if (reinterpret_cast<uintptr_t>(int_ws) % 16 != 0) {
    set_error("plan_upload: int workspace must be 16-byte aligned");
    return BSKV_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bskv_status s = cuda_check(cudaMemcpyAsync(int_ws, plan->meta.data(), meta_bytes,
                                                 cudaMemcpyHostToDevice, st),
                                 "plan_upload cudaMemcpyAsync"))
    return s;
  int32_t* counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(int_ws) + cnt_off);
  if (cnt_bytes) {
    if (bskv_status s = cuda_check(cudaMemsetAsync(counters, 0, cnt_bytes, st),
                                   "plan_upload cudaMemsetAsync"))
      return s;
  }
  plan->counters_dev = cnt_bytes ? counters : nullptr;
  plan->meta_dev = static_cast<const int32_t*>(int_ws);
  return BSKV_OK;
}
