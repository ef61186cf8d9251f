// pa_verify_run_static: verify attention for callers that cannot allocate
// device memory. Its scratch (device error word + split partials) is one
// file-scope device array of PA_STATIC_SCRATCH_BYTES that every GPU loading
// this library holds until exit. Host code reaches it through
// cudaGetSymbolAddress, once per device, with that device current.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/pa_verify.h"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
uint8_t* g_addr[kMaxDevices] = {};

}  // namespace

namespace pav {

// Device address of g_scratch on the current device (set up on first use).
int static_scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pav::report_error(PA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return pav::report_error(PA_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess || !ptr)
      return pav::report_error(PA_ERR_CUDA, (std::string("cudaGetSymbolAddress of the fixed scratch failed: ") +
                                             cudaGetErrorString(e)).c_str());
    g_addr[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_addr[dev];
  return PA_OK;
}

}  // namespace pav

extern "C" int pa_verify_run_static(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                                    const float* k_scale, const float* v_scale, const int32_t* block_table,
                                    const int32_t* context_lens, const int32_t* query_lens, float softmax_scale,
                                    void* out, pa_stream_t stream) {
  uint8_t* scratch = nullptr;
  const int rc = pav::static_scratch_address(&scratch);
  if (rc != PA_OK) return rc;
  return pav::enqueue_with_scratch(plan, q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, query_lens,
                                   softmax_scale, out, scratch, PA_STATIC_SCRATCH_BYTES,
                                   reinterpret_cast<cudaStream_t>(stream));
}
