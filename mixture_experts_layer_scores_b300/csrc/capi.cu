// Status codes, the per-device status word, and version.
#include <mutex>

#include "moe_internal.cuh"

// One status word per device (module-scope device variable; not a cudaMalloc).
static __device__ int g_moe_status = 0;

namespace moe {

int* device_status_word() {
  static std::mutex mu;
  static int* addr[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

}  // namespace moe

extern "C" const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_NAN_INPUT: return "MOE_ERR_NAN_INPUT";
  }
  return "MOE_ERR_UNKNOWN";
}

extern "C" moe_status_t moe_last_device_status(moe_stream_t stream) {
  int* w = moe::device_status_word();
  if (!w) return MOE_ERR_CUDA;
  cudaStream_t s = moe::as_cuda(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, w, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (host & moe::kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (host & (moe::kStatusBadExpertId | moe::kStatusBadToken)) return MOE_ERR_INVALID_ARG;
  if (host & moe::kStatusNonFiniteLogit) return MOE_ERR_NAN_INPUT;
  return MOE_OK;
}

extern "C" int moe_version(void) { return 100; }
