// Host helpers shared by every entry point, and the informational calls.
#include <atomic>

#include "common.cuh"

namespace moe {

int num_sms() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    dev = 0;
  }
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    (void)cudaGetLastError();
    sms = 1;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

int check_launch() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace moe

extern "C" const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype or alignment";
    case MOE_ERR_CUDA: return "CUDA launch failure";
    default: return "unknown error";
  }
}

extern "C" int moe_version(void) { return 100; }
