// Route build for callers that cannot allocate device memory.
//
// moe_route_build needs a small device scratch buffer (per-chunk expert
// counts). Some callers have no way to provide one: a plain C host that was
// handed only its input and output buffers, a plugin that runs under a host
// framework which owns the whole device memory pool and exposes no allocator,
// or a latency-critical loop where a cudaMalloc call (which may synchronise
// the device) is not acceptable. For them, the scratch lives in a fixed
// file-scope device array that the library brings with it.
//
// The array is part of the library's device image: every GPU on which the
// library is loaded keeps these bytes reserved until the process exits. On
// each device, the first call looks up the array's device address with
// cudaGetSymbolAddress (host code cannot use the array's name as a device
// pointer) and caches it for the life of the process; a device reset, after
// which the array may live elsewhere, is not detected (the header says so).
#include <mutex>

#include "common.cuh"

static __device__ __align__(256) int32_t g_route_scratch[MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES / sizeof(int32_t)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of g_route_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_build_noalloc(const int32_t* top_expert, int64_t n, int32_t num_experts,
                                       int32_t pad_multiple, int32_t* indices, int32_t* bin_ids, int32_t* bins,
                                       int32_t* padded_bins, int32_t* positions, int32_t* d_status,
                                       moe_stream_t stream) {
  if (n < 0 || num_experts < 1 || num_experts > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_route_build_workspace_size(n, num_experts);
  if (need == 0 || need > MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  // The counts the kernels keep in the scratch are fully written before they
  // are read, so the previous call's contents need no clearing.
  return moe_route_build(top_expert, n, num_experts, pad_multiple, indices, bin_ids, bins, padded_bins, positions,
                         scratch, MOE_ROUTE_BUILD_NOALLOC_MAX_BYTES, d_status, stream);
}
