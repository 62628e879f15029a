// Routing check: the consistency of a routing's index vectors, as the
// routing pages require it of the gathers' and scatters' inputs
// ("Build Triton-Ascend Binned MoE Routing", Guardrails: bins monotonic,
//  bins[-1] equal to the number of assignments, bin_ids aligned with the bin
//  boundaries; "Build Triton-Ascend Padded MoE Routing", Guardrails: padded
//  segments no shorter than the real counts, and Workflow step 1:
//  assignments sorted by expert, in increasing id within an expert), plus
// positions as the inverse permutation of indices.
//
// One grid-stride pass: each thread tests its experts and its sorted
// positions against every condition (nothing stops early), the warp ORs its
// threads' bits and one lane ORs them into the status word.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    check_routing_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ bin_ids,
                         const int32_t* __restrict__ bins, const int32_t* __restrict__ padded_bins,
                         const int32_t* __restrict__ positions, int64_t n, int32_t E, int32_t* status) {
  await_previous_kernel();
  int bits = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t e = tid; e < E; e += stride) {
    const int64_t start = e > 0 ? __ldg(bins + e - 1) : 0;
    const int64_t end = __ldg(bins + e);
    if (end < start || (e == 0 && end < 0)) bits |= MOE_STATUS_BAD_BINS;
    if (padded_bins != nullptr) {
      const int64_t pstart = e > 0 ? __ldg(padded_bins + e - 1) : 0;
      const int64_t pend = __ldg(padded_bins + e);
      if (pend < pstart || pend - pstart < end - start) bits |= MOE_STATUS_BAD_BINS;
    }
    if (e == E - 1 && end != n) bits |= MOE_STATUS_BAD_BINS;
  }
  for (int64_t i = tid; i < n; i += stride) {
    const int32_t e = __ldg(bin_ids + i);
    if (e < 0 || e >= E) {
      bits |= MOE_STATUS_BAD_EXPERT;
    } else if (i < (e > 0 ? (int64_t)__ldg(bins + e - 1) : 0) || i >= __ldg(bins + e)) {
      bits |= MOE_STATUS_BAD_BINS;
    }
    const int32_t a = __ldg(indices + i);
    if (a < 0 || a >= n) {
      bits |= MOE_STATUS_BAD_INDEX;
    } else if (positions != nullptr && __ldg(positions + a) != i) {
      bits |= MOE_STATUS_BAD_INDEX;
    }
    if (i > 0 && e == __ldg(bin_ids + i - 1) && a <= __ldg(indices + i - 1)) bits |= MOE_STATUS_BAD_INDEX;
  }
  bits = (int)__reduce_or_sync(0xffffffffu, (unsigned)bits);
  if (lane_id() == 0 && bits != 0) atomicOr(status, bits);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_check_routing(const int32_t* indices, const int32_t* bin_ids, const int32_t* bins,
                                 const int32_t* padded_bins, const int32_t* positions, int64_t n, int32_t E,
                                 int32_t* d_status, moe_stream_t stream) {
  if (n < 0 || n > INT32_MAX || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (bins == nullptr || d_status == nullptr || (n > 0 && (indices == nullptr || bin_ids == nullptr)))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {indices, bin_ids, bins, padded_bins, positions, d_status};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, 4)) return MOE_ERR_UNSUPPORTED;
  const int64_t work = n > E ? n : E;
  auto k = check_routing_kernel;
  launch(k, persistent_grid(k, kThreads, 0, (work + kThreads - 1) / kThreads), kThreads, 0,
         reinterpret_cast<cudaStream_t>(stream), indices, bin_ids, bins, padded_bins, positions, n, E, d_status);
  return check_launch();
}
