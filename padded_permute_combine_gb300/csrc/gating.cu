// Router top-k gating: logits -> (top_expert, weights), the step before the
// route build ("Fused MoE Dispatch (Triton, universal)": pipeline "router
// scores -> top-k gating -> permute"; usage example gating="softmax" |
// "sigmoid").
//
// One warp per token. Lane l holds logits l, l + 32, l + 64, ... of the row
// (coalesced loads), NaN read as -inf. The top_k experts are picked in
// top_k rounds of a warp arg-max over the not-yet-chosen logits, ties to the
// lower expert id, so the choice is an exact fp32 comparison. Scores are the
// softmax over the whole row (max-subtracted, fp32 exp and sums) or the
// logistic sigmoid of the chosen logits; weights are the chosen scores,
// renormalised over the chosen experts when asked. Rows whose logits are all
// -inf (or whose chosen scores sum to 0) take the limit of equal logits: a
// uniform softmax and weights 1 / top_k.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// (value, expert) pairs compare by value, then by the lower expert id.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) { return v > bv || (v == bv && e < be); }

template <int NPL>
__global__ void __launch_bounds__(kThreads)
    gating_kernel(const float* __restrict__ logits, int64_t T, int32_t E, int32_t K, int32_t mode, int32_t normalize,
                  int32_t* __restrict__ top_expert, float* __restrict__ weights) {
  await_previous_kernel();
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
    const float* row = logits + t * E;
    float v[NPL];
    unsigned taken = 0;  // bit j: expert lane + 32 j is chosen or does not exist
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + kWarp * j;
      if (e < E) {
        const float x = __ldg(row + e);
        v[j] = isnan(x) ? -INFINITY : x;
      } else {
        v[j] = -INFINITY;
        taken |= 1u << j;
      }
    }
    // Softmax normaliser over the whole row.
    float m = -INFINITY, z = 0.0f;
    if (mode == MOE_GATING_SOFTMAX) {
#pragma unroll
      for (int j = 0; j < NPL; ++j)
        if (!(taken >> j & 1u)) m = fmaxf(m, v[j]);
#pragma unroll
      for (int d = kWarp / 2; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
      if (m != -INFINITY) {
#pragma unroll
        for (int j = 0; j < NPL; ++j)
          if (!(taken >> j & 1u)) z += expf(v[j] - m);
#pragma unroll
        for (int d = kWarp / 2; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      }
    }
    // top_k rounds of warp arg-max; lane k keeps selection k (and k + 32).
    int sel_e0 = -1, sel_e1 = -1;
    float sel_v0 = 0.0f, sel_v1 = 0.0f;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int e = lane + kWarp * j;
        if (!(taken >> j & 1u) && better(v[j], e, bv, be)) {
          bv = v[j];
          be = e;
        }
      }
#pragma unroll
      for (int d = kWarp / 2; d > 0; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
        const int oe = __shfl_xor_sync(0xffffffffu, be, d);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & (kWarp - 1)) == lane) taken |= 1u << (be / kWarp);
      if (k == lane) {
        sel_e0 = be;
        sel_v0 = bv;
      } else if (k == lane + kWarp) {
        sel_e1 = be;
        sel_v1 = bv;
      }
    }
    // Scores of the chosen experts, then the optional renormalisation.
    auto score = [&](float x) {
      if (mode == MOE_GATING_SOFTMAX) return m == -INFINITY ? 1.0f / (float)E : expf(x - m) / z;
      return 1.0f / (1.0f + expf(-x));
    };
    const float sc0 = sel_e0 >= 0 ? score(sel_v0) : 0.0f;
    const float sc1 = sel_e1 >= 0 ? score(sel_v1) : 0.0f;
    float chosen_sum = sc0 + sc1;
    if (normalize) {
#pragma unroll
      for (int d = kWarp / 2; d > 0; d >>= 1) chosen_sum += __shfl_xor_sync(0xffffffffu, chosen_sum, d);
    }
    auto emit = [&](int e, float sc, int k) {
      if (e < 0) return;
      const int64_t o = t * K + k;
      top_expert[o] = e;
      weights[o] = normalize ? (chosen_sum > 0.0f ? sc / chosen_sum : 1.0f / (float)K) : sc;
    };
    emit(sel_e0, sc0, lane);
    emit(sel_e1, sc1, lane + kWarp);
  }
}

template <int NPL>
int launch_gating(const float* logits, int64_t T, int32_t E, int32_t K, int32_t mode, int32_t normalize,
                  int32_t* top_expert, float* weights, cudaStream_t s) {
  auto k = gating_kernel<NPL>;
  const int64_t work_ctas = (T + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, logits, T, E, K, mode, normalize, top_expert,
                                                                      weights);
  return check_launch();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_topk_gating(const float* logits, int64_t T, int32_t E, int32_t top_k, int32_t mode,
                               int32_t normalize, int32_t* top_expert, float* weights, moe_stream_t stream) {
  if (T < 0 || E < 1 || top_k < 1 || top_k > E || top_k > MOE_MAX_TOP_K) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_GATING_SOFTMAX && mode != MOE_GATING_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (E > MOE_GATING_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
  if (T * (int64_t)top_k > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (logits == nullptr || top_expert == nullptr || weights == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(top_expert, 4) || !aligned(weights, 4)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (E <= 32) return launch_gating<1>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
  if (E <= 64) return launch_gating<2>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
  if (E <= 128) return launch_gating<4>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
  if (E <= 256) return launch_gating<8>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
  if (E <= 512) return launch_gating<16>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
  return launch_gating<32>(logits, T, E, top_k, mode, normalize, top_expert, weights, s);
}
