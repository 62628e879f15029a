// Binned and padded scatter, the weighted "combine" of the MoE layer
// ("Build Triton-Ascend Binned MoE Routing": Workflow step 5, Guardrails;
//  "Build Triton-Ascend Padded MoE Routing": Workflow step 6, Guardrails).
//
// Token-major: one warp owns a column segment of one output token row and
// reduces the token's TOP_K slots into fp32 registers in slot order
// k = 0..TOP_K-1, from +0.0, with round-to-nearest adds and multiplies (no
// FMA contraction), then rounds once to the output type. Because every
// assignment id is unique, each output element has exactly one writer and no
// atomics are needed. A slot finds its expert row through the inverse
// permutation `positions`; slots dropped by capacity are skipped. Loads of
// up to four slots are issued before they are summed, to keep bytes in
// flight.
#include "common.cuh"
#include "vec_math.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

struct ScatterArgs {
  const char* xe;
  char* out;
  const int32_t* bin_ids;
  const int32_t* bins;
  const int32_t* padded_bins;  // nullptr: binned
  const float* weights;        // nullptr: unweighted
  const int32_t* positions;
  int64_t T;
  int64_t n;
  int64_t vecs;      // vectors per row
  int64_t seg_vecs;  // vectors per work item
  int64_t segs;      // work items per token
  int64_t xe_rows;
  int32_t E;
  int32_t capacity;
  int32_t top_k;
  int32_t* status;
};

// Row of the expert tensor holding assignment a, or -1 when it was dropped.
template <bool PADDED>
__device__ __forceinline__ int64_t slot_row(const ScatterArgs& g, int64_t a) {
  const int32_t i = __ldg(g.positions + a);
  if (i < 0 || i >= g.n) { flag_status(g.status, MOE_STATUS_BAD_INDEX); return -1; }
  const int32_t e = __ldg(g.bin_ids + i);
  if (e < 0 || e >= g.E) { flag_status(g.status, MOE_STATUS_BAD_EXPERT); return -1; }
  const int64_t start = e > 0 ? __ldg(g.bins + e - 1) : 0;
  const int64_t j = i - start;
  if (j < 0 || i >= __ldg(g.bins + e)) { flag_status(g.status, MOE_STATUS_BAD_BINS); return -1; }
  int64_t row;
  if (!PADDED) {
    if (j >= g.capacity) return -1;
    row = (int64_t)e * g.capacity + j;
  } else {
    row = (e > 0 ? __ldg(g.padded_bins + e - 1) : 0) + j;
  }
  if (row < 0 || row >= g.xe_rows) { flag_status(g.status, MOE_STATUS_BAD_BINS); return -1; }
  return row;
}

template <int VB, int U, typename ET, bool PADDED, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads) scatter_kernel(ScatterArgs g) {
  using L = Lanes<VB, ET>;
  using V = typename L::V;
  constexpr int NE = L::kElems;
  constexpr int KG = 4;  // slots whose loads are in flight together
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  const int64_t items = g.T * g.segs;
  const V* __restrict__ xe = reinterpret_cast<const V*>(g.xe);
  V* __restrict__ out = reinterpret_cast<V*>(g.out);

  for (int64_t item = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; item < items;
       item += warps) {
    const int64_t t = item / g.segs;
    const int64_t c_begin = (item - t * g.segs) * g.seg_vecs;
    const int64_t c_end = min(c_begin + g.seg_vecs, g.vecs);
    // Lane k (and k + 32) resolves slot k of this token.
    int64_t row_lo = -1, row_hi = -1;
    float w_lo = 1.0f, w_hi = 1.0f;
    if (lane < g.top_k) {
      const int64_t a = t * g.top_k + lane;
      row_lo = slot_row<PADDED>(g, a);
      if (WEIGHTED) w_lo = __ldg(g.weights + a);
    }
    if (lane + kWarp < g.top_k) {
      const int64_t a = t * g.top_k + lane + kWarp;
      row_hi = slot_row<PADDED>(g, a);
      if (WEIGHTED) w_hi = __ldg(g.weights + a);
    }
    for (int64_t c0 = c_begin; c0 < c_end; c0 += kWarp * U) {
      float acc[U][NE];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < NE; ++q) acc[u][q] = 0.0f;
      for (int kb = 0; kb < g.top_k; kb += KG) {
        int64_t r[KG];
        float w[KG];
        V v[KG][U];
#pragma unroll
        for (int q = 0; q < KG; ++q) {
          const int k = kb + q;
          const bool hi = k >= kWarp;
          r[q] = __shfl_sync(0xffffffffu, hi ? row_hi : row_lo, k & (kWarp - 1));
          w[q] = __shfl_sync(0xffffffffu, hi ? w_hi : w_lo, k & (kWarp - 1));
          if (k >= g.top_k) r[q] = -1;
          if (r[q] >= 0) {
            const V* src = xe + r[q] * g.vecs;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int64_t c = c0 + u * kWarp + lane;
              if (c < c_end) v[q][u] = ld_stream(src + c);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < KG; ++q) {
          if (r[q] < 0) continue;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + u * kWarp + lane;
            if (c >= c_end) continue;
#pragma unroll
            for (int e = 0; e < NE; ++e) {
              const float x = L::get(v[q][u], e);
              acc[u][e] = WEIGHTED ? __fadd_rn(acc[u][e], __fmul_rn(w[q], x)) : __fadd_rn(acc[u][e], x);
            }
          }
        }
      }
      V* dst = out + t * g.vecs;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * kWarp + lane;
        if (c < c_end) st_stream(dst + c, L::pack(acc[u]));
      }
    }
  }
}

__global__ void invert_kernel(const int32_t* __restrict__ indices, int64_t n, int32_t* __restrict__ positions,
                              int32_t* status) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t a = __ldg(indices + i);
    if (a >= 0 && a < n) positions[a] = (int32_t)i;
    else flag_status(status, MOE_STATUS_BAD_INDEX);
  }
}

template <int VB, typename ET, bool PADDED>
int launch_scatter(ScatterArgs g, cudaStream_t s) {
  constexpr int U = (VB == 16) ? 2 : 4;
  g.seg_vecs = (int64_t)kWarp * U * 2;
  g.segs = (g.vecs + g.seg_vecs - 1) / g.seg_vecs;
  const int64_t work_ctas = (g.T * g.segs + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  if (g.weights != nullptr) {
    auto k = scatter_kernel<VB, U, ET, PADDED, true>;
    k<<<persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s>>>(g);
  } else {
    auto k = scatter_kernel<VB, U, ET, PADDED, false>;
    k<<<persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s>>>(g);
  }
  return check_launch();
}

template <bool PADDED>
int run_scatter(ScatterArgs g, int32_t dtype, const int32_t* indices, void* workspace, size_t ws_bytes,
                cudaStream_t s) {
  const int eb = dtype_bytes(dtype);
  const int64_t row_bytes = g.vecs * eb;  // g.vecs holds H on entry
  const void* ptrs[] = {g.xe, g.out};
  const int vb = pick_vec_bytes(row_bytes, ptrs, 2, eb);
  if (vb == 0) return MOE_ERR_UNSUPPORTED;
  g.vecs = row_bytes / vb;
  if (g.positions == nullptr && g.n > 0) {
    if (workspace == nullptr || ws_bytes < moe_scatter_workspace_size(g.n) || !aligned(workspace, 4))
      return MOE_ERR_INVALID_ARG;
    int32_t* pos = static_cast<int32_t*>(workspace);
    const int64_t blocks = (g.n + 255) / 256;
    invert_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(indices, g.n, pos, g.status);
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
    g.positions = pos;
  }
  if (dtype == MOE_F32) {
    switch (vb) {
      case 16: return launch_scatter<16, float, PADDED>(g, s);
      case 8: return launch_scatter<8, float, PADDED>(g, s);
      default: return launch_scatter<4, float, PADDED>(g, s);
    }
  }
  switch (vb) {
    case 16: return launch_scatter<16, __nv_bfloat16, PADDED>(g, s);
    case 8: return launch_scatter<8, __nv_bfloat16, PADDED>(g, s);
    case 4: return launch_scatter<4, __nv_bfloat16, PADDED>(g, s);
    default: return launch_scatter<2, __nv_bfloat16, PADDED>(g, s);
  }
}

int scatter_checks(const void* xe, int32_t dtype, const int32_t* indices, const int32_t* bin_ids,
                   const int32_t* bins, const float* weights, const int32_t* positions, int64_t T, int64_t H,
                   int32_t E, int32_t top_k, const void* out, int32_t* d_status) {
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || H < 0 || E < 1 || E > MOE_MAX_EXPERTS || top_k < 1 || top_k > MOE_MAX_TOP_K)
    return MOE_ERR_INVALID_ARG;
  if (T * top_k > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (bins == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && H > 0 && (out == nullptr || indices == nullptr || bin_ids == nullptr)) return MOE_ERR_INVALID_ARG;
  const int eb = dtype_bytes(dtype);
  if ((xe && !aligned(xe, eb)) || (out && !aligned(out, eb))) return MOE_ERR_UNSUPPORTED;
  const void* p4[] = {indices, bin_ids, bins, weights, positions, d_status};
  for (const void* p : p4)
    if (p != nullptr && !aligned(p, 4)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_scatter_workspace_size(int64_t n) {
  if (n < 0) return 0;
  return ((size_t)n * sizeof(int32_t) + 255) / 256 * 256;
}

extern "C" int moe_binned_scatter(const void* xe, int32_t dtype, const int32_t* indices, const int32_t* bin_ids,
                                  const int32_t* bins, const float* weights, const int32_t* positions, int64_t T,
                                  int64_t H, int32_t E, int32_t capacity, int32_t top_k, void* out,
                                  void* workspace, size_t workspace_bytes, int32_t* d_status,
                                  moe_stream_t stream) {
  const int rc = scatter_checks(xe, dtype, indices, bin_ids, bins, weights, positions, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0 || H == 0) return MOE_OK;
  if (xe == nullptr && capacity > 0) return MOE_ERR_INVALID_ARG;
  ScatterArgs g{static_cast<const char*>(xe), static_cast<char*>(out), bin_ids, bins, nullptr, weights, positions,
                T, T * top_k, H, 0, 0, (int64_t)E * capacity, E, capacity, top_k, d_status};
  return run_scatter<false>(g, dtype, indices, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_padded_scatter(const void* xe, int32_t dtype, const int32_t* indices, const int32_t* bin_ids,
                                  const int32_t* bins, const int32_t* padded_bins, const float* weights,
                                  const int32_t* positions, int64_t T, int64_t H, int32_t E, int32_t top_k,
                                  int64_t xe_rows, void* out, void* workspace, size_t workspace_bytes,
                                  int32_t* d_status, moe_stream_t stream) {
  const int rc = scatter_checks(xe, dtype, indices, bin_ids, bins, weights, positions, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (padded_bins == nullptr || xe_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(padded_bins, 4)) return MOE_ERR_UNSUPPORTED;
  if (T == 0 || H == 0) return MOE_OK;
  if (xe == nullptr && xe_rows > 0) return MOE_ERR_INVALID_ARG;
  ScatterArgs g{static_cast<const char*>(xe), static_cast<char*>(out), bin_ids, bins, padded_bins, weights,
                positions, T, T * top_k, H, 0, 0, xe_rows, E, 0, top_k, d_status};
  return run_scatter<true>(g, dtype, indices, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}
