// Router-weight gradient, binned and padded
// ("Build Triton-Ascend Binned MoE Routing": Goal, Workflow step 6,
//  Guardrails "accumulate wgrad reductions in float32";
//  "Build Triton-Ascend Padded MoE Routing": Workflow step 6, Guardrails on
//  unique assignment ids and reductions across column tiles).
//
// Source-major: one warp owns one sorted position i at a time. When i is
// kept it streams the expert row and the gradient row of token
// indices[i] / TOP_K, and forms their dot product in fp32 with compensated
// summation (Ogita, Rump and Oishi, "Accurate Sum and Dot Product", SIAM J.
// Sci. Comput. 26(6), 2005, algorithm Dot2): every product and every partial
// sum carries its exact rounding error (TwoProduct via fma, Knuth's TwoSum),
// the errors are summed separately and added once at the end, and the warp
// reduction combines (sum, error) pairs the same way. For bf16 rows the
// products are exact and the running sums use packed f32x2 instructions, two
// independent compensated sums per register. The result is as
// accurate as a dot computed in twice the working precision and then
// rounded, independent of H. A dropped position writes 0. Every wgrad entry
// is written by exactly one warp because indices is a permutation.
#include "common.cuh"
#include "vec_math.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

struct WgradArgs {
  const char* xe;
  const char* grad;
  float* wgrad;
  const int32_t* indices;
  const int32_t* bin_ids;
  const int32_t* bins;
  const int32_t* padded_bins;  // nullptr: binned
  int64_t T;
  int64_t n;
  int64_t vecs;
  int64_t xe_rows;
  int32_t E;
  int32_t capacity;
  int32_t top_k;
  int32_t* status;
};

// Running compensated sum: value s plus accumulated rounding errors c.
struct Acc2 {
  float s = 0.0f, c = 0.0f;
  // Adds x * y. EXACT_PRODUCTS: the fp32 product is exact (bf16 operands).
  template <bool EXACT_PRODUCTS>
  __device__ __forceinline__ void add_product(float x, float y) {
    const float p = __fmul_rn(x, y);
    float e;
    two_sum(s, p, s, e);
    if (EXACT_PRODUCTS) {
      c = __fadd_rn(c, e);
    } else {
      const float pe = __fmaf_rn(x, y, -p);  // exact error of the product
      c = __fadd_rn(c, __fadd_rn(e, pe));
    }
  }
  __device__ __forceinline__ void merge(float s2, float c2) {
    float e;
    two_sum(s, s2, s, e);
    c = __fadd_rn(__fadd_rn(c, c2), e);
  }
};

// Two running compensated sums in the halves of packed f32x2 registers.
// Used for bf16 rows, whose products are exact in fp32 (8-bit x 8-bit
// significands), so only the sums carry rounding errors.
struct Acc2x2 {
  uint64_t s = 0ull, c = 0ull;
  __device__ __forceinline__ void add_exact(uint64_t p) {
    const uint64_t t = f2_add(s, p);
    const uint64_t bb = f2_sub(t, s);
    const uint64_t e = f2_add(f2_sub(s, f2_sub(t, bb)), f2_sub(p, bb));
    s = t;
    c = f2_add(c, e);
  }
  __device__ __forceinline__ void fold_into(Acc2& a) const {
    float s0, s1, c0, c1;
    f2_unpack(s, s0, s1);
    f2_unpack(c, c0, c1);
    a.merge(s0, c0);
    a.merge(s1, c1);
  }
};

template <int VB, int U, typename ET, bool PADDED>
__global__ void __launch_bounds__(kThreads) wgrad_kernel(WgradArgs g) {
  using L = Lanes<VB, ET>;
  using V = typename L::V;
  constexpr int NE = L::kElems;
  constexpr bool kExact = Elem<ET>::kBytes == 2;  // bf16 x bf16 fits in fp32
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  const V* __restrict__ xe = reinterpret_cast<const V*>(g.xe);
  const V* __restrict__ gr = reinterpret_cast<const V*>(g.grad);

  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; i < g.n; i += warps) {
    const int32_t a = __ldg(g.indices + i);
    if (a < 0 || a >= g.n) {
      if (lane == 0) flag_status(g.status, MOE_STATUS_BAD_INDEX);
      continue;
    }
    const int32_t e = __ldg(g.bin_ids + i);
    int64_t row = -1;
    if (e < 0 || e >= g.E) {
      if (lane == 0) flag_status(g.status, MOE_STATUS_BAD_EXPERT);
    } else {
      const int64_t start = e > 0 ? __ldg(g.bins + e - 1) : 0;
      const int64_t j = i - start;
      if (j < 0 || i >= __ldg(g.bins + e)) {
        if (lane == 0) flag_status(g.status, MOE_STATUS_BAD_BINS);
      } else if (!PADDED) {
        if (j < g.capacity) row = (int64_t)e * g.capacity + j;
      } else {
        row = (e > 0 ? __ldg(g.padded_bins + e - 1) : 0) + j;
      }
      if (row >= g.xe_rows) {
        if (lane == 0) flag_status(g.status, MOE_STATUS_BAD_BINS);
        row = -1;
      }
    }
    if (row < 0) {
      if (lane == 0) g.wgrad[a] = 0.0f;
      continue;
    }
    const V* xr = xe + row * g.vecs;
    const V* gv = gr + (int64_t)(a / g.top_k) * g.vecs;
    constexpr bool kPacked = kExact && NE % 2 == 0;
    Acc2 acc[2];
    Acc2x2 acc2[2];
    for (int64_t c0 = 0; c0 < g.vecs; c0 += kWarp * U) {
      V vx[U], vg[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * kWarp + lane;
        if (c < g.vecs) {
          vx[u] = ld_once(xr + c);  // each expert row is read once
          vg[u] = ld_keep(gv + c);  // the token's gradient row, once per kept slot
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * kWarp + lane;
        if (c < g.vecs) {
          if constexpr (kPacked) {
#pragma unroll
            for (int p = 0; p < NE / 2; ++p)
              acc2[p & 1].add_exact(f2_mul(f2_elems<ET>(vx[u], p), f2_elems<ET>(vg[u], p)));
          } else {
#pragma unroll
            for (int q = 0; q < NE; ++q) acc[q & 1].template add_product<kExact>(L::get(vx[u], q), L::get(vg[u], q));
          }
        }
      }
    }
    if constexpr (kPacked) {
      acc2[0].fold_into(acc[0]);
      acc2[1].fold_into(acc[1]);
    }
    acc[0].merge(acc[1].s, acc[1].c);
#pragma unroll
    for (int d = kWarp / 2; d > 0; d >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, acc[0].s, d);
      const float c2 = __shfl_xor_sync(0xffffffffu, acc[0].c, d);
      acc[0].merge(s2, c2);
    }
    if (lane == 0) g.wgrad[a] = __fadd_rn(acc[0].s, acc[0].c);
  }
}

template <int VB, typename ET, bool PADDED>
int launch_wgrad(const WgradArgs& g, cudaStream_t s) {
  constexpr int U = VB == 32 ? 2 : (VB == 16 ? 4 : 8);  // 64 bytes per lane and operand in flight
  auto k = wgrad_kernel<VB, U, ET, PADDED>;
  const int64_t work_ctas = (g.n + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  k<<<persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s>>>(g);
  return check_launch();
}

template <bool PADDED>
int run_wgrad(WgradArgs g, int32_t dtype, cudaStream_t s) {
  const int eb = dtype_bytes(dtype);
  const int64_t row_bytes = g.vecs * eb;  // g.vecs holds H on entry
  const void* ptrs[] = {g.xe, g.grad};
  const int vb = pick_vec_bytes(row_bytes, ptrs, 2, eb, 32);
  if (vb == 0) return MOE_ERR_UNSUPPORTED;
  g.vecs = row_bytes / vb;
  if (dtype == MOE_F32) {
    switch (vb) {
      case 32: return launch_wgrad<32, float, PADDED>(g, s);
      case 16: return launch_wgrad<16, float, PADDED>(g, s);
      case 8: return launch_wgrad<8, float, PADDED>(g, s);
      default: return launch_wgrad<4, float, PADDED>(g, s);
    }
  }
  switch (vb) {
    case 32: return launch_wgrad<32, __nv_bfloat16, PADDED>(g, s);
    case 16: return launch_wgrad<16, __nv_bfloat16, PADDED>(g, s);
    case 8: return launch_wgrad<8, __nv_bfloat16, PADDED>(g, s);
    case 4: return launch_wgrad<4, __nv_bfloat16, PADDED>(g, s);
    default: return launch_wgrad<2, __nv_bfloat16, PADDED>(g, s);
  }
}

int wgrad_checks(const void* xe, const void* grad, int32_t dtype, const int32_t* indices, const int32_t* bin_ids,
                 const int32_t* bins, int64_t T, int64_t H, int32_t E, int32_t top_k, const float* wgrad,
                 int32_t* d_status) {
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || H < 0 || E < 1 || E > MOE_MAX_EXPERTS || top_k < 1 || top_k > MOE_MAX_TOP_K)
    return MOE_ERR_INVALID_ARG;
  if (T * top_k > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (bins == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (wgrad == nullptr || indices == nullptr || bin_ids == nullptr)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && H > 0 && grad == nullptr) return MOE_ERR_INVALID_ARG;
  const int eb = dtype_bytes(dtype);
  if ((xe && !aligned(xe, eb)) || (grad && !aligned(grad, eb))) return MOE_ERR_UNSUPPORTED;
  const void* p4[] = {indices, bin_ids, bins, wgrad, d_status};
  for (const void* p : p4)
    if (p != nullptr && !aligned(p, 4)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_binned_wgrad(const void* xe, const void* grad, int32_t dtype, const int32_t* indices,
                                const int32_t* bin_ids, const int32_t* bins, int64_t T, int64_t H, int32_t E,
                                int32_t capacity, int32_t top_k, float* wgrad, int32_t* d_status,
                                moe_stream_t stream) {
  const int rc = wgrad_checks(xe, grad, dtype, indices, bin_ids, bins, T, H, E, top_k, wgrad, d_status);
  if (rc != MOE_OK) return rc;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (xe == nullptr && capacity > 0 && H > 0) return MOE_ERR_INVALID_ARG;
  WgradArgs g{static_cast<const char*>(xe), static_cast<const char*>(grad), wgrad, indices, bin_ids, bins, nullptr,
              T, T * top_k, H, (int64_t)E * capacity, E, capacity, top_k, d_status};
  return run_wgrad<false>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_padded_wgrad(const void* xe, const void* grad, int32_t dtype, const int32_t* indices,
                                const int32_t* bin_ids, const int32_t* bins, const int32_t* padded_bins, int64_t T,
                                int64_t H, int32_t E, int32_t top_k, int64_t xe_rows, float* wgrad,
                                int32_t* d_status, moe_stream_t stream) {
  const int rc = wgrad_checks(xe, grad, dtype, indices, bin_ids, bins, T, H, E, top_k, wgrad, d_status);
  if (rc != MOE_OK) return rc;
  if (padded_bins == nullptr || xe_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(padded_bins, 4)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (xe == nullptr && xe_rows > 0 && H > 0) return MOE_ERR_INVALID_ARG;
  WgradArgs g{static_cast<const char*>(xe), static_cast<const char*>(grad), wgrad, indices, bin_ids, bins,
              padded_bins, T, T * top_k, H, xe_rows, E, 0, top_k, d_status};
  return run_wgrad<true>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}
