// Dense routing map -> fixed-width top-k compaction, and its backward
// (Megatron-Core API docs, core.transformer.moe.megakernel.mok.route_adapter:
//  RoutingMapToIndices forward / backward, routing_map_to_mok_inputs).
//
// Forward: one warp per token row. Each lane reads a few consecutive bytes
// of the int8 map (one vector load), __vcmpne4 turns them into a
// nonzero-byte mask, and a warp prefix sum of the per-lane counts gives
// each route its output slot in increasing expert order; the first topk are
// emitted with their probabilities and the rest of the row is padded with
// -1 / 0.0f.
// Rows of at most 64 experts with topk <= 8 take one thread per row instead
// (32 rows per warp in flight).
// Backward: for rows of at most 2048 experts in whole float4s, a warp builds
// a block of consecutive rows in shared memory and stores it with coalesced
// 16-byte stores; else one thread per 16
// dense columns when rows are whole 16-column chunks and topk <= 8 (the
// row's slots loaded once, four float4 stores of zeros, the slots stored
// over them);
// else one warp per row when the row is whole float4s (slots broadcast by
// shuffles, one float4 store per lane and 128-column chunk); other shapes
// take one thread per dense output, scanning the row's slots.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;



// Bit b of the result is set when byte b of w is nonzero.
__device__ __forceinline__ unsigned nonzero_bytes(uint32_t w) {
  const uint32_t m = __vcmpne4(w, 0u) & 0x80808080u;
  return ((m >> 7) | (m >> 14) | (m >> 21) | (m >> 28)) & 0xFu;
}

// Nonzero-byte mask of the C bytes of a map row a lane owns (C = 1, 2, 4,
// 8 or 16 with an aligned row; otherwise bytes one at a time).
template <int C>
__device__ __forceinline__ unsigned lane_route_mask(const int8_t* p, int valid) {
  if constexpr (C == 16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    return nonzero_bytes(v.x) | (nonzero_bytes(v.y) << 4) | (nonzero_bytes(v.z) << 8) | (nonzero_bytes(v.w) << 12);
  } else if constexpr (C == 8) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    return nonzero_bytes(v.x) | (nonzero_bytes(v.y) << 4);
  } else if constexpr (C == 4) {
    return nonzero_bytes(__ldg(reinterpret_cast<const uint32_t*>(p)));
  } else if constexpr (C == 2) {
    const uint32_t v = __ldg(reinterpret_cast<const uint16_t*>(p));
    return nonzero_bytes(v) & 0x3u;
  } else {
    unsigned m = 0;
    for (int b = 0; b < valid; ++b) m |= (__ldg(p + b) != 0 ? 1u : 0u) << b;
    return m;
  }
}

// One warp per token row. Lane l owns the C consecutive experts
// [base + l*C, base + (l+1)*C) of a 32*C-expert window; an exclusive warp
// prefix of the per-lane route counts gives every route its output slot, so
// routes are emitted in increasing expert order. Windows repeat until the
// row ends or topk routes are out; lanes then fill the remaining slots with
// -1 / 0.0f.
template <int C>
__global__ void __launch_bounds__(kThreads)
    compaction_fwd_kernel(const float* __restrict__ probs, const int8_t* __restrict__ rmap, int64_t T, int32_t E,
                          int32_t topk, float* __restrict__ probs_indices, int32_t* __restrict__ indices) {
  await_previous_kernel();
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
    const int8_t* row = rmap + t * E;
    const float* prow = probs + t * E;
    float* po = probs_indices + t * topk;
    int32_t* io = indices + t * topk;
    int emitted = 0;
    for (int base = 0; base < E && emitted < topk; base += kWarp * C) {
      const int first = base + lane * C;
      const int valid = min(C, E - first);
      unsigned mask = valid > 0 ? lane_route_mask<C>(row + first, valid) : 0u;
      const int cnt = __popc(mask);
      int excl = cnt;
#pragma unroll
      for (int d = 1; d < kWarp; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, excl, d);
        if (lane >= d) excl += v;
      }
      const int total = __shfl_sync(0xffffffffu, excl, kWarp - 1);
      int j = emitted + excl - cnt;
      while (mask != 0u && j < topk) {
        const int e = first + __ffs(mask) - 1;
        mask &= mask - 1u;
        io[j] = e;
        po[j] = __ldg(prow + e);
        ++j;
      }
      emitted += total;
    }
    for (int j = emitted + lane; j < topk; j += kWarp) {
      io[j] = -1;
      po[j] = 0.0f;
    }
  }
}

// Forward, one thread per token row, for maps of at most 64 experts in whole
// 16-byte vectors and topk <= 8 (the Qwen2-MoE-57B shape: E = 64, topk = 8):
// the row's NV map vectors give a 64-bit route mask, the first topk routes
// in increasing expert order are taken from it, and their probabilities are
// loaded together before the row's outputs are stored. A warp handles 32
// rows at once instead of one.
template <int NV>
__global__ void __launch_bounds__(kThreads)
    compaction_fwd_row_kernel(const float* __restrict__ probs, const int8_t* __restrict__ rmap, int64_t T, int32_t E,
                              int32_t topk, float* __restrict__ probs_indices, int32_t* __restrict__ indices,
                              bool vec_out) {
  await_previous_kernel();
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += (int64_t)gridDim.x * blockDim.x) {
    const uint4* mrow = reinterpret_cast<const uint4*>(rmap + t * E);
    uint64_t mask = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const uint4 w = __ldg(mrow + v);
      const uint64_t m16 = nonzero_bytes(w.x) | (nonzero_bytes(w.y) << 4) | (nonzero_bytes(w.z) << 8) |
                           (nonzero_bytes(w.w) << 12);
      mask |= m16 << (16 * v);
    }
    int32_t e[8];
    float p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      e[j] = -1;
      if (j < topk && mask != 0ull) {
        e[j] = __ffsll((long long)mask) - 1;
        mask &= mask - 1ull;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) p[j] = e[j] >= 0 ? __ldg(probs + t * E + e[j]) : 0.0f;
    float* po = probs_indices + t * topk;
    int32_t* io = indices + t * topk;
    if (vec_out) {  // topk == 8, rows 16-byte aligned
      reinterpret_cast<float4*>(po)[0] = make_float4(p[0], p[1], p[2], p[3]);
      reinterpret_cast<float4*>(po)[1] = make_float4(p[4], p[5], p[6], p[7]);
      reinterpret_cast<int4*>(io)[0] = make_int4(e[0], e[1], e[2], e[3]);
      reinterpret_cast<int4*>(io)[1] = make_int4(e[4], e[5], e[6], e[7]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < topk) {
          po[j] = p[j];
          io[j] = e[j];
        }
    }
  }
}

// Backward, one thread per 16 dense columns of a row (E a multiple of 16,
// 16-byte aligned output, topk <= 8): the row's compact slots are loaded
// once (the row's other threads hit L1), the 16 columns are zeroed with four
// float4 stores, and the slots that fall in them are stored over the zeros.
__global__ void __launch_bounds__(kThreads)
    compaction_bwd_chunk_kernel(const float* __restrict__ gpi, const int32_t* __restrict__ indices, int64_t T,
                                int32_t E, int32_t topk, float* __restrict__ grad_probs, int32_t* status) {
  await_previous_kernel();
  const int64_t chunks = E / 16;
  const int64_t total = T * chunks;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = q / chunks;
    const int c0 = (int)(q - t * chunks) * 16;
    int32_t e[8];
    float v[8];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      e[j] = -1;
      v[j] = 0.0f;
      if (j < topk) {
        e[j] = __ldg(indices + t * topk + j);
        v[j] = __ldg(gpi + t * topk + j);
        bad |= (e[j] < -1 || e[j] >= E);
      }
    }
    if (bad && c0 == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
    // zeros first, then the slots that land here in increasing slot order:
    // the same thread's later store wins, so a repeated index keeps the
    // highest slot
    float* row = grad_probs + t * E + c0;
    float4* dst = reinterpret_cast<float4*>(row);
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const unsigned d = (unsigned)(e[j] - c0);
      if (d < 16u) row[d] = v[j];
    }
  }
}

// Staged backward for rows of at most kStageFloats = 2048 experts in
// whole float4s: a warp takes R = min(32, 2048 / E) consecutive rows at a
// time (32 rows of the Qwen2-MoE-57B shape, E = 64; 8 of the DeepSeek-V3
// shape, E = 256). Their dense fp32 rows are one contiguous block of at
// most 8 KB, built in the warp's slice of shared memory (zeroed, then lane
// r < R stores row r's slots in increasing slot order, so a repeated index
// keeps the highest slot) and written to HBM with coalesced 16-byte stores
// (lane l takes chunks l, l+32, ...): every dense element is written once,
// as part of whole lines. (A staged forward, which loads the whole
// probability block in the same round as the map, measured slower than
// reading the routed entries directly: 10.2 vs 8.4 us at 65 536 x 64.)
constexpr int kStageWarps = 4;
constexpr int kStageThreads = kStageWarps * kWarp;
constexpr int kStageFloats = 2048;           // one warp's block: 8 KB
constexpr int kStageChunks = kStageFloats / 4;

__global__ void __launch_bounds__(kStageThreads)
    compaction_bwd_staged_kernel(const float* __restrict__ gpi, const int32_t* __restrict__ indices, int64_t T,
                                 int32_t E, int32_t topk, float* __restrict__ grad_probs, int32_t* status) {
  await_previous_kernel();
  __shared__ float4 stage[kStageWarps][kStageChunks];
  const int warp = threadIdx.x / kWarp, lane = lane_id();
  const int R = min(kWarp, kStageFloats / E);  // rows per block
  float4* blk = stage[warp];
  float* srow = reinterpret_cast<float*>(blk) + lane * E;
  for (int64_t t0 = ((int64_t)blockIdx.x * kStageWarps + warp) * R; t0 < T;
       t0 += (int64_t)gridDim.x * kStageWarps * R) {
    const int rows = (int)min((int64_t)R, T - t0);
    const int nchunk = rows * E / 4;
    int32_t e[8];
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      e[j] = -1;
      v[j] = 0.0f;
      if (j < topk && lane < rows) {
        e[j] = __ldg(indices + (t0 + lane) * topk + j);
        v[j] = __ldg(gpi + (t0 + lane) * topk + j);
      }
    }
#pragma unroll
    for (int u = 0; u < kStageChunks / kWarp; ++u) {
      const int c = u * kWarp + lane;
      if (c < nchunk) blk[c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if ((unsigned)e[j] < (unsigned)E) srow[e[j]] = v[j];
      else bad |= e[j] != -1;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
    __syncwarp();
    float4* dst = reinterpret_cast<float4*>(grad_probs + t0 * E);
#pragma unroll
    for (int u = 0; u < kStageChunks / kWarp; ++u) {
      const int c = u * kWarp + lane;
      if (c < nchunk) dst[c] = blk[c];
    }
    __syncwarp();  // the block is read before it is zeroed again
  }
}

// G = dense outputs per thread (4 with float4 stores, else 1).
template <int G>
__global__ void __launch_bounds__(kThreads)
    compaction_bwd_kernel(const float* __restrict__ gpi, const int32_t* __restrict__ indices, int64_t T, int32_t E,
                          int32_t topk, float* __restrict__ grad_probs, int32_t* status) {
  await_previous_kernel();
  const int64_t groups_per_row = E / G;
  const int64_t total = T * groups_per_row;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = q / groups_per_row;
    const int e0 = (int)(q - t * groups_per_row) * G;
    float o[G];
#pragma unroll
    for (int u = 0; u < G; ++u) o[u] = 0.0f;
    const int32_t* irow = indices + t * topk;
    const float* grow = gpi + t * topk;
    bool bad = false;
    for (int j = 0; j < topk; ++j) {
      const int32_t e = __ldg(irow + j);
      const unsigned d = (unsigned)(e - e0);
      if (d < (unsigned)G) {
#pragma unroll
        for (int u = 0; u < G; ++u)
          if (d == (unsigned)u) o[u] = __ldg(grow + j);
      }
      bad |= (e < -1 || e >= E);
    }
    if (bad && e0 == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
    if (G == 4) {
      *reinterpret_cast<float4*>(grad_probs + t * E + e0) = make_float4(o[0], o[G > 1 ? 1 : 0], o[G > 2 ? 2 : 0],
                                                                        o[G > 3 ? 3 : 0]);
    } else {
      grad_probs[t * E + e0] = o[0];
    }
  }
}

// Backward, one warp per row (E a multiple of 4, 16-byte aligned output):
// lane j holds compact slot k0 + j; the slots are broadcast in increasing j
// and each lane keeps the ones that fall in its four columns of the current
// 128-column chunk (a repeated index keeps the highest j), then stores them
// with one float4 store. Every dense element is written exactly once.
__global__ void __launch_bounds__(kThreads)
    compaction_bwd_warp_kernel(const float* __restrict__ gpi, const int32_t* __restrict__ indices, int64_t T,
                               int32_t E, int32_t topk, float* __restrict__ grad_probs, int32_t* status) {
  await_previous_kernel();
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
    const int32_t* irow = indices + t * topk;
    const float* grow = gpi + t * topk;
    float4* drow = reinterpret_cast<float4*>(grad_probs + t * E);
    bool bad = false;
    for (int c0 = 0; c0 < E; c0 += 4 * kWarp) {
      const int col = c0 + 4 * lane;  // first of this lane's four columns
      float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
      for (int k0 = 0; k0 < topk; k0 += kWarp) {
        const int nj = min(kWarp, topk - k0);
        int32_t e = -1;
        float v = 0.0f;
        if (lane < nj) {
          e = __ldg(irow + k0 + lane);
          v = __ldg(grow + k0 + lane);
          bad |= (e < -1 || e >= E);
        }
        for (int j = 0; j < nj; ++j) {
          const int32_t ej = __shfl_sync(0xffffffffu, e, j);
          const float vj = __shfl_sync(0xffffffffu, v, j);
          const unsigned d = (unsigned)(ej - col);
          if (d == 0u) o0 = vj;
          if (d == 1u) o1 = vj;
          if (d == 2u) o2 = vj;
          if (d == 3u) o3 = vj;
        }
      }
      if (col < E) drow[col / 4] = make_float4(o0, o1, o2, o3);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
  }
}

template <typename K>
int grid_for(K k, int64_t work) {
  return persistent_grid(k, kThreads, 0, (work + kThreads - 1) / kThreads);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_routing_map_to_indices_fwd(const float* probs, const int8_t* routing_map, int64_t T, int32_t E,
                                              int32_t topk, float* probs_indices, int32_t* indices,
                                              moe_stream_t stream) {
  if (T < 0 || E < 1 || topk < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (probs == nullptr || routing_map == nullptr || probs_indices == nullptr || indices == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(probs, 4) || !aligned(probs_indices, 4) || !aligned(indices, 4)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (E <= 64 && E % 16 == 0 && topk <= 8 && aligned(routing_map, 16)) {
    const bool vec_out = topk == 8 && aligned(probs_indices, 16) && aligned(indices, 16);
    const int64_t ctas = (T + kThreads - 1) / kThreads;
    auto run = [&](auto k) {
      launch(k, persistent_grid(k, kThreads, 0, ctas), kThreads, 0, s, probs, routing_map, T, E, topk, probs_indices,
             indices, vec_out);
    };
    switch (E / 16) {
      case 1: run(compaction_fwd_row_kernel<1>); break;
      case 2: run(compaction_fwd_row_kernel<2>); break;
      case 3: run(compaction_fwd_row_kernel<3>); break;
      default: run(compaction_fwd_row_kernel<4>);
    }
    return check_launch();
  }
  // Bytes per lane: the widest C in {16, 8, 4, 2} that divides E, keeps every
  // map row aligned to C and leaves at most half of the warp idle; else one
  // byte at a time.
  int C = 1;
  for (int c = 16; c >= 2; c >>= 1) {
    if (E % c == 0 && aligned(routing_map, c) && E >= kWarp * c / 2) {
      C = c;
      break;
    }
  }
  const int64_t work_ctas = (T + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  switch (C) {
    case 16: {
      auto k = compaction_fwd_kernel<16>;
      launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, probs, routing_map, T, E, topk,
                                                                          probs_indices, indices);
      break;
    }
    case 8: {
      auto k = compaction_fwd_kernel<8>;
      launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, probs, routing_map, T, E, topk,
                                                                          probs_indices, indices);
      break;
    }
    case 4: {
      auto k = compaction_fwd_kernel<4>;
      launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, probs, routing_map, T, E, topk,
                                                                          probs_indices, indices);
      break;
    }
    case 2: {
      auto k = compaction_fwd_kernel<2>;
      launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, probs, routing_map, T, E, topk,
                                                                          probs_indices, indices);
      break;
    }
    default: {
      auto k = compaction_fwd_kernel<1>;
      launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, probs, routing_map, T, E, topk,
                                                                          probs_indices, indices);
    }
  }
  return check_launch();
}

extern "C" int moe_routing_map_to_indices_bwd(const float* grad_probs_indices, const int32_t* indices, int64_t T,
                                              int32_t E, int32_t topk, float* grad_probs, int32_t* d_status,
                                              moe_stream_t stream) {
  if (T < 0 || E < 1 || topk < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (grad_probs_indices == nullptr || indices == nullptr || grad_probs == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(grad_probs_indices, 4) || !aligned(indices, 4) || !aligned(grad_probs, 4) ||
      (d_status && !aligned(d_status, 4)))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (E <= kStageFloats && E % 4 == 0 && topk <= 8 && aligned(grad_probs, 16)) {
    auto k = compaction_bwd_staged_kernel;
    const int64_t rows = kStageFloats / E < kWarp ? kStageFloats / E : kWarp;
    const int64_t ctas = (T + rows * kStageWarps - 1) / (rows * kStageWarps);
    launch(k, persistent_grid(k, kStageThreads, 0, ctas), kStageThreads, 0, s, grad_probs_indices, indices, T, E,
           topk, grad_probs, d_status);
  } else if (E % 16 == 0 && topk <= 8 && aligned(grad_probs, 16)) {
    auto k = compaction_bwd_chunk_kernel;
    launch(k, grid_for(k, T * (E / 16)), kThreads, 0, s, grad_probs_indices, indices, T, E, topk, grad_probs, d_status);
  } else if (E % 4 == 0 && aligned(grad_probs, 16)) {
    auto k = compaction_bwd_warp_kernel;
    launch(k, grid_for(k, T * kWarp), kThreads, 0, s, grad_probs_indices, indices, T, E, topk, grad_probs, d_status);
  } else {
    auto k = compaction_bwd_kernel<1>;
    launch(k, grid_for(k, T * E), kThreads, 0, s, grad_probs_indices, indices, T, E, topk, grad_probs, d_status);
  }
  return check_launch();
}
