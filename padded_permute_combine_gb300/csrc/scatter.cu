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
// permutation `positions`; slots dropped by capacity are compacted away
// (ballot + __fns keeps slot order), and the loads of up to eight kept slots
// are issued before they are summed, to keep bytes in flight. For 16-byte
// rows with top_k <= 8 the chunks travel by cp.async into a per-warp
// shared-memory ring instead of registers (scatter_async_kernel), which lets
// more warps per SM keep more bytes in flight. Sums use Blackwell's packed
// f32x2 add, still rounding each operation to nearest, so the result is
// bit-identical to the scalar sequence.
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
  bool offsets32;  // every vector index of xe fits in 32 bits
  int32_t E;
  int32_t capacity;
  int32_t top_k;
  int32_t* status;
  const int32_t* indices = nullptr;  // checked against positions before a slot is followed
};

// Row of the expert tensor holding assignment a, or -1 when it was dropped.
// The positions entry is checked against indices (indices[positions[a]] must
// be a), so positions left over from another routing are flagged, never
// followed.
template <bool PADDED>
__device__ __forceinline__ int64_t slot_row(const ScatterArgs& g, int64_t a) {
  const int32_t i = __ldg(g.positions + a);
  if (i < 0 || i >= g.n) { flag_status(g.status, MOE_STATUS_BAD_INDEX); return -1; }
  const int32_t back = __ldg(g.indices + i);  // issued together with the bin_ids load
  const int32_t e = __ldg(g.bin_ids + i);
  if (back != a) { flag_status(g.status, MOE_STATUS_BAD_INDEX); return -1; }
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

// Adds the elements of one expert-row vector (scaled when WEIGHTED) to the
// accumulators, each 64-bit acc2 register holding a pair of fp32 sums. The
// scaling multiplies are scalar __fmul_rn, which is never merged into a
// fused multiply-add, so every term is rounded on its own before the
// (packed, round-to-nearest) add, exactly as in the scalar definition.
template <typename ET, typename V, int NP, bool WEIGHTED>
__device__ __forceinline__ void add_vec_packed(uint64_t (&acc2)[NP], const V& v, float w) {
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const uint64_t x2 = f2_elems<ET>(v, p);
    if (WEIGHTED) {
      float lo, hi;
      f2_unpack(x2, lo, hi);
      acc2[p] = f2_add(acc2[p], f2_pack(__float_as_uint(__fmul_rn(w, lo)), __float_as_uint(__fmul_rn(w, hi))));
    } else {
      acc2[p] = f2_add(acc2[p], x2);
    }
  }
}

template <int VB, typename ET, bool WEIGHTED>
__device__ __forceinline__ void add_vec_scalar(float (&acc)[Lanes<VB, ET>::kElems],
                                               const typename Lanes<VB, ET>::V& v, float w) {
#pragma unroll
  for (int e = 0; e < Lanes<VB, ET>::kElems; ++e) {
    const float x = Lanes<VB, ET>::get(v, e);
    acc[e] = WEIGHTED ? __fadd_rn(acc[e], __fmul_rn(w, x)) : __fadd_rn(acc[e], x);
  }
}

// Lane j receives the j-th kept slot (in slot order) of the 32 slots whose
// rows and weights the lanes hold; returns the number of kept slots.
__device__ __forceinline__ int compact_kept(int64_t& row, float& w) {
  const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
  const int nk = __popc(mask);
  const int lane = lane_id();
  const int src = lane < nk ? (int)__fns(mask, 0, lane + 1) : 0;
  const int64_t r = __shfl_sync(0xffffffffu, row, src);
  const float ww = __shfl_sync(0xffffffffu, w, src);
  row = lane < nk ? r : -1;
  w = ww;
  return nk;
}

// Sum of the nk kept rows' vectors held in v, stored at dst + c.
template <int KQ, int VB, typename ET, bool WEIGHTED>
__device__ __forceinline__ void sum_store(const typename Lanes<VB, ET>::V (&v)[KQ], const float (&w)[8], int nk,
                                          typename Lanes<VB, ET>::V* dst) {
  using L = Lanes<VB, ET>;
  using V = typename L::V;
  constexpr int NE = L::kElems;
  constexpr bool kPacked = (NE % 2) == 0;
  constexpr int NP = kPacked ? NE / 2 : 1;
  float acc[NE];
  if constexpr (kPacked) {
    uint64_t acc2[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) acc2[p] = 0ull;
#pragma unroll
    for (int q = 0; q < KQ; ++q)
      if (q < nk) add_vec_packed<ET, V, NP, WEIGHTED>(acc2, v[q], w[q]);
#pragma unroll
    for (int p = 0; p < NP; ++p) f2_unpack(acc2[p], acc[2 * p], acc[2 * p + 1]);
  } else {
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int q = 0; q < KQ; ++q)
      if (q < nk) add_vec_scalar<VB, ET, WEIGHTED>(acc, v[q], w[q]);
  }
  st_stream(dst, L::pack(acc));
}

// Streams columns [c_begin, c_end) of one output row from nk (<= KQ) kept
// expert rows held as 32-bit vector offsets, one warp-wide chunk per pass.
// When the registers allow, the passes are software-pipelined over two
// buffers: the loads of the next chunk are issued before the current chunk
// is summed, so each lane keeps up to 2 * nk loads in flight.
template <int KQ, int VB, typename ET, bool WEIGHTED>
__device__ __forceinline__ void stream_kept(const typename Lanes<VB, ET>::V* __restrict__ xe,
                                            typename Lanes<VB, ET>::V* __restrict__ dst, const uint32_t (&off)[8],
                                            const float (&w)[8], int nk, int64_t c_begin, int64_t c_end, int lane) {
  using V = typename Lanes<VB, ET>::V;
  if constexpr (KQ * VB > 64) {
    // Eight wide rows already fill the register budget: no second buffer.
    for (int64_t c = c_begin + lane; c - lane < c_end; c += kWarp) {
      V a[KQ];
#pragma unroll
      for (int q = 0; q < KQ; ++q)
        if (q < nk && c < c_end) a[q] = ld_stream(xe + c + off[q]);
      if (c < c_end) sum_store<KQ, VB, ET, WEIGHTED>(a, w, nk, dst + c);
    }
    return;
  }
  V a[KQ], b[KQ];
  int64_t c = c_begin + lane;
#pragma unroll
  for (int q = 0; q < KQ; ++q)
    if (q < nk && c < c_end) a[q] = ld_stream(xe + c + off[q]);
  while (c - lane < c_end) {
    const int64_t cn = c + kWarp;
#pragma unroll
    for (int q = 0; q < KQ; ++q)
      if (q < nk && cn < c_end) b[q] = ld_stream(xe + cn + off[q]);
    if (c < c_end) sum_store<KQ, VB, ET, WEIGHTED>(a, w, nk, dst + c);
    c = cn;
    if (c - lane >= c_end) break;
    const int64_t cm = c + kWarp;
#pragma unroll
    for (int q = 0; q < KQ; ++q)
      if (q < nk && cm < c_end) a[q] = ld_stream(xe + cm + off[q]);
    if (c < c_end) sum_store<KQ, VB, ET, WEIGHTED>(b, w, nk, dst + c);
    c = cm;
  }
}

constexpr int kKeptInFlight = 8;  // kept slots whose loads are issued together
constexpr int kRareGroup = 4;     // slots per group when more than kKeptInFlight are kept
#ifndef MOE_SCATTER_MIN_BLOCKS
#define MOE_SCATTER_MIN_BLOCKS 2
#endif
constexpr int kMinBlocks = MOE_SCATTER_MIN_BLOCKS;  // CTAs per SM the register budget must allow
// Vectors per work item, at most (DeepSeek-V3 rows of 896 vectors: two
// items of 448; measured 128 / 256 / 448 / 896: binned 0.1020 / 0.0939 /
// 0.0923 / 0.0968 ms, padded 0.1730 / 0.1695 / 0.1675 / 0.1690 ms).
#ifndef MOE_SCATTER_SEG
#define MOE_SCATTER_SEG 448
#endif
constexpr int64_t kSegTarget = MOE_SCATTER_SEG;

template <int VB, typename ET, bool PADDED, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads, kMinBlocks) scatter_kernel(ScatterArgs g) {
  await_previous_kernel();
  using L = Lanes<VB, ET>;
  using V = typename L::V;
  constexpr int NE = L::kElems;
  constexpr int KR = kKeptInFlight;
  constexpr int KG = kRareGroup;
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
    // Lane k (and k + 32) resolves slot k of this token, then the kept slots
    // of each half are compacted to the low lanes, keeping slot order.
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
    int n_lo = compact_kept(row_lo, w_lo);
    int n_hi = g.top_k > kWarp ? compact_kept(row_hi, w_hi) : 0;
    if (n_hi > 0 && n_lo + n_hi <= kWarp) {
      // Append the kept upper-half slots after the lower-half ones.
      const int src = (lane - n_lo) & (kWarp - 1);
      const int64_t rh = __shfl_sync(0xffffffffu, row_hi, src);
      const float wh = __shfl_sync(0xffffffffu, w_hi, src);
      if (lane >= n_lo && lane < n_lo + n_hi) {
        row_lo = rh;
        w_lo = wh;
      }
      n_lo += n_hi;
      n_hi = 0;
    }
    V* dst = out + t * g.vecs;
    if (g.offsets32 && n_hi == 0 && n_lo <= KR) {
      // Common case: every kept row stays in registers (as a 32-bit vector
      // offset into xe) for the whole segment, and all their loads are in
      // flight together.
      uint32_t off0[KR];
      float w0[KR];
#pragma unroll
      for (int q = 0; q < KR; ++q) {
        const int64_t r = __shfl_sync(0xffffffffu, row_lo, q);
        off0[q] = (uint32_t)((r < 0 ? 0 : r) * g.vecs);
        w0[q] = __shfl_sync(0xffffffffu, w_lo, q);
      }
      if (n_lo > 4) stream_kept<8, VB, ET, WEIGHTED>(xe, dst, off0, w0, n_lo, c_begin, c_end, lane);
      else stream_kept<4, VB, ET, WEIGHTED>(xe, dst, off0, w0, n_lo, c_begin, c_end, lane);
    } else {
      // More than KR kept slots (large TOP_K): groups of KG, low half first,
      // rows fetched from the compacted lanes on every pass.
      for (int64_t c0 = c_begin; c0 < c_end; c0 += kWarp) {
        const int64_t c = c0 + lane;
        const bool in = c < c_end;
        float acc[NE];
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = 0.0f;
        for (int h = 0; h < 2; ++h) {
          const int nh = h == 0 ? n_lo : n_hi;
          for (int g0 = 0; g0 < nh; g0 += KG) {
            V v[KG];
            float wq[KG];
#pragma unroll
            for (int q = 0; q < KG; ++q) {
              const int64_t r = __shfl_sync(0xffffffffu, h == 0 ? row_lo : row_hi, (g0 + q) & (kWarp - 1));
              wq[q] = __shfl_sync(0xffffffffu, h == 0 ? w_lo : w_hi, (g0 + q) & (kWarp - 1));
              if (g0 + q < nh && in) v[q] = ld_stream(xe + r * g.vecs + c);
            }
#pragma unroll
            for (int q = 0; q < KG; ++q)
              if (g0 + q < nh && in) add_vec_scalar<VB, ET, WEIGHTED>(acc, v[q], wq[q]);
          }
        }
        if (in) st_stream(dst + c, L::pack(acc));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Asynchronous-copy variant (16-byte rows, 32-bit offsets, top_k <= 8): the
// kept rows' chunks are copied global -> shared with cp.async into a
// per-warp ring of kAsyncSlots 512-byte slots, so the bytes in flight do not
// occupy registers. A lane copies, and later reads back, only its own 16
// bytes of every slot, so the only synchronisation is the lane's own
// cp.async.wait_group. Chunks in flight per warp: kAsyncSlots / KQ, i.e.
// 8, 4 or 2 for at most 2, 4 or 8 kept rows.

constexpr int kAsyncThreads = 128;
constexpr int kAsyncWarps = kAsyncThreads / kWarp;
constexpr int kAsyncSlots = 16;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int KQ, typename ET, bool WEIGHTED>
__device__ __forceinline__ void stream_kept_async(const uint4* __restrict__ xe, uint4* __restrict__ dst, uint4* ring,
                                                  const uint32_t (&off)[8], const float (&w)[8], int nk,
                                                  int64_t c_begin, int64_t c_end, int lane) {
  constexpr int DC = kAsyncSlots / KQ;  // chunks in flight
  const int64_t nch = (c_end - c_begin + kWarp - 1) / kWarp;
  auto issue = [&](int64_t j) {
    const int64_t c = c_begin + j * kWarp + lane;
    if (j < nch && c < c_end) {
      uint4* slot = ring + (int)(j % DC) * KQ * kWarp + lane;
#pragma unroll
      for (int q = 0; q < KQ; ++q)
        if (q < nk) cp_async16(slot + q * kWarp, xe + c + off[q]);
    }
    cp_async_commit();  // possibly empty: keeps one group per chunk
  };
#pragma unroll
  for (int d = 0; d < DC - 1; ++d) issue(d);
  for (int64_t j = 0; j < nch; ++j) {
    issue(j + DC - 1);
    cp_async_wait<DC - 1>();  // this lane's copies of chunk j have landed
    const int64_t c = c_begin + j * kWarp + lane;
    if (c < c_end) {
      const uint4* slot = ring + (int)(j % DC) * KQ * kWarp + lane;
      uint4 v[KQ];
#pragma unroll
      for (int q = 0; q < KQ; ++q)
        if (q < nk) v[q] = slot[q * kWarp];
      sum_store<KQ, 16, ET, WEIGHTED>(v, w, nk, dst + c);
    }
  }
  cp_async_wait<0>();
}

// Binned tokens keep few rows (2 to 5 of 8 at the DeepSeek-V3 batch), so
// more resident warps pay: the binned kernel is held to 80 registers (6 CTAs
// per SM); the padded one (8 rows per token) measured faster without the cap.
template <typename ET, bool PADDED, bool WEIGHTED>
__global__ void __launch_bounds__(kAsyncThreads, PADDED ? 1 : 6) scatter_async_kernel(ScatterArgs g) {
  await_previous_kernel();
  __shared__ uint4 ring_all[kAsyncWarps * kAsyncSlots * kWarp];
  const int lane = lane_id();
  uint4* ring = ring_all + (threadIdx.x / kWarp) * kAsyncSlots * kWarp;
  const int64_t warps = (int64_t)gridDim.x * kAsyncWarps;
  const int64_t items = g.T * g.segs;
  const uint4* __restrict__ xe = reinterpret_cast<const uint4*>(g.xe);
  uint4* __restrict__ out = reinterpret_cast<uint4*>(g.out);
  for (int64_t item = (int64_t)blockIdx.x * kAsyncWarps + threadIdx.x / kWarp; item < items; item += warps) {
    const int64_t t = item / g.segs;
    const int64_t c_begin = (item - t * g.segs) * g.seg_vecs;
    const int64_t c_end = min(c_begin + g.seg_vecs, g.vecs);
    int64_t row = -1;
    float wt = 1.0f;
    if (lane < g.top_k) {
      const int64_t a = t * g.top_k + lane;
      row = slot_row<PADDED>(g, a);
      if (WEIGHTED) wt = __ldg(g.weights + a);
    }
    const int nk = compact_kept(row, wt);
    uint32_t off[8];
    float w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int64_t r = __shfl_sync(0xffffffffu, row, q);
      off[q] = (uint32_t)((r < 0 ? 0 : r) * g.vecs);
      w[q] = __shfl_sync(0xffffffffu, wt, q);
    }
    uint4* dst = out + t * g.vecs;
    if (nk <= 2) stream_kept_async<2, ET, WEIGHTED>(xe, dst, ring, off, w, nk, c_begin, c_end, lane);
    else if (nk <= 4) stream_kept_async<4, ET, WEIGHTED>(xe, dst, ring, off, w, nk, c_begin, c_end, lane);
    else stream_kept_async<8, ET, WEIGHTED>(xe, dst, ring, off, w, nk, c_begin, c_end, lane);
  }
}

__global__ void invert_kernel(const int32_t* __restrict__ indices, int64_t n, int32_t* __restrict__ positions,
                              int32_t* status) {
  await_previous_kernel();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t a = __ldg(indices + i);
    if (a >= 0 && a < n) positions[a] = (int32_t)i;
    else flag_status(status, MOE_STATUS_BAD_INDEX);
  }
}

// Items per warp of the asynchronous scatter's grid (0: persistent grid).
// One: a CTA per four token segments, so the block scheduler gives the
// later CTAs to the SMs that finish first and tokens' uneven kept counts
// even out across SMs (DeepSeek-V3 batch, items of 224 vectors: binned
// 0.0966 -> 0.0938 ms, padded 0.1766 -> 0.1693; two items per warp
// 0.0942 / 0.1697).
#ifndef MOE_SCATTER_ITEMS
#define MOE_SCATTER_ITEMS 1
#endif

template <int VB, typename ET, bool PADDED>
int launch_scatter(ScatterArgs g, cudaStream_t s) {
  // Column segments of at most kSegTarget vectors, rounded to whole warp passes.
  g.segs = (g.vecs + kSegTarget - 1) / kSegTarget;
  g.seg_vecs = ((g.vecs + g.segs - 1) / g.segs + kWarp - 1) / kWarp * kWarp;
  g.segs = (g.vecs + g.seg_vecs - 1) / g.seg_vecs;
  g.offsets32 = (uint64_t)g.xe_rows * (uint64_t)g.vecs <= 0xffffffffull;
  if constexpr (VB == 16) {
    if (g.offsets32 && g.top_k <= kKeptInFlight) {
      const int64_t actas = (g.T * g.segs + kAsyncWarps - 1) / kAsyncWarps;
      if (g.weights != nullptr) {
        auto k = scatter_async_kernel<ET, PADDED, true>;
        launch(k, balanced_grid(k, kAsyncThreads, 0, actas, MOE_SCATTER_ITEMS), kAsyncThreads, 0, s, g);
      } else {
        auto k = scatter_async_kernel<ET, PADDED, false>;
        launch(k, balanced_grid(k, kAsyncThreads, 0, actas, MOE_SCATTER_ITEMS), kAsyncThreads, 0, s, g);
      }
      return check_launch();
    }
  }
  const int64_t work_ctas = (g.T * g.segs + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  if (g.weights != nullptr) {
    auto k = scatter_kernel<VB, ET, PADDED, true>;
    launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, g);
  } else {
    auto k = scatter_kernel<VB, ET, PADDED, false>;
    launch(k, persistent_grid(k, kThreads, 0, work_ctas), kThreads, 0, s, g);
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
  g.indices = indices;
  if (g.positions == nullptr && g.n > 0) {
    if (workspace == nullptr || ws_bytes < moe_scatter_workspace_size(g.n) || !aligned(workspace, 4))
      return MOE_ERR_INVALID_ARG;
    int32_t* pos = static_cast<int32_t*>(workspace);
    const int64_t blocks = (g.n + 255) / 256;
    launch(invert_kernel, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s, indices, g.n, pos, g.status);
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
                T, T * top_k, H, 0, 0, (int64_t)E * capacity, false, E, capacity, top_k, d_status};
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
                positions, T, T * top_k, H, 0, 0, xe_rows, false, E, 0, top_k, d_status};
  return run_scatter<true>(g, dtype, indices, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}
