// Binned and padded gather, the "permute" of the MoE layer
// ("Build Triton-Ascend Binned MoE Routing": Goal, Workflow step 3,
//  Implementation Pattern, Guardrails;
//  "Build Triton-Ascend Padded MoE Routing": Goal, Workflow steps 4-5,
//  Implementation Pattern, Guardrails).
//
// Every output row is produced exactly once, as a copy of its source token
// row or as zeros (unused capacity / padding), so no clearing pass is
// needed. Two schedules:
//  - token-major (the usual case, see "token-major path" below): one warp
//    reads a token row once and writes it to each of the token's kept
//    output rows, so x leaves HBM once instead of once per kept slot;
//  - destination-major (gather_kernel; tiny outputs, and the last few rows
//    of the token-major schedule when it has to build the positions in the
//    output's tail): one warp owns one output row, finds its
//    source assignment through bins and indices (a padded row finds its
//    expert by binary search over padded_bins) and streams the row; token
//    rows are loaded evict-last there, as up to TOP_K rows copy the same
//    token.
// Rows move as VB-byte vectors (256-bit loads and stores when the row and
// pointers allow) with U vectors per lane in flight; the bin vectors are
// staged in shared memory. The weighted variant (the gradient of the combine
// with respect to the expert rows, d row(a) = w[a] * dy[a / TOP_K]) scales
// each copied row by its assignment's weight on the way through.
#include "common.cuh"
#include "vec_math.cuh"
#include "bulk.cuh"

#include <atomic>
#include <type_traits>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kStageMax = 1024;  // experts whose bins are staged in shared memory

struct GatherArgs {
  const char* x;
  char* out;
  const int32_t* indices;
  const int32_t* bins;
  const int32_t* padded_bins;  // nullptr: binned
  const float* weights;        // weighted gather only: scale of each assignment
  int64_t n;
  int64_t rows_out;
  int64_t vecs;  // vectors per row
  int32_t E;
  int32_t capacity;
  int32_t top_k;
  int32_t* status;
  int64_t T = 0;
  int64_t row_begin = 0;              // first row the destination-major kernel writes
  const int32_t* positions = nullptr;  // token-major path: inverse of indices (the caller's, or in the tail of out)
  int64_t segs = 1;      // token-major path: work items per token (column segments of its row)
  int64_t seg_len = 0;   // vectors (register pass) or bytes (bulk-copy pass) per segment
};

// Assignment id whose token fills output row `row`, or -1 for a zero row.
template <bool PADDED>
__device__ __forceinline__ int64_t source_assignment(const GatherArgs& g, const int32_t* sb, const int32_t* spb,
                                                int64_t row) {
  int32_t e;
  int64_t j, seg_len = 0;
  if (!PADDED) {
    e = (int32_t)(row / g.capacity);
    j = row - (int64_t)e * g.capacity;
  } else {
    if (row >= spb[g.E - 1]) return -1;  // beyond the last padded segment
    // first expert whose inclusive padded end exceeds row
    int lo = 0, hi = g.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (spb[mid] > row) hi = mid; else lo = mid + 1;
    }
    e = lo;
    const int64_t pstart = e > 0 ? spb[e - 1] : 0;
    j = row - pstart;
    seg_len = (int64_t)spb[e] - pstart;
  }
  const int64_t start = e > 0 ? sb[e - 1] : 0;
  const int64_t count = (int64_t)sb[e] - start;
  if (count < 0 || (PADDED && (count > seg_len || j < 0))) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  if (j >= count) return -1;
  const int64_t i = start + j;
  if (i < 0 || i >= g.n) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  const int32_t a = __ldg(g.indices + i);
  if (a < 0 || a >= g.n) {
    flag_status(g.status, MOE_STATUS_BAD_INDEX);
    return -1;
  }
  return a;
}

// v scaled by w element-wise, each product rounded to nearest (fp32) and,
// for bf16 rows, rounded once more to bf16 (nearest even).
template <typename ET, typename V>
__device__ __forceinline__ V scale_vec(const V& v, float w) {
  if constexpr (sizeof(V) == 2) {
    const float x = __uint_as_float((uint32_t)v << 16);
    __nv_bfloat16 b = __float2bfloat16_rn(__fmul_rn(w, x));
    return *reinterpret_cast<uint16_t*>(&b);
  } else {
    V r;
#pragma unroll
    for (int q = 0; q < Words<V>::N; ++q) {
      const uint32_t word = Words<V>::get(v, q);
      if constexpr (Elem<ET>::kBytes == 4) {
        Words<V>::set(r, q, __float_as_uint(__fmul_rn(w, __uint_as_float(word))));
      } else {
        Words<V>::set(r, q, pack_bf16x2(__fmul_rn(w, __uint_as_float(word << 16)),
                                        __fmul_rn(w, __uint_as_float(word & 0xffff0000u))));
      }
    }
    return r;
  }
}

// ST = void: plain row copy; float / __nv_bfloat16: each row scaled by the
// weight of its assignment (the weighted gather).
template <int VB, int U, bool PADDED, typename ST>
__global__ void __launch_bounds__(kThreads) gather_kernel(GatherArgs g) {
  await_previous_kernel();
  constexpr bool kWeighted = !std::is_void<ST>::value;
  using V = typename Vec<VB>::T;
  __shared__ int32_t sbins[kStageMax];
  __shared__ int32_t spbins[PADDED ? kStageMax : 1];
  const bool staged = g.E <= kStageMax;
  if (staged) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      sbins[e] = __ldg(g.bins + e);
      if (PADDED) spbins[e] = __ldg(g.padded_bins + e);
    }
    __syncthreads();
  }
  const int32_t* sb = staged ? sbins : g.bins;
  const int32_t* spb = PADDED ? (staged ? spbins : g.padded_bins) : nullptr;
  if (PADDED && threadIdx.x == 0 && blockIdx.x == 0 && spb[g.E - 1] > g.rows_out)
    flag_status(g.status, MOE_STATUS_ROWS_MISMATCH);

  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  const V* __restrict__ x = reinterpret_cast<const V*>(g.x);
  V* __restrict__ out = reinterpret_cast<V*>(g.out);
  for (int64_t row = g.row_begin + (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
       row < g.rows_out; row += warps) {
    const int64_t a = source_assignment<PADDED>(g, sb, spb, row);
    V* dst = out + row * g.vecs;
    if (a >= 0) {
      const V* s = x + (a / g.top_k) * g.vecs;
      float w = 1.0f;
      if constexpr (kWeighted) w = __ldg(g.weights + a);
      for (int64_t c0 = 0; c0 < g.vecs; c0 += kWarp * U) {
        V v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + u * kWarp + lane;
          if (c < g.vecs) v[u] = ld_keep(s + c);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + u * kWarp + lane;
          if constexpr (kWeighted) {
            if (c < g.vecs) st_stream(dst + c, scale_vec<ST>(v[u], w));
          } else {
            if (c < g.vecs) st_stream(dst + c, v[u]);
          }
        }
      }
    } else {
      const V z = zero_vec<V>();
      for (int64_t c = lane; c < g.vecs; c += kWarp) st_stream(dst + c, z);
    }
  }
}

// ------------------------------------------------------- token-major path
//
// The gather reads each token row once. One warp per token resolves the
// token's TOP_K slots to output rows through the inverse permutation of
// indices (positions[a] = sorted position of assignment a, checked against
// indices before it is followed) and copies the token row to every kept
// row, and the same launch zero-fills the unused rows. The positions come
// from the caller (the route build writes them): one launch. Without them,
// when the output is larger than n int32 values (every realistic shape),
// (1) the inverse permutation is first written into the last bytes of `out`
// itself, so no workspace is needed, (2) the token pass runs on it, and
// (3) the few rows that overlap that borrowed tail are then produced
// destination-major by gather_kernel, overwriting it.

__global__ void positions_kernel(const int32_t* __restrict__ indices, int64_t n, int32_t* __restrict__ positions,
                                 int32_t* status) {
  await_previous_kernel();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t a = __ldg(indices + i);
    if (a >= 0 && a < n) positions[a] = (int32_t)i;
    else flag_status(status, MOE_STATUS_BAD_INDEX);
  }
}

// Output row of sorted position i, or -1 when capacity drops it (or the
// bins are inconsistent with it, which is flagged).
template <bool PADDED>
__device__ __forceinline__ int64_t position_row(const GatherArgs& g, const int32_t* sb, const int32_t* spb,
                                                int64_t i) {
  int lo = 0, hi = g.E - 1;  // first expert whose inclusive end exceeds i
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sb[mid] > i) hi = mid; else lo = mid + 1;
  }
  const int64_t start = lo > 0 ? sb[lo - 1] : 0;
  const int64_t j = i - start;
  if (sb[lo] <= i || j < 0) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  if (!PADDED) return j < g.capacity ? (int64_t)lo * g.capacity + j : -1;
  const int64_t pstart = lo > 0 ? spb[lo - 1] : 0;
  if (j >= (int64_t)spb[lo] - pstart) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  if (pstart + j >= g.rows_out) {
    flag_status(g.status, MOE_STATUS_ROWS_MISMATCH);
    return -1;
  }
  return pstart + j;
}

// Whether output row r receives no token (unused capacity or padding).
template <bool PADDED>
__device__ __forceinline__ bool is_zero_row(const GatherArgs& g, const int32_t* sb, const int32_t* spb, int64_t r) {
  int32_t e;
  int64_t j;
  if (!PADDED) {
    e = (int32_t)(r / g.capacity);
    j = r - (int64_t)e * g.capacity;
  } else {
    if (r >= spb[g.E - 1]) return true;
    int lo = 0, hi = g.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (spb[mid] > r) hi = mid; else lo = mid + 1;
    }
    e = lo;
    j = r - (e > 0 ? spb[e - 1] : 0);
  }
  return j >= (int64_t)sb[e] - (e > 0 ? sb[e - 1] : 0);
}

#ifndef MOE_GATHER_MINB
#define MOE_GATHER_MINB 4
#endif
template <int VB, int U, bool PADDED, typename ST>
__global__ void __launch_bounds__(kThreads, VB == 32 ? MOE_GATHER_MINB : 1)
gather_token_kernel(GatherArgs g) {
  await_previous_kernel();
  constexpr bool kWeighted = !std::is_void<ST>::value;
  constexpr int KQ = 8;  // kept slots whose rows are written per sweep of the token row
  constexpr unsigned kAll = 0xffffffffu;
  using V = typename Vec<VB>::T;
  __shared__ int32_t sbins[kStageMax];
  __shared__ int32_t spbins[PADDED ? kStageMax : 1];
  const bool staged = g.E <= kStageMax;
  if (staged) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      sbins[e] = __ldg(g.bins + e);
      if (PADDED) spbins[e] = __ldg(g.padded_bins + e);
    }
    __syncthreads();
  }
  const int32_t* sb = staged ? sbins : g.bins;
  const int32_t* spb = PADDED ? (staged ? spbins : g.padded_bins) : nullptr;
  if (blockIdx.x == 0) {
    // bins nondecreasing, ending at most at n; padded segments hold their counts
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      const int32_t prev = e > 0 ? sb[e - 1] : 0;
      bool ok = sb[e] >= prev && (e < g.E - 1 || sb[e] <= g.n);
      if (PADDED) ok = ok && (int64_t)spb[e] - (e > 0 ? spb[e - 1] : 0) >= (int64_t)sb[e] - prev;
      if (!ok) flag_status(g.status, MOE_STATUS_BAD_BINS);
    }
    if (PADDED && threadIdx.x == 0 && spb[g.E - 1] > g.rows_out) flag_status(g.status, MOE_STATUS_ROWS_MISMATCH);
  }

  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  const V* __restrict__ x = reinterpret_cast<const V*>(g.x);
  V* __restrict__ out = reinterpret_cast<V*>(g.out);
  const int64_t token_items = g.T * g.segs;
  const int64_t items = token_items + g.row_begin;  // token segments, then the rows this kernel may zero-fill
  for (int64_t item = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; item < items;
       item += warps) {
    if (item >= token_items) {
      const int64_t r = item - token_items;
      if (is_zero_row<PADDED>(g, sb, spb, r)) {
        V* dst = out + r * g.vecs;
        const V z = zero_vec<V>();
        for (int64_t c = lane; c < g.vecs; c += kWarp) st_stream(dst + c, z);
      }
      continue;
    }
    const int64_t t = item / g.segs;
    const int64_t c_begin = (item - t * g.segs) * g.seg_len;
    const int64_t c_end = min(c_begin + g.seg_len, g.vecs);
    const V* src = x + t * g.vecs;
    for (int k0 = 0; k0 < g.top_k; k0 += kWarp) {
      // lane k resolves slot k0 + k; rows in the borrowed tail are left to the last pass
      const int64_t a = t * g.top_k + k0 + lane;
      int64_t row = -1;
      float w = 1.0f;
      if (k0 + lane < g.top_k) {
        const int32_t i = __ldg(g.positions + a);
        if (i < 0 || i >= g.n || __ldg(g.indices + i) != a) {
          flag_status(g.status, MOE_STATUS_BAD_INDEX);
        } else {
          row = position_row<PADDED>(g, sb, spb, i);
          if (row >= g.row_begin) row = -1;
        }
        if (kWeighted && row >= 0) w = __ldg(g.weights + a);
      }
      const unsigned kept = __ballot_sync(kAll, row >= 0);
      const int nk = __popc(kept);
      const int from = lane < nk ? (int)__fns(kept, 0, lane + 1) : 0;
      const int64_t krow = __shfl_sync(kAll, row, from);  // lane q: row of the q-th kept slot
      const float kw = __shfl_sync(kAll, w, from);
      for (int q0 = 0; q0 < nk; q0 += KQ) {
        const int nq = min(KQ, nk - q0);
        V* dst[KQ];
        float wq[KQ];
#pragma unroll
        for (int q = 0; q < KQ; ++q) {
          const int64_t r = __shfl_sync(kAll, krow, (q0 + q) & (kWarp - 1));
          dst[q] = out + (q < nq ? r : 0) * g.vecs;
          wq[q] = __shfl_sync(kAll, kw, (q0 + q) & (kWarp - 1));
        }
        for (int64_t c0 = c_begin; c0 < c_end; c0 += kWarp * U) {
          V v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + u * kWarp + lane;
            if (c < c_end) v[u] = ld_stream(src + c);
          }
#pragma unroll
          for (int q = 0; q < KQ; ++q) {
            if (q < nq) {
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + u * kWarp + lane;
                if constexpr (kWeighted) {
                  if (c < c_end) st_stream(dst[q] + c, scale_vec<ST>(v[u], wq[q]));
                } else {
                  if (c < c_end) st_stream(dst[q] + c, v[u]);
                }
              }
            }
          }
        }
      }
    }
  }
}

// ------------------------------------------------- bulk-copy token pass (TMA)
//
// The plain gather's token pass with the Tensor Memory Accelerator doing
// the copies: per row chunk, lane 0 of a warp issues one bulk load of the
// token row chunk into shared memory (completion tracked by an mbarrier)
// and one bulk store of it to each kept output row; zero rows are bulk
// stores of a zeroed chunk (binned: by the same warps after their token
// segments; padded: by extra warps of the CTA that do nothing else). One instruction moves up to kTmaChunk bytes, so
// the load/store units are no longer the limit (the register path issues
// one 32-byte store per lane per vector and stalls on their queue). Each
// warp alternates two chunk buffers, so a chunk's load overlaps the
// previous chunk's stores. Every mbarrier wait is bounded: after kSpinLimit
// polls the warp sets MOE_STATUS_TIMEOUT, waits once more (bounded) for the
// load it issued, drains its stores and stops; the output of that launch is
// then undefined.

#ifndef MOE_GATHER_TMA
#define MOE_GATHER_TMA 1
#endif
#ifndef MOE_GATHER_SEGS
#define MOE_GATHER_SEGS 1  // column segments per token, register pass
#endif
#ifndef MOE_TMA_SEGS
#define MOE_TMA_SEGS 2  // column segments per token, bulk-copy pass (two items of a 14 KB row measured best)
#endif
#ifndef MOE_TMA_WARPS
#define MOE_TMA_WARPS 4
#endif
constexpr int kTmaWarps = MOE_TMA_WARPS;
// Padded outputs: 4 more warps per CTA only zero-fill the padding rows,
// concurrently with the copy warps (0.230 -> 0.224 ms at the DeepSeek-V3
// batch). Binned outputs measured faster with the copy warps zero-filling
// after their token segments (no extra warps).
constexpr int kPaddedZeroWarps = 4;  // 1 / 2 / 8 measured 0.256 / 0.222 / 0.229 ms vs 0.222
template <bool PADDED>
__host__ __device__ constexpr int zero_warps() { return PADDED ? kPaddedZeroWarps : 0; }
template <bool PADDED>
__host__ __device__ constexpr int tma_threads() { return (kTmaWarps + zero_warps<PADDED>()) * kWarp; }
#ifndef MOE_TMA_CHUNK
#define MOE_TMA_CHUNK 8192
#endif
constexpr int kTmaChunk = MOE_TMA_CHUNK;  // bytes per staged row chunk
constexpr size_t kTmaSmem = (size_t)kTmaChunk * (1 + 2 * kTmaWarps) + 16 * kTmaWarps;
// Items per copy warp of the bulk-copy gather's grid (0: persistent grid).
// The persistent grid measured faster: one item per warp (each CTA stages
// the bins and zeroes its chunk again) took binned 0.203 vs 0.177 ms,
// padded 0.266 vs 0.226 on the DeepSeek-V3 batch.
#ifndef MOE_GATHER_ITEMS
#define MOE_GATHER_ITEMS 0
#endif

template <bool PADDED>
__global__ void __launch_bounds__(tma_threads<PADDED>(), 1) gather_tma_kernel(GatherArgs g, int64_t row_bytes) {
  await_previous_kernel();
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ __align__(128) unsigned char tsm[];
  __shared__ int32_t sbins[kStageMax];
  __shared__ int32_t spbins[PADDED ? kStageMax : 1];
  const int warp = threadIdx.x / kWarp, lane = lane_id();
  unsigned char* zero = tsm;
  constexpr int kZeroWarps = zero_warps<PADDED>();
  const bool copier = warp < kTmaWarps;
  unsigned char* bufs = tsm + (size_t)kTmaChunk * (1 + 2 * (copier ? warp : 0));
  uint64_t* bars = reinterpret_cast<uint64_t*>(tsm + (size_t)kTmaChunk * (1 + 2 * kTmaWarps)) + 2 * (copier ? warp : 0);
  for (int q = threadIdx.x; q < kTmaChunk / 16; q += blockDim.x) reinterpret_cast<uint4*>(zero)[q] = make_uint4(0, 0, 0, 0);
  if (lane == 0 && copier) {
    mbar_init(smem_u32(bars));
    mbar_init(smem_u32(bars + 1));
  }
  const bool staged = g.E <= kStageMax;
  if (staged) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      sbins[e] = __ldg(g.bins + e);
      if (PADDED) spbins[e] = __ldg(g.padded_bins + e);
    }
  }
  fence_mbarrier_init();
  fence_async_shared();  // the zero chunk and the barriers, for the bulk-copy unit
  __syncthreads();
  const int32_t* sb = staged ? sbins : g.bins;
  const int32_t* spb = PADDED ? (staged ? spbins : g.padded_bins) : nullptr;
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      const int32_t prev = e > 0 ? sb[e - 1] : 0;
      bool ok = sb[e] >= prev && (e < g.E - 1 || sb[e] <= g.n);
      if (PADDED) ok = ok && (int64_t)spb[e] - (e > 0 ? spb[e - 1] : 0) >= (int64_t)sb[e] - prev;
      if (!ok) flag_status(g.status, MOE_STATUS_BAD_BINS);
    }
    if (PADDED && threadIdx.x == 0 && spb[g.E - 1] > g.rows_out) flag_status(g.status, MOE_STATUS_ROWS_MISMATCH);
  }

  if (kZeroWarps > 0 && !copier) {
    // Zero-fill warps: candidate rows below row_begin, strided over the
    // grid's zero warps, concurrently with the copy warps' token segments.
    const int64_t zwarps = (int64_t)gridDim.x * kZeroWarps;
    for (int64_t r = (int64_t)blockIdx.x * kZeroWarps + (warp - kTmaWarps); r < g.row_begin; r += zwarps) {
      if (lane == 0 && is_zero_row<PADDED>(g, sb, spb, r)) {
        for (int64_t off = 0; off < row_bytes; off += kTmaChunk)
          bulk_store(g.out + r * row_bytes + off, smem_u32(zero), (uint32_t)min((int64_t)kTmaChunk, row_bytes - off));
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();  // the stores have read the zero chunk
    return;
  }
  const int64_t warps = (int64_t)gridDim.x * kTmaWarps;
  const int64_t token_items = g.T * g.segs;
  // token segments, then (unless zero warps do them) the rows this kernel may zero-fill
  const int64_t items = token_items + (kZeroWarps > 0 ? 0 : g.row_begin);
  uint32_t parity = 0;                       // bit b: parity of buffer b's next completion
  int use = 0;                               // buffer of the next chunk
  bool ok = true;
  for (int64_t item = (int64_t)blockIdx.x * kTmaWarps + warp; item < items && ok; item += warps) {
    if (item >= token_items) {
      const int64_t r = item - token_items;
      if (lane == 0 && is_zero_row<PADDED>(g, sb, spb, r)) {
        for (int64_t off = 0; off < row_bytes; off += kTmaChunk)
          bulk_store(g.out + r * row_bytes + off, smem_u32(zero), (uint32_t)min((int64_t)kTmaChunk, row_bytes - off));
        bulk_commit();
      }
      continue;
    }
    const int64_t t = item / g.segs;
    const int64_t b_begin = (item - t * g.segs) * g.seg_len;
    const int64_t b_end = min(b_begin + g.seg_len, row_bytes);
    for (int k0 = 0; k0 < g.top_k && ok; k0 += kWarp) {
      const int64_t a = t * g.top_k + k0 + lane;
      int64_t row = -1;
      if (k0 + lane < g.top_k) {
        const int32_t i = __ldg(g.positions + a);
        if (i < 0 || i >= g.n || __ldg(g.indices + i) != a) {
          flag_status(g.status, MOE_STATUS_BAD_INDEX);
        } else {
          row = position_row<PADDED>(g, sb, spb, i);
          if (row >= g.row_begin) row = -1;
        }
      }
      const unsigned kept = __ballot_sync(kAll, row >= 0);
      const int nk = __popc(kept);
      if (nk == 0) continue;
      const int from = lane < nk ? (int)__fns(kept, 0, lane + 1) : 0;
      const int64_t krow = __shfl_sync(kAll, row, from);  // lane q: row of the q-th kept slot
      for (int64_t off = b_begin; off < b_end; off += kTmaChunk) {
        const uint32_t bytes = (uint32_t)min((int64_t)kTmaChunk, b_end - off);
        const uint32_t buf = smem_u32(bufs + (size_t)use * kTmaChunk);
        const uint32_t bar = smem_u32(bars + use);
        bool got = true;
        if (lane == 0) {
          bulk_wait_read_but_one();  // the stores that last read this buffer have finished
          bulk_load(buf, g.x + t * row_bytes + off, bytes, bar);
          const uint32_t ph = (parity >> use) & 1u;
          got = mbar_wait(bar, ph);
          // On a timeout, wait once more (bounded) so that the load does not
          // land in shared memory after the CTA has gone.
          if (!got) (void)mbar_wait(bar, ph);
          parity ^= 1u << use;
        }
        ok = __shfl_sync(kAll, (int)got, 0) != 0;
        if (!ok) break;
        for (int q = 0; q < nk; ++q) {
          const int64_t r = __shfl_sync(kAll, krow, q);
          if (lane == 0) bulk_store(g.out + r * row_bytes + off, buf, bytes);
        }
        if (lane == 0) bulk_commit();
        use ^= 1;
      }
    }
  }
  if (lane == 0) {
    if (!ok) flag_status(g.status, MOE_STATUS_TIMEOUT);
    bulk_wait_all();  // the stores have read shared memory and written the output
  }
}

// Launches the bulk-copy token pass; false when the rows or pointers do not
// meet the 16-byte rule of the bulk copies (the register path runs instead).
template <bool PADDED>
bool launch_gather_tma(const GatherArgs& g, int64_t row_bytes, cudaStream_t s, int* rc) {
  if (!MOE_GATHER_TMA || row_bytes % 16 != 0 || !aligned(g.x, 16) || !aligned(g.out, 16)) return false;
  auto k = gather_tma_kernel<PADDED>;
  // The dynamic shared-memory opt-in is per device; set it once per device
  // (concurrent callers may both set it, which is harmless).
  constexpr int kMaxDevices = 64;
  static std::atomic<int> configured[kMaxDevices];
  int dev = 0;
  (void)cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (!cached || configured[dev].load(std::memory_order_relaxed) == 0) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmaSmem) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (cached) configured[dev].store(1, std::memory_order_relaxed);
  }
  GatherArgs gt = g;
  gt.segs = MOE_TMA_SEGS;
  gt.seg_len = ((row_bytes + gt.segs - 1) / gt.segs + 15) / 16 * 16;  // bytes, 16-byte multiples
  gt.segs = (row_bytes + gt.seg_len - 1) / gt.seg_len;
  const int64_t work_ctas = (gt.T * gt.segs + gt.row_begin + kTmaWarps - 1) / kTmaWarps;
  launch(k, balanced_grid(k, tma_threads<PADDED>(), kTmaSmem, work_ctas, MOE_GATHER_ITEMS), tma_threads<PADDED>(),
         kTmaSmem, s, gt, row_bytes);
  *rc = check_launch();
  return true;
}

template <int VB, bool PADDED, typename ST>
int launch_gather(GatherArgs g, int64_t row_bytes, cudaStream_t s) {
  // 128 bytes per lane in flight; the weighted pass (a scale per kept row)
  // keeps 64 so that it fits 4 CTAs per SM without spilling: padded
  // DeepSeek-V3 batch 0.243 -> 0.229 ms (binned unchanged, 0.186 ms) against
  // 128 bytes at 2 CTAs per SM (128 registers).
  constexpr int U = VB == 32 ? (std::is_void<ST>::value ? 4 : 2) : (VB >= 8 ? 8 : 16);
  constexpr int kWarps = kThreads / kWarp;
  g.segs = MOE_GATHER_SEGS;
  g.seg_len = ((g.vecs + g.segs - 1) / g.segs + kWarp - 1) / kWarp * kWarp;  // vectors, whole warp passes
  g.segs = g.seg_len > 0 ? (g.vecs + g.seg_len - 1) / g.seg_len : 1;
  if (g.positions != nullptr) {
    // The caller's positions (from its route build): one token pass over every row.
    g.row_begin = g.rows_out;
    int rc = MOE_OK;
    if (std::is_void<ST>::value && launch_gather_tma<PADDED>(g, row_bytes, s, &rc)) return rc;
    auto kt = gather_token_kernel<VB, U, PADDED, ST>;
    launch(kt, persistent_grid(kt, kThreads, 0, (g.T * g.segs + g.row_begin + kWarps - 1) / kWarps), kThreads, 0, s, g);
    return check_launch();
  }
  // Borrow the last 4n bytes of the output (16-byte aligned) for the
  // positions when the rows before them are at least some of the output.
  const uint64_t total = (uint64_t)g.rows_out * (uint64_t)row_bytes;
  const uint64_t need = 4ull * (uint64_t)g.n;
  g.row_begin = 0;
  if (g.n > 0 && total >= need + 16 + (uint64_t)row_bytes) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(g.out);
    const uintptr_t p = (base + total - need) & ~(uintptr_t)15;
    g.positions = reinterpret_cast<const int32_t*>(p);
    g.row_begin = (int64_t)((p - base) / (uint64_t)row_bytes);  // rows wholly before the positions
    const int64_t blocks = (g.n + 255) / 256;
    launch(positions_kernel, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s, 
        g.indices, g.n, reinterpret_cast<int32_t*>(p), g.status);
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
    int rc = MOE_OK;
    if (!(std::is_void<ST>::value && launch_gather_tma<PADDED>(g, row_bytes, s, &rc))) {
      auto kt = gather_token_kernel<VB, U, PADDED, ST>;
      launch(kt, persistent_grid(kt, kThreads, 0, (g.T * g.segs + g.row_begin + kWarps - 1) / kWarps), kThreads, 0, s, g);
      rc = check_launch();
    }
    if (rc != MOE_OK) return MOE_ERR_CUDA;
  }
  auto k = gather_kernel<VB, U, PADDED, ST>;  // rows [row_begin, rows_out), destination-major
  launch(k, persistent_grid(k, kThreads, 0, (g.rows_out - g.row_begin + kWarps - 1) / kWarps), kThreads, 0, s, g);
  return check_launch();
}

template <bool PADDED, typename ST>
int dispatch_vec(GatherArgs g, int elem, cudaStream_t s) {
  const int64_t row_bytes = g.vecs * elem;  // g.vecs holds H on entry
  const void* ptrs[] = {g.x, g.out};
  const int vb = pick_vec_bytes(row_bytes, ptrs, 2, elem, 32);
  if (vb == 0) return MOE_ERR_UNSUPPORTED;
  g.vecs = row_bytes / vb;
  switch (vb) {
    case 32: return launch_gather<32, PADDED, ST>(g, row_bytes, s);
    case 16: return launch_gather<16, PADDED, ST>(g, row_bytes, s);
    case 8: return launch_gather<8, PADDED, ST>(g, row_bytes, s);
    case 4: return launch_gather<4, PADDED, ST>(g, row_bytes, s);
    default:
      if constexpr (std::is_same<ST, float>::value) return MOE_ERR_UNSUPPORTED;  // fp32 rows are 4-byte multiples
      else return launch_gather<2, PADDED, ST>(g, row_bytes, s);
  }
}

template <bool PADDED>
int dispatch_gather(GatherArgs g, int32_t dtype, cudaStream_t s) {
  const int elem = dtype_bytes(dtype);
  if (g.weights == nullptr) return dispatch_vec<PADDED, void>(g, elem, s);
  if (dtype == MOE_F32) return dispatch_vec<PADDED, float>(g, elem, s);
  return dispatch_vec<PADDED, __nv_bfloat16>(g, elem, s);
}

int gather_checks(const void* x, int32_t dtype, const int32_t* indices, const int32_t* bins, int64_t T, int64_t H,
                  int32_t E, int32_t top_k, const void* out, int32_t* d_status) {
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || H < 0 || E < 1 || E > MOE_MAX_EXPERTS || top_k < 1 || top_k > MOE_MAX_TOP_K)
    return MOE_ERR_INVALID_ARG;
  if (T * top_k > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (bins == nullptr || (T > 0 && (x == nullptr || indices == nullptr))) return MOE_ERR_INVALID_ARG;
  const int eb = dtype_bytes(dtype);
  if ((x && !aligned(x, eb)) || (out && !aligned(out, eb))) return MOE_ERR_UNSUPPORTED;
  if (!aligned(indices, 4) || !aligned(bins, 4) || (d_status && !aligned(d_status, 4))) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_binned_gather(const void* x, int32_t dtype, const int32_t* indices, const int32_t* bins,
                                 const int32_t* positions, int64_t T, int64_t H, int32_t E, int32_t capacity,
                                 int32_t top_k, void* out, int32_t* d_status, moe_stream_t stream) {
  const int rc = gather_checks(x, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (positions != nullptr && !aligned(positions, 4)) return MOE_ERR_UNSUPPORTED;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)E * capacity;
  if (rows == 0 || H == 0) return MOE_OK;
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(x), static_cast<char*>(out), indices, bins, nullptr, nullptr, T * top_k,
               rows, H, E, capacity, top_k, d_status};
  g.T = T;
  g.positions = positions;
  return dispatch_gather<false>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_padded_gather(const void* x, int32_t dtype, const int32_t* indices, const int32_t* bins,
                                 const int32_t* padded_bins, const int32_t* positions, int64_t T, int64_t H,
                                 int32_t E, int32_t top_k, void* out, int64_t out_rows, int32_t* d_status,
                                 moe_stream_t stream) {
  const int rc = gather_checks(x, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (padded_bins == nullptr || out_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(padded_bins, 4) || (positions != nullptr && !aligned(positions, 4))) return MOE_ERR_UNSUPPORTED;
  if (out_rows == 0 || H == 0) return MOE_OK;
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(x), static_cast<char*>(out), indices, bins, padded_bins, nullptr, T * top_k,
               out_rows, H, E, 0, top_k, d_status};
  g.T = T;
  g.positions = positions;
  return dispatch_gather<true>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_binned_gather_weighted(const void* dy, int32_t dtype, const int32_t* indices, const int32_t* bins,
                                          const float* weights, const int32_t* positions, int64_t T, int64_t H,
                                          int32_t E, int32_t capacity, int32_t top_k, void* out, int32_t* d_status,
                                          moe_stream_t stream) {
  const int rc = gather_checks(dy, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  if ((weights != nullptr && !aligned(weights, 4)) || (positions != nullptr && !aligned(positions, 4)))
    return MOE_ERR_UNSUPPORTED;
  if (T > 0 && weights == nullptr) return MOE_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)E * capacity;
  if (rows == 0 || H == 0) return MOE_OK;
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(dy), static_cast<char*>(out), indices, bins, nullptr, weights, T * top_k,
               rows, H, E, capacity, top_k, d_status};
  g.T = T;
  g.positions = positions;
  return dispatch_gather<false>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_padded_gather_weighted(const void* dy, int32_t dtype, const int32_t* indices, const int32_t* bins,
                                          const int32_t* padded_bins, const float* weights,
                                          const int32_t* positions, int64_t T, int64_t H, int32_t E, int32_t top_k,
                                          void* out, int64_t out_rows, int32_t* d_status, moe_stream_t stream) {
  const int rc = gather_checks(dy, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (padded_bins == nullptr || out_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(padded_bins, 4) || (weights != nullptr && !aligned(weights, 4)) ||
      (positions != nullptr && !aligned(positions, 4)))
    return MOE_ERR_UNSUPPORTED;
  if (T > 0 && weights == nullptr) return MOE_ERR_INVALID_ARG;
  if (out_rows == 0 || H == 0) return MOE_OK;
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(dy), static_cast<char*>(out), indices, bins, padded_bins, weights,
               T * top_k, out_rows, H, E, 0, top_k, d_status};
  g.T = T;
  g.positions = positions;
  return dispatch_gather<true>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}

// Route build and gather in one call: the gather consumes the positions the
// route build writes, so it needs neither the inverse-permutation pass nor
// the borrowed output tail (route build's three launches + one token pass).
static int route_then_gather(const int32_t* top_expert, int32_t E, int32_t pad_multiple, int32_t* indices,
                             int32_t* bin_ids, int32_t* bins, int32_t* padded_bins, int32_t* positions,
                             void* workspace, size_t workspace_bytes, GatherArgs g, int32_t dtype, bool padded,
                             cudaStream_t s) {
  if (positions == nullptr || (padded && padded_bins == nullptr)) return MOE_ERR_INVALID_ARG;
  if (g.out == nullptr && g.rows_out > 0 && g.vecs > 0) return MOE_ERR_INVALID_ARG;
  const int rc = moe_route_build(top_expert, g.n, E, pad_multiple, indices, bin_ids, bins, padded_bins, positions,
                                 workspace, workspace_bytes, g.status, reinterpret_cast<moe_stream_t>(s));
  if (rc != MOE_OK || g.rows_out == 0 || g.vecs == 0) return rc;
  g.positions = positions;
  return padded ? dispatch_gather<true>(g, dtype, s) : dispatch_gather<false>(g, dtype, s);
}

extern "C" int moe_route_build_binned_gather(const int32_t* top_expert, const void* x, int32_t dtype, int64_t T,
                                             int64_t H, int32_t E, int32_t top_k, int32_t capacity,
                                             int32_t pad_multiple, int32_t* indices, int32_t* bin_ids,
                                             int32_t* bins, int32_t* padded_bins, int32_t* positions, void* out,
                                             void* workspace, size_t workspace_bytes, int32_t* d_status,
                                             moe_stream_t stream) {
  const int rc = gather_checks(x, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(x), static_cast<char*>(out), indices, bins, nullptr, nullptr, T * top_k,
               (int64_t)E * capacity, H, E, capacity, top_k, d_status};
  g.T = T;
  return route_then_gather(top_expert, E, pad_multiple, indices, bin_ids, bins, padded_bins, positions, workspace,
                           workspace_bytes, g, dtype, false, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int moe_route_build_padded_gather(const int32_t* top_expert, const void* x, int32_t dtype, int64_t T,
                                             int64_t H, int32_t E, int32_t top_k, int32_t pad_multiple,
                                             int32_t* indices, int32_t* bin_ids, int32_t* bins,
                                             int32_t* padded_bins, int32_t* positions, void* out, int64_t out_rows,
                                             void* workspace, size_t workspace_bytes, int32_t* d_status,
                                             moe_stream_t stream) {
  const int rc = gather_checks(x, dtype, indices, bins, T, H, E, top_k, out, d_status);
  if (rc != MOE_OK) return rc;
  if (out_rows < 0) return MOE_ERR_INVALID_ARG;
  GatherArgs g{static_cast<const char*>(x), static_cast<char*>(out), indices, bins, padded_bins, nullptr,
               T * top_k, out_rows, H, E, 0, top_k, d_status};
  g.T = T;
  return route_then_gather(top_expert, E, pad_multiple, indices, bin_ids, bins, padded_bins, positions, workspace,
                           workspace_bytes, g, dtype, true, reinterpret_cast<cudaStream_t>(stream));
}
