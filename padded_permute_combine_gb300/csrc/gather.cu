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

// Routing data the token pass reads: FRESH = written earlier in the same
// launch by other CTAs (coherent loads through L2), else unchanged for the
// whole launch (read-only path).
template <bool FRESH>
__device__ __forceinline__ int32_t ld_route(const int32_t* p) {
  if constexpr (FRESH) return __ldcg(p);
  else return __ldg(p);
}

// The bulk-copy pass itself, after the caller has staged bins (and padded
// bins) in sb / spb (or points them at global memory): every thread of the
// CTA calls it. `tsm` is the kTmaSmem bytes of dynamic shared memory.
template <bool PADDED, bool FRESH>
__device__ __forceinline__ void tma_copy_pass(const GatherArgs& g, int64_t row_bytes, const int32_t* sb,
                                              const int32_t* spb, unsigned char* tsm) {
  constexpr unsigned kAll = 0xffffffffu;
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
  fence_mbarrier_init();
  fence_async_shared();  // the zero chunk and the barriers, for the bulk-copy unit
  __syncthreads();
  if (blockIdx.x == 0) {
    if (!FRESH) {  // bins computed in the same launch need no check
      for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
        const int32_t prev = e > 0 ? sb[e - 1] : 0;
        bool ok = sb[e] >= prev && (e < g.E - 1 || sb[e] <= g.n);
        if (PADDED) ok = ok && (int64_t)spb[e] - (e > 0 ? spb[e - 1] : 0) >= (int64_t)sb[e] - prev;
        if (!ok) flag_status(g.status, MOE_STATUS_BAD_BINS);
      }
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
        const int32_t i = ld_route<FRESH>(g.positions + a);
        if (i < 0 || i >= g.n || ld_route<FRESH>(g.indices + i) != a) {
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

template <bool PADDED>
__global__ void __launch_bounds__(tma_threads<PADDED>(), 1) gather_tma_kernel(GatherArgs g, int64_t row_bytes) {
  await_previous_kernel();
  extern __shared__ __align__(128) unsigned char tsm[];
  __shared__ int32_t sbins[kStageMax];
  __shared__ int32_t spbins[PADDED ? kStageMax : 1];
  const bool staged = g.E <= kStageMax;
  if (staged) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) {
      sbins[e] = __ldg(g.bins + e);
      if (PADDED) spbins[e] = __ldg(g.padded_bins + e);
    }
  }
  tma_copy_pass<PADDED, false>(g, row_bytes, staged ? sbins : g.bins,
                               PADDED ? (staged ? spbins : g.padded_bins) : nullptr, tsm);
}

// ------------------------------------- route build + bulk-copy gather, one launch
//
// One cooperative launch (every CTA resident at once) runs the route build
// and the gather's token pass, the phases separated by grid barriers:
//   A  CTA c counts the expert ids of its chunk of assignments (contiguous,
//      one sub-range per warp, per-warp counts kept in shared memory) and
//      writes them as row c of the count matrix;
//   B1 one warp per expert turns its column into an exclusive prefix over
//      the chunks and writes the expert's total;
//   B2 every CTA scans the totals over experts into bins and padded_bins
//      (CTA 0 writes them out; every CTA keeps them staged for C) and gives
//      each assignment of its chunk its stable sorted position (expert start
//      + the chunk prefix + the warp prefix + the rank among equal ids in a
//      warp round), writing indices, bin_ids and positions;
//   C  the bulk-copy token pass, reading those positions (coherent loads).
// The barrier counts CTA arrivals in one 64-bit word of the workspace whose
// upper 48 bits carry a per-call tag, so the word needs no initialisation
// (a stale value from an earlier call is re-tagged by the first arrival,
// and the last CTA to leave clears it, so a CUDA graph replaying the launch
// with the same tag starts from zero); each wait is bounded and a CTA that
// gives up sets MOE_STATUS_TIMEOUT and leaves, so every CTA ends. The caller opts in through the workspace size:
// at the DeepSeek-V3 shape, 16 to 8192 tokens, it measured slower than the
// route build's launches chained to the token pass (8192 tokens: binned
// 0.191 vs 0.185 ms, padded 0.236 vs 0.228; 16 tokens: 22.5 vs 17.9 us),
// each barrier costing 2-3 us across the grid, more than a chained launch.

struct RouteGatherArgs {
  const int32_t* top_expert;
  int32_t* indices;
  int32_t* bin_ids;
  int32_t* bins;
  int32_t* padded_bins;
  int32_t* positions;
  int32_t* counts;              // [grid][E] count matrix, then [E] totals
  unsigned long long* barrier;  // the barrier word
  unsigned long long tag;       // this call's tag (low 16 bits zero)
  int32_t m;                    // padding multiple
  int64_t chunk;                // assignments per CTA
  uint32_t slack = 0;           // added to every barrier's target (testing: makes the waits run out)
};

constexpr unsigned long long kTagMask = ~0xffffull;

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Arrival b (1, 2, 3) at the grid barrier of a launch of `grid` CTAs: waits
// (bounded) until every CTA of this call has arrived b times, plus `slack`
// (testing). The word's low 15 bits count arrivals; bit 15 marks a failed
// launch: a CTA that gives up sets it, so a later launch with the same tag
// (a CUDA graph replayed after a failure) cannot take the stale count for
// its own and stops too. An arrival that finds the count outside this
// barrier's window stops likewise. Stopping sets MOE_STATUS_TIMEOUT. Every
// thread of the CTA calls it; all get the result.
constexpr unsigned long long kFailedBit = 0x8000ull;
__device__ bool grid_barrier(const RouteGatherArgs& f, uint32_t b, uint32_t grid, int32_t* status) {
  __shared__ int passed;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's writes before its arrival
    bool arrived = false, in_window = false;
    for (int it = 0; it < 4096 && !arrived; ++it) {
      const unsigned long long cur = ld_acquire_u64(f.barrier);
      if ((cur & kTagMask) == f.tag) {
        const uint32_t before = (uint32_t)(atomicAdd(f.barrier, 1ull) & 0xffffull);
        in_window = before >= (b - 1) * grid && before < b * grid;  // the failed bit is outside every window
        arrived = true;
      } else if (atomicCAS(f.barrier, cur, f.tag | 1ull) == cur) {
        in_window = b == 1;  // first arrival of this call: the word is re-tagged
        arrived = true;
      }
    }
    bool ok = false;
    const uint32_t target = b * grid + f.slack;
    for (int it = 0; arrived && in_window && it < kSpinLimit; ++it) {
      const unsigned long long cur = ld_acquire_u64(f.barrier);
      if ((cur & kTagMask) != f.tag || (cur & kFailedBit)) break;
      if ((uint32_t)(cur & 0xffffull) >= target) {
        ok = true;
        break;
      }
      __nanosleep(64);
    }
    if (!ok) {
      flag_status(status, MOE_STATUS_TIMEOUT);
      if (arrived) atomicOr(f.barrier, kFailedBit);
    }
    __threadfence();
    passed = ok;
  }
  __syncthreads();
  return passed != 0;
}

// After the last barrier: the CTA whose departure completes the count
// clears the word, so that a later launch with the same tag (a CUDA graph
// replayed) starts from zero. Every CTA has passed the last barrier by then.
__device__ void grid_depart(const RouteGatherArgs& f, uint32_t barriers, uint32_t grid) {
  if (threadIdx.x == 0) {
    const unsigned long long before = atomicAdd(f.barrier, 1ull);
    if ((before & kTagMask) == f.tag && (uint32_t)(before & 0xffffull) == (barriers + 1) * grid - 1)
      atomicExch(f.barrier, 0ull);
  }
}

// Exclusive scan over experts of v[e] (in place) and of its rounding up to
// multiples of m (into pv); every thread of the CTA calls it.
__device__ void scan_experts(int64_t* v, int64_t* pv, int32_t E, int32_t m, int64_t (*wsum)[2]) {
  const int nt = blockDim.x, lane = lane_id(), warp = threadIdx.x / kWarp;
  const int per = (E + nt - 1) / nt;
  const int lo = min((int)threadIdx.x * per, (int)E), hi = min(lo + per, (int)E);
  int64_t s = 0, ps = 0;
  for (int e = lo; e < hi; ++e) {
    s += v[e];
    ps += (v[e] + m - 1) / m * m;
  }
  int64_t xs = s, xps = ps;  // inclusive over the warp's threads
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int64_t a = __shfl_up_sync(0xffffffffu, xs, d);
    const int64_t b = __shfl_up_sync(0xffffffffu, xps, d);
    if (lane >= d) {
      xs += a;
      xps += b;
    }
  }
  if (lane == kWarp - 1) {
    wsum[warp][0] = xs;
    wsum[warp][1] = xps;
  }
  __syncthreads();
  int64_t run = xs - s, prun = xps - ps;
  for (int w = 0; w < warp; ++w) {
    run += wsum[w][0];
    prun += wsum[w][1];
  }
  for (int e = lo; e < hi; ++e) {
    const int64_t c = v[e];
    v[e] = run;
    pv[e] = prun;
    run += c;
    prun += (c + m - 1) / m * m;
  }
  __syncthreads();
}

template <bool PADDED>
__global__ void __launch_bounds__(tma_threads<PADDED>(), 1)
    route_gather_kernel(GatherArgs g, int64_t row_bytes, RouteGatherArgs f) {
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kWarpsCta = tma_threads<PADDED>() / kWarp;
  extern __shared__ __align__(128) unsigned char tsm[];
  __shared__ int32_t sbins[kStageMax];
  __shared__ int32_t spbins[PADDED ? kStageMax : 1];
  __shared__ int64_t wsum[kWarpsCta][2];
  const int E = g.E;
  const int warp = threadIdx.x / kWarp, lane = lane_id();
  const int64_t G = gridDim.x;
  // Phases A and B use the bulk-copy buffers' shared memory:
  int32_t* whist = reinterpret_cast<int32_t*>(tsm);  // [warps][E]: counts, then running offsets
  int64_t* sstart = reinterpret_cast<int64_t*>(tsm + ((size_t)kWarpsCta * E * 4 + 7) / 8 * 8);  // [E]
  int64_t* spstart = sstart + E;                                                            // [E]
  int32_t* stotal = reinterpret_cast<int32_t*>(spstart + E);                                // [E]
  int32_t* spre = stotal + E;                                                               // [E]
  int32_t* totals = f.counts + G * E;

  // A: per-warp counts over contiguous sub-ranges of the chunk.
  const int64_t c0 = min((int64_t)blockIdx.x * f.chunk, g.n), c1 = min(c0 + f.chunk, g.n);
  const int64_t sub = (c1 - c0 + kWarpsCta - 1) / kWarpsCta;
  const int64_t s0 = min(c0 + warp * sub, c1), s1 = min(s0 + sub, c1);
  for (int q = threadIdx.x; q < kWarpsCta * E; q += blockDim.x) whist[q] = 0;
  __syncthreads();
  int32_t* mine = whist + warp * E;
  for (int64_t b = s0; b < s1; b += kWarp) {
    int32_t e = -1;
    if (b + lane < s1) {
      e = __ldg(f.top_expert + b + lane);
      if (e < 0 || e >= E) {
        flag_status(g.status, MOE_STATUS_BAD_EXPERT);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(kAll, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t c = 0;
    for (int w = 0; w < kWarpsCta; ++w) c += whist[w * E + e];
    f.counts[(int64_t)blockIdx.x * E + e] = c;
  }
  if (!grid_barrier(f, 1, (uint32_t)G, g.status)) return;

  // B1: a warp per expert: exclusive prefix of its column over the chunks,
  // kColPer chunks per lane loaded at once and held in registers.
  constexpr int kColPer = 16;
  for (int64_t e = (int64_t)blockIdx.x * kWarpsCta + warp; e < E; e += G * kWarpsCta) {
    int32_t carry = 0;
    for (int64_t q0 = 0; q0 < G; q0 += kWarp * kColPer) {
      const int64_t qb = q0 + (int64_t)lane * kColPer;
      int32_t v[kColPer];
      int32_t s = 0;
#pragma unroll
      for (int j = 0; j < kColPer; ++j) {
        v[j] = qb + j < G ? __ldcg(f.counts + (qb + j) * E + e) : 0;
        s += v[j];
      }
      int32_t x = s;  // inclusive over lanes
#pragma unroll
      for (int d = 1; d < kWarp; d <<= 1) {
        const int32_t y = __shfl_up_sync(kAll, x, d);
        if (lane >= d) x += y;
      }
      int32_t run = carry + x - s;
#pragma unroll
      for (int j = 0; j < kColPer; ++j) {
        if (qb + j < G) f.counts[(qb + j) * E + e] = run;
        run += v[j];
      }
      carry += __shfl_sync(kAll, x, kWarp - 1);
    }
    if (lane == 0) totals[e] = carry;
  }
  if (!grid_barrier(f, 2, (uint32_t)G, g.status)) return;

  // B2: bins from the totals, then this chunk's sorted positions.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int32_t t = __ldcg(totals + e);
    stotal[e] = t;
    sstart[e] = t;
    spre[e] = __ldcg(f.counts + (int64_t)blockIdx.x * E + e);
  }
  __syncthreads();
  scan_experts(sstart, spstart, E, f.m, wsum);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int32_t b = (int32_t)(sstart[e] + stotal[e]);
    const int32_t pb = (int32_t)(spstart[e] + ((int64_t)stotal[e] + f.m - 1) / f.m * f.m);
    sbins[e] = b;
    if (PADDED) spbins[e] = pb;
    if (blockIdx.x == 0) {
      f.bins[e] = b;
      if (f.padded_bins != nullptr) f.padded_bins[e] = pb;
    }
    int32_t run = (int32_t)sstart[e] + spre[e];
    for (int w = 0; w < kWarpsCta; ++w) {
      const int32_t c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = lanemask_lt();
  for (int64_t b = s0; b < s1; b += kWarp) {
    const int64_t a = b + lane;
    int32_t e = -1;
    if (a < s1) {
      e = __ldg(f.top_expert + a);
      if (e < 0 || e >= E) {
        e = -1;
        f.positions[a] = -1;  // left out of every output (already flagged)
      }
    }
    const unsigned peers = __match_any_sync(kAll, e);
    if (e >= 0) {
      const int32_t dst = mine[e] + __popc(peers & lt);
      if (dst >= 0 && dst < g.n) {
        f.indices[dst] = (int32_t)a;
        f.bin_ids[dst] = e;
        f.positions[a] = dst;
      } else {
        flag_status(g.status, MOE_STATUS_BAD_BINS);  // only on a broken barrier
        f.positions[a] = -1;
      }
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  if (!grid_barrier(f, 3, (uint32_t)G, g.status)) return;
  grid_depart(f, 3, (uint32_t)G);

  // C: the token pass over the positions just written.
  tma_copy_pass<PADDED, true>(g, row_bytes, sbins, PADDED ? spbins : nullptr, tsm);
}

// Sets the dynamic shared-memory opt-in of a bulk-copy kernel once per device
// (concurrent callers may both set it, which is harmless); false on failure.
template <typename Kernel>
bool allow_tma_smem(Kernel k, std::atomic<int>* configured, int n_devices) {
  int dev = 0;
  (void)cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < n_devices;
  if (cached && configured[dev].load(std::memory_order_relaxed) != 0) return true;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmaSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  if (cached) configured[dev].store(1, std::memory_order_relaxed);
  return true;
}

// CTAs of the one-launch route build + gather on this device (all resident
// at once), 0 when it cannot run here.
template <bool PADDED>
int64_t route_gather_grid() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> configured[kMaxDevices];
  auto k = route_gather_kernel<PADDED>;
  if (!allow_tma_smem(k, configured, kMaxDevices)) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, tma_threads<PADDED>(), kTmaSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const int64_t grid = (int64_t)per_sm * num_sms();
  return grid * 4 < (int64_t)kFailedBit ? grid : 0;  // three barriers' arrivals and the departures fit the count bits
}

// Workspace of the one-launch path: the [grid][E] count matrix and [E]
// totals (int32), then the 8-byte barrier word.
size_t route_gather_workspace(int64_t grid, int32_t E) {
  return ((size_t)(grid * E + E) * sizeof(int32_t) + 7) / 8 * 8 + 8;
}

std::atomic<unsigned long long> g_route_gather_calls{0};
std::atomic<uint32_t> g_barrier_slack{0};  // moe_test_barrier_slack

// Launches route build + bulk-copy gather as one cooperative kernel; false
// when it does not apply (rows or pointers off the bulk-copy rules, too many
// experts to stage, too small a workspace, or the launch refused), and the
// caller then takes the multi-launch path.
template <bool PADDED>
bool launch_route_gather(const GatherArgs& g, int64_t row_bytes, RouteGatherArgs f, void* workspace,
                         size_t workspace_bytes, cudaStream_t s, int* rc) {
  if (!MOE_GATHER_TMA || row_bytes % 16 != 0 || !aligned(g.x, 16) || !aligned(g.out, 16)) return false;
  if (g.E > kStageMax || g.n < 1 || g.rows_out < 1 || !aligned(workspace, 8)) return false;
  GatherArgs gt = g;
  gt.row_begin = gt.rows_out;
  gt.segs = MOE_TMA_SEGS;
  gt.seg_len = ((row_bytes + gt.segs - 1) / gt.segs + 15) / 16 * 16;  // bytes, 16-byte multiples
  gt.segs = (row_bytes + gt.seg_len - 1) / gt.seg_len;
  // As many CTAs as the token pass has work for (a copy warp per token
  // segment), at most all that fit at once and at least one per SM (the
  // zero rows, most of a small batch's padded output, need that many bulk-
  // store issuers): the grid barriers cost less on a smaller grid.
  const int64_t resident = route_gather_grid<PADDED>();
  const int64_t work = (gt.T * gt.segs + kTmaWarps - 1) / kTmaWarps;
  const int64_t grid = min(resident, max((int64_t)num_sms(), work));
  if (resident < 1 || workspace_bytes < route_gather_workspace(grid, g.E)) return false;
  f.counts = static_cast<int32_t*>(workspace);
  f.barrier = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) +
                                                    route_gather_workspace(grid, g.E) - 8);
  f.tag = ((g_route_gather_calls.fetch_add(1, std::memory_order_relaxed) + 1) & 0xffffffffffffull) << 16;
  f.chunk = (g.n + grid - 1) / grid;
  f.slack = g_barrier_slack.load(std::memory_order_relaxed);
  gt.positions = f.positions;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(tma_threads<PADDED>());
  cfg.dynamicSmemBytes = kTmaSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barriers end
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, route_gather_kernel<PADDED>, gt, row_bytes, f) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  *rc = MOE_OK;
  return true;
}

// Launches the bulk-copy token pass; false when the rows or pointers do not
// meet the 16-byte rule of the bulk copies (the register path runs instead).
template <bool PADDED>
bool launch_gather_tma(const GatherArgs& g, int64_t row_bytes, cudaStream_t s, int* rc) {
  if (!MOE_GATHER_TMA || row_bytes % 16 != 0 || !aligned(g.x, 16) || !aligned(g.out, 16)) return false;
  auto k = gather_tma_kernel<PADDED>;
  constexpr int kMaxDevices = 64;
  static std::atomic<int> configured[kMaxDevices];
  if (!allow_tma_smem(k, configured, kMaxDevices)) return false;
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
  // One launch when every host check of the route build passes and the
  // bulk-copy pass applies; otherwise the route build's launches and the
  // token pass (which also report any invalid argument).
  const void* rptrs[] = {top_expert, indices, bin_ids, bins, padded_bins, positions};
  bool route_ok = g.n > 0 && pad_multiple >= 1 && g.n + (int64_t)E * (pad_multiple - 1) <= INT32_MAX &&
                  top_expert != nullptr && indices != nullptr && bin_ids != nullptr && bins != nullptr &&
                  workspace != nullptr && workspace_bytes >= moe_route_build_workspace_size(g.n, E) &&
                  g.rows_out > 0 && g.vecs > 0 && (g.weights == nullptr);
  for (const void* p : rptrs) route_ok = route_ok && (p == nullptr || aligned(p, 4));
  if (route_ok) {
    const int64_t row_bytes = g.vecs * dtype_bytes(dtype);  // g.vecs holds H here
    RouteGatherArgs f{top_expert, indices, bin_ids, bins, padded_bins, positions, nullptr, nullptr, 0, pad_multiple, 0};
    int rc = MOE_OK;
    if (padded ? launch_route_gather<true>(g, row_bytes, f, workspace, workspace_bytes, s, &rc)
               : launch_route_gather<false>(g, row_bytes, f, workspace, workspace_bytes, s, &rc))
      return rc;
  }
  const int rc = moe_route_build(top_expert, g.n, E, pad_multiple, indices, bin_ids, bins, padded_bins, positions,
                                 workspace, workspace_bytes, g.status, reinterpret_cast<moe_stream_t>(s));
  if (rc != MOE_OK || g.rows_out == 0 || g.vecs == 0) return rc;
  g.positions = positions;
  return padded ? dispatch_gather<true>(g, dtype, s) : dispatch_gather<false>(g, dtype, s);
}

extern "C" void moe_test_barrier_slack(uint32_t extra) { g_barrier_slack.store(extra, std::memory_order_relaxed); }

extern "C" size_t moe_route_build_gather_workspace_size(int64_t n, int32_t num_experts) {
  const size_t route = moe_route_build_workspace_size(n, num_experts);
  if (route == 0 || num_experts > kStageMax) return route;
  const int64_t grid = max(route_gather_grid<true>(), route_gather_grid<false>());
  if (grid < 1) return route;
  const size_t fused = (route_gather_workspace(grid, num_experts) + 255) / 256 * 256;
  return fused > route ? fused : route;
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
