// Route build: stable counting sort of expert choices by expert id
// ("Build Triton-Ascend Padded MoE Routing", Workflow steps 1-3;
//  "Build Triton-Ascend Binned MoE Routing", Workflow steps 1-2).
//
// Three launches, no inter-CTA waiting (two when chunks x experts is small:
// the scatter CTAs then each do the scan's work for themselves):
//   1. hist:    CTA g counts the expert ids of its chunk -> counts[g][e].
//   2. scan:    one CTA turns each expert's column of counts into a prefix
//               over chunks and writes bins and padded_bins.
//   3. scatter: CTA g re-reads its chunk and gives every assignment its
//               stable rank (expert start bins[e-1] + the chunk prefix +
//               the rank inside the chunk): warps own consecutive
//               sub-chunks, a warp-level
//               multi-split (__match_any_sync + popc of lower peers) ranks
//               lanes within a round, and per-warp running counters in
//               shared memory carry ranks across rounds and warps.
#include "common.cuh"

namespace moe {
namespace {

// Chunks of 16 warps x 2 rounds (1024 assignments): 64 CTAs at the
// DeepSeek-V3 size (65 536 assignments), whose 64 x 256 count matrix each
// scatter CTA can read to derive its own prefixes. 4 rounds (32 CTAs) took
// 15.9 us, 2 rounds 14.7 us, 1 round (128 CTAs, too many counts for the
// fused scan, so three launches) 17.5 us.
constexpr int kRounds = 2;      // 32-element rounds per warp and chunk
constexpr int kMaxWarps = 16;   // warps per CTA of the hist / scatter passes
constexpr int kSmemBudget = 48 * 1024;  // per-warp counters of the scatter pass
constexpr int kScanThreads = 1024;
// The scan folds into the scatter pass (two launches instead of three) when
// every scatter CTA can afford to read the whole chunk x expert count matrix.
#ifndef MOE_ROUTE_FUSED_MAX_COUNTS
#define MOE_ROUTE_FUSED_MAX_COUNTS 16384
#endif
constexpr int64_t kFusedMaxCounts = MOE_ROUTE_FUSED_MAX_COUNTS;
constexpr int32_t kFusedMaxExperts = 256;

struct RouteShape {
  int warps;      // warps per CTA of the hist / scatter passes
  int64_t chunk;  // assignments per CTA
  int64_t ctas;   // number of chunks
};

RouteShape route_shape(int64_t n, int32_t E) {
  RouteShape s;
  const int w = kSmemBudget / (4 * E);
  s.warps = w > kMaxWarps ? kMaxWarps : (w < 1 ? 1 : w);
  s.chunk = (int64_t)s.warps * kWarp * kRounds;
  s.ctas = n > 0 ? (n + s.chunk - 1) / s.chunk : 1;
  return s;
}

__device__ __forceinline__ int32_t load_expert(const int32_t* top_expert, int64_t p, int64_t n, int32_t E,
                                               int32_t* status) {
  if (p >= n) return -1;
  const int32_t v = __ldg(top_expert + p);
  if (v >= 0 && v < E) return v;
  flag_status(status, MOE_STATUS_BAD_EXPERT);
  return -1;
}

__global__ void route_hist_kernel(const int32_t* __restrict__ top_expert, int64_t n, int32_t E,
                                  int32_t* __restrict__ counts, int32_t* status) {
  await_previous_kernel();
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x / kWarp, lane = lane_id();
  const int64_t base = (int64_t)blockIdx.x * blockDim.x * kRounds + (int64_t)warp * kWarp * kRounds;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int32_t e = load_expert(top_expert, base + r * kWarp + lane, n, E, status);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Single CTA. counts[g][e] becomes the number of expert-e assignments in the
// chunks before g (a column prefix); bins and padded_bins are written. The
// scatter pass adds expert e's start, bins[e-1], to get the first sorted
// position of chunk g's assignments to e.
__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(int32_t* __restrict__ counts, int64_t G, int32_t E,
                                                                   int32_t m, int32_t* __restrict__ bins,
                                                                   int32_t* __restrict__ padded_bins) {
  await_previous_kernel();
  __shared__ int32_t start[MOE_MAX_EXPERTS];
  __shared__ int64_t warp_sum[kScanThreads / kWarp][2];
  // Column pass: exclusive prefix over chunks, total per expert.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = 0;
    int64_t g = 0;
    for (; g + 8 <= G; g += 8) {
      int32_t c[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) c[q] = counts[(g + q) * E + e];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        counts[(g + q) * E + e] = run;
        run += c[q];
      }
    }
    for (; g < G; ++g) {
      const int32_t c = counts[g * E + e];
      counts[g * E + e] = run;
      run += c;
    }
    start[e] = run;  // total count of expert e for now
  }
  __syncthreads();
  // Exclusive scan over experts of the counts and of the padded counts.
  const int per = (E + kScanThreads - 1) / kScanThreads;
  const int lo = threadIdx.x * per;
  const int hi = min(lo + per, (int)E);
  int64_t s = 0, ps = 0;
  for (int e = lo; e < hi; ++e) {
    const int64_t c = start[e];
    s += c;
    ps += (c + m - 1) / m * m;
  }
  const int lane = lane_id(), warp = threadIdx.x / kWarp;
  int64_t xs = s, xps = ps;
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int64_t a = __shfl_up_sync(0xffffffffu, xs, d);
    const int64_t b = __shfl_up_sync(0xffffffffu, xps, d);
    if (lane >= d) { xs += a; xps += b; }
  }
  if (lane == kWarp - 1) { warp_sum[warp][0] = xs; warp_sum[warp][1] = xps; }
  __syncthreads();
  if (warp == 0) {
    int64_t a = warp_sum[lane][0], b = warp_sum[lane][1];
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
      const int64_t ua = __shfl_up_sync(0xffffffffu, a, d);
      const int64_t ub = __shfl_up_sync(0xffffffffu, b, d);
      if (lane >= d) { a += ua; b += ub; }
    }
    warp_sum[lane][0] = a;
    warp_sum[lane][1] = b;
  }
  __syncthreads();
  int64_t run = xs - s + (warp > 0 ? warp_sum[warp - 1][0] : 0);
  int64_t prun = xps - ps + (warp > 0 ? warp_sum[warp - 1][1] : 0);
  for (int e = lo; e < hi; ++e) {
    const int64_t c = start[e];
    run += c;
    prun += (c + m - 1) / m * m;
    bins[e] = (int32_t)run;
    if (padded_bins != nullptr) padded_bins[e] = (int32_t)prun;
  }
}

// Exclusive block scan over experts of v[e] (in place) and of its rounding
// up to multiples of m (into pv, when pv is not null); every thread of the
// block takes part. Returns nothing; the inclusive values are v + count.
__device__ void block_scan_experts(int64_t* v, int64_t* pv, int32_t E, int32_t m, int64_t (*warp_sum)[2]) {
  const int nt = blockDim.x, lane = lane_id(), warp = threadIdx.x / kWarp;
  const int per = (E + nt - 1) / nt;
  const int lo = threadIdx.x * per;
  const int hi = min(lo + per, (int)E);
  int64_t s = 0, ps = 0;
  for (int e = lo; e < hi; ++e) {
    s += v[e];
    ps += (v[e] + m - 1) / m * m;
  }
  int64_t xs = s, xps = ps;
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
    const int64_t a = __shfl_up_sync(0xffffffffu, xs, d);
    const int64_t b = __shfl_up_sync(0xffffffffu, xps, d);
    if (lane >= d) { xs += a; xps += b; }
  }
  if (lane == kWarp - 1) { warp_sum[warp][0] = xs; warp_sum[warp][1] = xps; }
  __syncthreads();
  if (warp == 0) {
    const int nw = nt / kWarp;
    int64_t a = lane < nw ? warp_sum[lane][0] : 0, b = lane < nw ? warp_sum[lane][1] : 0;
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
      const int64_t ua = __shfl_up_sync(0xffffffffu, a, d);
      const int64_t ub = __shfl_up_sync(0xffffffffu, b, d);
      if (lane >= d) { a += ua; b += ub; }
    }
    if (lane < nw) { warp_sum[lane][0] = a; warp_sum[lane][1] = b; }
  }
  __syncthreads();
  int64_t run = xs - s + (warp > 0 ? warp_sum[warp - 1][0] : 0);
  int64_t prun = xps - ps + (warp > 0 ? warp_sum[warp - 1][1] : 0);
  for (int e = lo; e < hi; ++e) {
    const int64_t c = v[e];
    v[e] = run;
    run += c;
    if (pv != nullptr) {
      pv[e] = prun;
      prun += (c + m - 1) / m * m;
    }
  }
  __syncthreads();
}

// FUSED (few chunks, E <= kFusedMaxExperts): `offsets` holds the raw
// per-chunk counts of the hist pass and every CTA derives what the scan pass
// would have given it — its column prefix over the chunks before it and the
// exclusive scan over experts of the totals — from the whole count matrix
// (read from L2, with every thread of the CTA summing a share of the chunks
// of one expert); CTA 0 also writes bins and padded_bins. One launch fewer,
// and still no CTA waits on another. The chunk's expert ids are loaded
// first, so their latency overlaps the count reads (route build at the
// DeepSeek-V3 batch 14.7 -> 14.0 us with both).
template <bool FUSED>
__global__ void route_scatter_kernel(const int32_t* __restrict__ top_expert, int64_t n, int32_t E,
                                     const int32_t* __restrict__ offsets, int64_t G, int32_t m,
                                     int32_t* __restrict__ bins, int32_t* __restrict__ padded_bins,
                                     int32_t* __restrict__ indices, int32_t* __restrict__ bin_ids,
                                     int32_t* __restrict__ positions) {
  await_previous_kernel();
  extern __shared__ int32_t whist[];  // [warps][E]: per-warp running offsets; FUSED: then 4 x [E] int64
  __shared__ int64_t warp_sum[kMaxWarps][2];
  const int warps = blockDim.x / kWarp;
  const int warp = threadIdx.x / kWarp, lane = lane_id();
  // This chunk's expert ids first: their loads overlap the count reads below.
  const int64_t base = (int64_t)blockIdx.x * blockDim.x * kRounds + (int64_t)warp * kWarp * kRounds;
  int32_t ex[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) ex[r] = load_expert(top_expert, base + r * kWarp + lane, n, E, nullptr);
  int64_t* spre = reinterpret_cast<int64_t*>(whist + ((warps * E + 1) & ~1));  // prefix over earlier chunks
  int64_t* stot = spre + E;                                                     // total per expert
  int64_t* sst = stot + E;                                                      // exclusive start per expert
  int64_t* spst = sst + E;                                                      // padded start (CTA 0)
  if (FUSED) {
    // Column sums over the chunks, split over `parts` threads per expert
    // (their partial sums parked in whist before it is cleared), loads
    // issued eight at a time.
    int parts = (int)(blockDim.x / E);
    if (parts > warps / 2) parts = warps / 2;
    if (parts < 1) parts = 1;
    const int64_t per = (G + parts - 1) / parts;
    for (int t = threadIdx.x; t < E * parts; t += blockDim.x) {
      const int e = t % E, part = t / E;
      const int64_t g0 = part * per, g1 = min(G, g0 + per);
      int32_t pre = 0, tot = 0;
      int64_t g = g0;
      for (; g + 8 <= g1; g += 8) {
        int32_t c[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) c[q] = __ldg(offsets + (g + q) * E + e);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pre += (g + q) < (int64_t)blockIdx.x ? c[q] : 0;
          tot += c[q];
        }
      }
      for (; g < g1; ++g) {
        const int32_t c = __ldg(offsets + g * E + e);
        pre += g < (int64_t)blockIdx.x ? c : 0;
        tot += c;
      }
      whist[(2 * part) * E + e] = pre;
      whist[(2 * part + 1) * E + e] = tot;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int64_t pre = 0, tot = 0;
      for (int part = 0; part < parts; ++part) {
        pre += whist[(2 * part) * E + e];
        tot += whist[(2 * part + 1) * E + e];
      }
      spre[e] = pre;
      stot[e] = tot;
      sst[e] = tot;
    }
    __syncthreads();
    block_scan_experts(sst, blockIdx.x == 0 ? spst : nullptr, E, m, warp_sum);
    if (blockIdx.x == 0) {
      for (int e = threadIdx.x; e < E; e += blockDim.x) {
        bins[e] = (int32_t)(sst[e] + stot[e]);
        if (padded_bins != nullptr) padded_bins[e] = (int32_t)(spst[e] + (stot[e] + m - 1) / m * m);
      }
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < warps * E; q += blockDim.x) whist[q] = 0;
  __syncthreads();
  int32_t* mine = whist + warp * E;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const unsigned peers = __match_any_sync(0xffffffffu, ex[r]);
    if (ex[r] >= 0 && lane == __ffs(peers) - 1) mine[ex[r]] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = FUSED ? (int32_t)(spre[e] + sst[e]) : offsets[(int64_t)blockIdx.x * E + e] + (e > 0 ? bins[e - 1] : 0);
    for (int w = 0; w < warps; ++w) {
      const int32_t c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int32_t e = ex[r];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int32_t dst = mine[e] + __popc(peers & lt);
      const int32_t a = (int32_t)(base + r * kWarp + lane);
      indices[dst] = a;
      bin_ids[dst] = e;
      if (positions != nullptr) positions[a] = dst;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_build_workspace_size(int64_t n, int32_t num_experts) {
  if (n < 0 || num_experts < 1 || num_experts > MOE_MAX_EXPERTS) return 0;
  const RouteShape s = route_shape(n, num_experts);
  const size_t bytes = (size_t)s.ctas * (size_t)num_experts * sizeof(int32_t);
  return (bytes + 255) / 256 * 256;
}

extern "C" int moe_route_build(const int32_t* top_expert, int64_t n, int32_t E, int32_t pad_multiple,
                               int32_t* indices, int32_t* bin_ids, int32_t* bins, int32_t* padded_bins,
                               int32_t* positions, void* workspace, size_t workspace_bytes, int32_t* d_status,
                               moe_stream_t stream) {
  if (n < 0 || n > INT32_MAX || E < 1 || E > MOE_MAX_EXPERTS || pad_multiple < 1) return MOE_ERR_INVALID_ARG;
  if (n + (int64_t)E * (pad_multiple - 1) > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (bins == nullptr || workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (top_expert == nullptr || indices == nullptr || bin_ids == nullptr)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_route_build_workspace_size(n, E)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {top_expert, indices, bin_ids, bins, padded_bins, positions, workspace, d_status};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, 4)) return MOE_ERR_UNSUPPORTED;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const RouteShape shape = route_shape(n, E);
  int32_t* counts = static_cast<int32_t*>(workspace);
  const int threads = shape.warps * kWarp;
  launch(route_hist_kernel, (unsigned)shape.ctas, threads, E * sizeof(int32_t), s, top_expert, n, E, counts, d_status);
  const size_t whist_bytes = (size_t)shape.warps * E * sizeof(int32_t);
  if (n > 0 && E <= kFusedMaxExperts && shape.ctas * E <= kFusedMaxCounts) {
    const size_t smem = (whist_bytes + 7) / 8 * 8 + 4 * (size_t)E * sizeof(int64_t);
    launch(route_scatter_kernel<true>, (unsigned)shape.ctas, threads, smem, s, top_expert, n, E, counts, shape.ctas,
           pad_multiple, bins, padded_bins, indices, bin_ids, positions);
    return check_launch();
  }
  launch(route_scan_kernel, 1, kScanThreads, 0, s, counts, shape.ctas, E, pad_multiple, bins, padded_bins);
  if (n > 0)
    launch(route_scatter_kernel<false>, (unsigned)shape.ctas, threads, whist_bytes, s, top_expert, n, E, counts,
           shape.ctas, pad_multiple, bins, padded_bins, indices, bin_ids, positions);
  return check_launch();
}
