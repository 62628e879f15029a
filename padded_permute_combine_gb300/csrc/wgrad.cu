// Router-weight gradient, binned and padded
// ("Build Triton-Ascend Binned MoE Routing": Goal, Workflow step 6,
//  Guardrails "accumulate wgrad reductions in float32";
//  "Build Triton-Ascend Padded MoE Routing": Workflow step 6, Guardrails on
//  unique assignment ids and reductions across column tiles).
//
// Padded layout, two launches: the first writes the inverse permutation of
// `indices` into the caller's wgrad buffer (it has exactly n 32-bit slots),
// so no workspace is needed; the second gives one warp one assignment at a
// time in assignment order, so the TOP_K assignments of a token run on
// neighbouring warps and share the token's gradient row through L1: each
// gradient row leaves HBM about once, each expert row once. Binned layout,
// one launch: capacity drops a contiguous tail of every expert's bin, so
// the warps walk only the kept rows (in four phases, each a quarter of
// every expert's rows, i.e. roughly a quarter of the tokens, so a token's
// gradient row stays in L2 between its slots), and a thread-per-slot pass
// writes the dropped slots' 0.
//
// Each dot product is formed in fp32 with compensated summation (Ogita, Rump
// and Oishi, "Accurate Sum and Dot Product", SIAM J. Sci. Comput. 26(6),
// 2005, algorithm Dot2): every product and every partial
// sum carries its exact rounding error (TwoProduct via fma, Knuth's TwoSum),
// the errors are summed separately and added once at the end, and the warp
// reduction combines (sum, error) pairs the same way. For bf16 rows the
// products are exact and the running sums use packed f32x2 instructions, two
// independent compensated sums per register. The result is as accurate as a
// dot computed in twice the working precision and then rounded, independent
// of H. A dropped slot writes 0.
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
  const int32_t* positions = nullptr;  // padded: the caller's inverse of indices (else built in wgrad)
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

// Load of a positions entry that the same kernel later overwrites with an
// fp32 result (no read-only path, ordered against the stores).
__device__ __forceinline__ int32_t ld_position(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Inverse permutation of indices, written into the caller's wgrad buffer
// (n int32 values in its n fp32 slots): positions[indices[i]] = i. The token
// pass reads each slot once and then overwrites it with the result.
__global__ void positions_kernel(const int32_t* __restrict__ indices, int64_t n, int32_t* positions,
                                 int32_t* status) {
  await_previous_kernel();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t a = __ldg(indices + i);
    if (a >= 0 && a < n) positions[a] = (int32_t)i;
    else flag_status(status, MOE_STATUS_BAD_INDEX);
  }
}

// Expert row of sorted position i holding expert e, or -1 when capacity
// drops it or the routing data are inconsistent (status flagged).
template <bool PADDED>
__device__ __forceinline__ int64_t expert_row(const WgradArgs& g, int64_t i, int32_t e) {
  if (e < 0 || e >= g.E) {
    flag_status(g.status, MOE_STATUS_BAD_EXPERT);
    return -1;
  }
  const int64_t start = e > 0 ? __ldg(g.bins + e - 1) : 0;
  const int64_t j = i - start;
  if (j < 0 || i >= __ldg(g.bins + e)) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  int64_t row;
  if (!PADDED) {
    if (j >= g.capacity) return -1;
    row = (int64_t)e * g.capacity + j;
  } else {
    row = (e > 0 ? __ldg(g.padded_bins + e - 1) : 0) + j;
  }
  if (row < 0 || row >= g.xe_rows) {
    flag_status(g.status, MOE_STATUS_BAD_BINS);
    return -1;
  }
  return row;
}

// Row of assignment a, whose sorted position comes from the positions pass
// and is checked against indices, so a stale entry (indices not a
// permutation) is caught rather than followed.
template <bool PADDED>
__device__ __forceinline__ int64_t assignment_row(const WgradArgs& g, int64_t a) {
  const int32_t i = g.positions != nullptr ? __ldg(g.positions + a)
                                            : ld_position(reinterpret_cast<const int32_t*>(g.wgrad) + a);
  if (i < 0 || i >= g.n) {
    flag_status(g.status, MOE_STATUS_BAD_INDEX);
    return -1;
  }
  const int32_t back = __ldg(g.indices + i);  // both loads issued together
  const int32_t e = __ldg(g.bin_ids + i);
  if (back != a) {
    flag_status(g.status, MOE_STATUS_BAD_INDEX);
    return -1;
  }
  return expert_row<PADDED>(g, i, e);
}

// Row of sorted position i and its assignment a (-1 when out of range).
template <bool PADDED>
__device__ __forceinline__ int64_t sorted_row(const WgradArgs& g, int64_t i, int32_t& a) {
  a = __ldg(g.indices + i);
  const int32_t e = __ldg(g.bin_ids + i);
  if (a < 0 || a >= g.n) {
    flag_status(g.status, MOE_STATUS_BAD_INDEX);
    a = -1;
    return -1;
  }
  return expert_row<PADDED>(g, i, e);
}

// One warp owns one item at a time; lane 0 resolves it to an expert row and
// an assignment and broadcasts them, and a dropped slot writes 0. Items are
//  - BY_ASSIGNMENT: assignments in increasing id, so the TOP_K assignments
//    of a token run on neighbouring warps of one CTA and read the token's
//    gradient row through L1 at about the same time (each gradient row
//    leaves HBM about once);
//  - otherwise sorted positions in increasing order, so kept expert rows are
//    read in address order and the positions pass is not needed; gradient
//    rows are loaded evict-last for their later slots.
// Compensated dot product of one expert row and one gradient row (vecs
// vectors each), summed by the whole warp; every lane returns the result.
// L1_GRAD: the gradient row goes through L1 (neighbouring warps read the
// same row); otherwise it is loaded evict-last for its later readers.
// ROT: rotate the vector registers (next pass's loads issued as each vector
// is summed); the binned kept-row walk measured 0.1022 -> 0.1009 ms with it
// at the DeepSeek-V3 batch, while the padded walk, which must stay within
// 64 registers for its occupancy, needs 76 with it and measured slower.
template <int VB, int U, typename ET, bool L1_GRAD, bool ROT = false>
__device__ __forceinline__ float row_dot(const typename Lanes<VB, ET>::V* __restrict__ xr,
                                         const typename Lanes<VB, ET>::V* __restrict__ gv, int64_t vecs, int lane) {
  using L = Lanes<VB, ET>;
  using V = typename L::V;
  constexpr int NE = L::kElems;
  constexpr bool kExact = Elem<ET>::kBytes == 2;  // bf16 x bf16 fits in fp32
  constexpr bool kPacked = kExact && NE % 2 == 0;
  Acc2 acc[2];
  Acc2x2 acc2[2];
  auto load = [&](V (&vx)[U], V (&vg)[U], int64_t c0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u * kWarp + lane;
      if (c < vecs) {
        vx[u] = ld_once(xr + c);  // each expert row is read once
        vg[u] = L1_GRAD ? ld_l1(gv + c) : ld_keep(gv + c);
      }
    }
  };
  auto add = [&](const V (&vx)[U], const V (&vg)[U], int64_t c0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u * kWarp + lane;
      if (c < vecs) {
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
  };
  if constexpr (ROT) {
    // Rotating registers: as soon as vector u of a pass has been summed, its
    // registers receive the loads of vector u of the next pass, so loads are
    // in flight while the pass's other vectors are summed, in no more
    // registers than one pass holds.
    V vx[U], vg[U];
    load(vx, vg, 0);
    for (int64_t c0 = 0; c0 < vecs; c0 += kWarp * U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + u * kWarp + lane;
        if (c < vecs) {
          if constexpr (kPacked) {
#pragma unroll
            for (int p = 0; p < NE / 2; ++p)
              acc2[p & 1].add_exact(f2_mul(f2_elems<ET>(vx[u], p), f2_elems<ET>(vg[u], p)));
          } else {
#pragma unroll
            for (int q = 0; q < NE; ++q)
              acc[q & 1].template add_product<kExact>(L::get(vx[u], q), L::get(vg[u], q));
          }
        }
        const int64_t cn = c + kWarp * U;
        if (cn < vecs) {
          vx[u] = ld_once(xr + cn);
          vg[u] = L1_GRAD ? ld_l1(gv + cn) : ld_keep(gv + cn);
        }
      }
    }
  } else {
    // Each pass loads its vectors, then sums them.
    for (int64_t c0 = 0; c0 < vecs; c0 += kWarp * U) {
      V vx[U], vg[U];
      load(vx, vg, c0);
      add(vx, vg, c0);
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
  return __fadd_rn(acc[0].s, acc[0].c);
}

template <int VB, int U, typename ET, bool PADDED, bool BY_ASSIGNMENT>
__global__ void __launch_bounds__(kThreads) wgrad_kernel(WgradArgs g) {
  await_previous_kernel();
  using V = typename Lanes<VB, ET>::V;
  const int lane = lane_id();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
  const V* __restrict__ xe = reinterpret_cast<const V*>(g.xe);
  const V* __restrict__ gr = reinterpret_cast<const V*>(g.grad);

  for (int64_t item = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; item < g.n;
       item += warps) {
    int64_t row = 0;
    int32_t a = (int32_t)item;
    if (lane == 0) {
      if constexpr (BY_ASSIGNMENT) row = assignment_row<PADDED>(g, a);
      else row = sorted_row<PADDED>(g, item, a);
      if (row < 0 && a >= 0) g.wgrad[a] = 0.0f;
    }
    row = __shfl_sync(0xffffffffu, row, 0);
    a = __shfl_sync(0xffffffffu, a, 0);
    if (row < 0) continue;
    const float r = row_dot<VB, U, ET, BY_ASSIGNMENT>(xe + row * g.vecs, gr + (a / g.top_k) * g.vecs, g.vecs, lane);
    if (lane == 0) g.wgrad[a] = r;
  }
}

// Binned rows, kept slots only. Capacity drops a contiguous tail of each
// expert's bin, so the kept slots are the first min(count_e, capacity)
// rows of each expert: each CTA stages bins and prefix sums of the kept
// counts in shared memory, and the warps walk kept slots k = 0 .. kept-1
// (expert e by binary search on a prefix, then row e*capacity + j, sorted
// position bins[e-1] + j), resolving 32 of them at once (one per lane,
// their index loads overlapping). The walk goes in kKeptParts phases: phase
// p takes rows [floor(c*p/P), floor(c*(p+1)/P)) of every expert (c its kept
// count), in row order. An expert's rows are in token order, so a phase
// covers roughly a P-th of the tokens and the gradient rows it reads stay
// in L2 for those tokens' later slots (DRAM reads 618 MB in one phase, 565
// MB in eight, for 544 MB of expert rows plus one gradient row per token
// at the DeepSeek-V3 batch). Dropped slots never reach a warp:
// a grid-stride pass over the sorted positions, one thread each, writes
// their 0 first. The data checks of the sorted walk are kept: bins
// decreasing or past n, a bin_ids entry that disagrees with bins, an
// indices entry outside [0, n).
constexpr int kKeptStage = 1024;  // experts whose bins fit the shared-memory stage
// Phases of the kept walk: 1 / 2 / 3 / 4 / 6 / 8 measured 0.105 / 0.104 /
// 0.103 / 0.102 / 0.103 / 0.103 ms at the DeepSeek-V3 batch.
constexpr int kKeptParts = 4;

template <int VB, int U, typename ET>
__global__ void __launch_bounds__(kThreads, 4) wgrad_kept_kernel(WgradArgs g) {
  await_previous_kernel();
  using V = typename Lanes<VB, ET>::V;
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kPer = kKeptStage / kThreads;
  __shared__ int32_t sbins[kKeptStage];
  // squant[q-1][e]: inclusive prefix over experts of floor(kept_e * q / P),
  // q = 1..P; squant[P-1] is the prefix of the kept counts themselves.
  __shared__ int32_t squant[kKeptParts][kKeptStage];
  __shared__ int32_t swarp[kKeptParts][kThreads / kWarp];
  int32_t* skept = squant[kKeptParts - 1];
  __shared__ int64_t srow[kThreads];
  __shared__ int32_t sa[kThreads];
  const int tid = threadIdx.x, lane = lane_id(), warp = tid / kWarp;
  for (int e = tid; e < g.E; e += kThreads) sbins[e] = __ldg(g.bins + e);
  __syncthreads();
  // Kept count per expert, then an inclusive block scan (kPer experts per thread).
  // and of its parts' boundaries (floor(count * q / P) rows, q = 1..P).
  int32_t kq[kKeptParts][kPer];
  int32_t run[kKeptParts];
#pragma unroll
  for (int q = 0; q < kKeptParts; ++q) run[q] = 0;
#pragma unroll
  for (int v = 0; v < kPer; ++v) {
    const int e = tid * kPer + v;
    int32_t c = 0;
    if (e < g.E) {
      const int32_t prev = e > 0 ? sbins[e - 1] : 0;
      const bool ok = sbins[e] >= prev && (e < g.E - 1 || sbins[e] <= g.n) && prev >= 0;
      if (!ok && blockIdx.x == 0) flag_status(g.status, MOE_STATUS_BAD_BINS);
      c = ok ? min(sbins[e] - prev, g.capacity) : 0;
    }
#pragma unroll
    for (int q = 0; q < kKeptParts; ++q) {
      run[q] += (int32_t)((int64_t)c * (q + 1) / kKeptParts);
      kq[q][v] = run[q];
    }
  }
  int32_t incl[kKeptParts];
#pragma unroll
  for (int q = 0; q < kKeptParts; ++q) incl[q] = run[q];
#pragma unroll
  for (int d = 1; d < kWarp; d <<= 1) {
#pragma unroll
    for (int q = 0; q < kKeptParts; ++q) {
      const int32_t x = __shfl_up_sync(kAll, incl[q], d);
      if (lane >= d) incl[q] += x;
    }
  }
  if (lane == kWarp - 1) {
#pragma unroll
    for (int q = 0; q < kKeptParts; ++q) swarp[q][warp] = incl[q];
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kKeptParts; ++q) {
    int32_t before = incl[q] - run[q];
    for (int w = 0; w < warp; ++w) before += swarp[q][w];
#pragma unroll
    for (int v = 0; v < kPer; ++v) {
      const int e = tid * kPer + v;
      if (e < g.E) squant[q][e] = before + kq[q][v];
    }
  }
  __syncthreads();

  // Dropped slots (and slots whose data are inconsistent) get 0.
  const int64_t threads = (int64_t)gridDim.x * kThreads;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + tid; i < g.n; i += threads) {
    const int32_t e = __ldg(g.bin_ids + i);
    bool zero;
    if (e < 0 || e >= g.E) {
      flag_status(g.status, MOE_STATUS_BAD_EXPERT);
      zero = true;
    } else {
      const int64_t start = e > 0 ? sbins[e - 1] : 0;
      if (i < start || i >= sbins[e]) {
        flag_status(g.status, MOE_STATUS_BAD_BINS);
        zero = true;
      } else {
        zero = i - start >= g.capacity;
      }
    }
    if (zero) {
      const int32_t a = __ldg(g.indices + i);
      if (a >= 0 && a < g.n) g.wgrad[a] = 0.0f;
      else flag_status(g.status, MOE_STATUS_BAD_INDEX);
    }
  }

  const int64_t kept = skept[g.E - 1];
  const int64_t warps = (int64_t)gridDim.x * (kThreads / kWarp);
  const int64_t first = (int64_t)blockIdx.x * (kThreads / kWarp) + warp;
  const V* __restrict__ xe = reinterpret_cast<const V*>(g.xe);
  const V* __restrict__ gr = reinterpret_cast<const V*>(g.grad);
  for (int64_t base = first; base < kept; base += kWarp * warps) {
    const int64_t k = base + lane * warps;
    int64_t row = -1;
    int32_t a = -1;
    if (k < kept) {
      // P phases: phase p takes rows [floor(c*p/P), floor(c*(p+1)/P)) of
      // every expert (c its kept count). An expert's rows are in token order,
      // so each phase covers roughly a P-th of the tokens, and the gradient
      // rows of a phase are few enough to stay in L2 for the token's later
      // slots.
      int p = 0;
      int64_t base_k = 0;
      while (p + 1 < kKeptParts && k >= (int64_t)squant[p][g.E - 1]) {
        base_k = squant[p][g.E - 1];
        ++p;
      }
      const int32_t* hiq = squant[p];
      const int32_t* loq = p > 0 ? squant[p - 1] : nullptr;
      const int64_t kk = k - base_k;
      int lo = 0, hi = g.E - 1;  // first expert whose prefix (of this phase's rows) passes kk
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int64_t pm = (int64_t)hiq[mid] - (loq ? loq[mid] : 0);
        if (pm > kk) hi = mid;
        else lo = mid + 1;
      }
      const int64_t lo_lo = loq ? loq[lo] : 0;                          // prefix up to lo of this phase's start
      const int64_t lo_prev = lo > 0 ? (loq ? loq[lo - 1] : 0) : 0;     // prefix before lo of this phase's start
      const int64_t hi_prev = lo > 0 ? hiq[lo - 1] : 0;
      const int64_t j = (lo_lo - lo_prev) + kk - (hi_prev - lo_prev);
      const int64_t i = (lo > 0 ? sbins[lo - 1] : 0) + j;
      if (i >= g.n) {
        flag_status(g.status, MOE_STATUS_BAD_BINS);
      } else {
        a = __ldg(g.indices + i);
        const int32_t e = __ldg(g.bin_ids + i);
        if (a < 0 || a >= g.n) {
          flag_status(g.status, MOE_STATUS_BAD_INDEX);
          a = -1;
        } else if (e != lo) {
          flag_status(g.status, MOE_STATUS_BAD_BINS);  // the zero pass wrote this slot
          a = -1;
        } else {
          row = (int64_t)lo * g.capacity + j;
        }
      }
    }
    // The batch waits in shared memory, so its registers are free for the dots.
    __syncwarp();
    srow[tid] = row;
    sa[tid] = a;
    __syncwarp();
    const int n_here = (int)min((int64_t)kWarp, (kept - base + warps - 1) / warps);
    for (int q = 0; q < n_here; ++q) {
      const int64_t r = srow[warp * kWarp + q];
      const int32_t aq = sa[warp * kWarp + q];
      if (r < 0) continue;
      const float d = row_dot<VB, U, ET, false, true>(xe + r * g.vecs, gr + (aq / g.top_k) * g.vecs, g.vecs, lane);
      if (lane == 0) g.wgrad[aq] = d;
    }
  }
}

// Padded rows hold every assignment (TOP_K per token): assignment order,
// which reads each gradient row once, measured fastest there. Binned rows
// hold only the slots within capacity (fewer per token, so fewer gradient
// re-reads, which L2 catches): the kept rows in row order, measured fastest
// there; with more experts than the shared-memory stage holds, the sorted
// walk over every position (dropped ones write 0) instead.
#ifndef MOE_WGRAD_KEPT
#define MOE_WGRAD_KEPT 1
#endif
// Items per warp of the slot-walk grid (0: persistent grid). Two: a CTA per
// sixteen slots, balanced across SMs by the block scheduler (padded
// DeepSeek-V3 batch 0.1766 persistent, 0.1738 at one item per warp, 0.1725
// at two). The kept-row walk stays
// persistent (0.102 -> 0.127 ms with a CTA per eight slots): each of its
// CTAs first stages the bins and the phase prefixes, and its phases keep
// the gradient rows in L2 only while all warps sweep them together.
#ifndef MOE_WGRAD_ITEMS
#define MOE_WGRAD_ITEMS 2
#endif

template <int VB, typename ET, bool PADDED>
int launch_wgrad(const WgradArgs& g, cudaStream_t s) {
  constexpr bool kByAssignment = PADDED;
  if (kByAssignment && g.positions == nullptr) {
    const int64_t blocks = (g.n + 255) / 256;
    launch(positions_kernel, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s,
        g.indices, g.n, reinterpret_cast<int32_t*>(g.wgrad), g.status);
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  }
  constexpr int U = VB == 32 ? 2 : (VB == 16 ? 4 : 8);  // 64 bytes per lane and operand in flight
  if (!PADDED && MOE_WGRAD_KEPT && g.E <= kKeptStage) {
    auto kk = wgrad_kept_kernel<VB, U, ET>;
    const int64_t work_ctas = (g.n + (kThreads / kWarp) - 1) / (kThreads / kWarp);  // a warp per slot at most
    launch(kk, persistent_grid(kk, kThreads, 0, work_ctas), kThreads, 0, s, g);
    return check_launch();
  }
  auto k = wgrad_kernel<VB, U, ET, PADDED, kByAssignment>;
  const int64_t work_ctas = (g.n + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  launch(k, balanced_grid(k, kThreads, 0, work_ctas, MOE_WGRAD_ITEMS), kThreads, 0, s, g);
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
                                const int32_t* bin_ids, const int32_t* bins, const int32_t* padded_bins,
                                const int32_t* positions, int64_t T, int64_t H, int32_t E, int32_t top_k,
                                int64_t xe_rows, float* wgrad, int32_t* d_status, moe_stream_t stream) {
  const int rc = wgrad_checks(xe, grad, dtype, indices, bin_ids, bins, T, H, E, top_k, wgrad, d_status);
  if (rc != MOE_OK) return rc;
  if (padded_bins == nullptr || xe_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(padded_bins, 4) || (positions != nullptr && !aligned(positions, 4))) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (xe == nullptr && xe_rows > 0 && H > 0) return MOE_ERR_INVALID_ARG;
  WgradArgs g{static_cast<const char*>(xe), static_cast<const char*>(grad), wgrad, indices, bin_ids, bins,
              padded_bins, T, T * top_k, H, xe_rows, E, 0, top_k, d_status};
  g.positions = positions;
  return run_wgrad<true>(g, dtype, reinterpret_cast<cudaStream_t>(stream));
}
