// Shared device and host helpers of the routing library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_route.h"

namespace moe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- device

__device__ __forceinline__ void flag_status(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

__device__ __forceinline__ int lane_id() { return (int)(threadIdx.x & 31u); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 32 bytes moved by one 256-bit load or store (sm_100 and later).
struct alignas(32) u32x8 {
  uint32_t w[8];
};

// Vector of VB bytes used for row copies.
template <int VB> struct Vec;
template <> struct Vec<32> { using T = u32x8; };
template <> struct Vec<16> { using T = uint4; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<4> { using T = uint32_t; };
template <> struct Vec<2> { using T = uint16_t; };

// Read-only load of data that is not re-read through L1.
__device__ __forceinline__ u32x8 ld_stream(const u32x8* p) {
  u32x8 v;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_stream(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 256-bit loads with an L2 eviction priority: ld_keep marks the lines
// evict-last (rows re-read by later warps: token rows of the gather, gradient
// rows of wgrad), ld_once evict-first (rows read exactly once). Narrower
// vectors take ld_stream.
__device__ __forceinline__ u32x8 ld_keep(const u32x8* p) {
  u32x8 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_last.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p));
  return v;
}
__device__ __forceinline__ u32x8 ld_once(const u32x8* p) {
  u32x8 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p));
  return v;
}
template <typename V> __device__ __forceinline__ V ld_keep(const V* p) { return ld_stream(p); }
template <typename V> __device__ __forceinline__ V ld_once(const V* p) { return ld_stream(p); }

// Read-only load that allocates in L1: for rows that neighbouring warps of
// the same CTA read at about the same time.
__device__ __forceinline__ u32x8 ld_l1(const u32x8* p) {
  u32x8 v;
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_l1(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ uint2 ld_l1(const uint2* p) { return __ldg(p); }
__device__ __forceinline__ uint32_t ld_l1(const uint32_t* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }
__device__ __forceinline__ uint16_t ld_l1(const uint16_t* p) { return __ldg(reinterpret_cast<const unsigned short*>(p)); }

// Store of write-once output: evict-first so it does not push reused inputs out of L2.
__device__ __forceinline__ void st_stream(u32x8* p, const u32x8& v) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
               "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_stream(uint32_t* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_stream(uint16_t* p, uint16_t v) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

template <typename V> __device__ __forceinline__ V zero_vec();
template <> __device__ __forceinline__ u32x8 zero_vec<u32x8>() {
  u32x8 v;
#pragma unroll
  for (int q = 0; q < 8; ++q) v.w[q] = 0u;
  return v;
}
template <> __device__ __forceinline__ uint4 zero_vec<uint4>() { return make_uint4(0, 0, 0, 0); }
template <> __device__ __forceinline__ uint2 zero_vec<uint2>() { return make_uint2(0, 0); }
template <> __device__ __forceinline__ uint32_t zero_vec<uint32_t>() { return 0u; }
template <> __device__ __forceinline__ uint16_t zero_vec<uint16_t>() { return (uint16_t)0; }

// Element access inside a 32-bit word, as fp32.
template <typename E> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float get(uint32_t w, int half) { (void)half; return __uint_as_float(w); }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  // half 0 = low 16 bits (the element at the lower address).
  __device__ __forceinline__ static float get(uint32_t w, int half) {
    return __uint_as_float(half ? (w & 0xffff0000u) : (w << 16));
  }
};

// fp32 -> bf16 pair (round to nearest even), low element first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Error-free transformation of a sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Programmatic dependent launch (every kernel of the library is launched
// with it, see launch()): the kernel's grid may be launched while the
// previous kernel on the stream is still finishing, so it waits here for
// that kernel's results before its first global-memory access. No kernel
// triggers its dependents early: the next grid launches as this one's CTAs
// exit. (Triggering at kernel start let the next grid's CTAs settle on the
// SMs unevenly while this one still ran, and the persistent grid-stride
// kernels then lost more than the overlap gained: 1.11 vs 0.99 ms per
// DeepSeek-V3-shaped routing step.) With a previous kernel that was
// launched without the attribute, the wait is a no-op.
__device__ __forceinline__ void await_previous_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ host

int num_sms();       // SMs of the current device (cached per device)
int check_launch();  // MOE_OK or MOE_ERR_CUDA after a launch
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int dtype_bytes(int32_t dtype) { return dtype == MOE_F32 ? 4 : (dtype == MOE_BF16 ? 2 : 0); }

// Widest vector (max_bytes, ..., 4 or 2 bytes, at least min_bytes) that
// divides the row and keeps every given pointer aligned; 0 if none.
inline int pick_vec_bytes(int64_t row_bytes, const void* const* ptrs, int nptrs, int min_bytes, int max_bytes = 16) {
  for (int vb = max_bytes; vb >= min_bytes; vb >>= 1) {
    if (row_bytes % vb) continue;
    bool ok = true;
    for (int q = 0; q < nptrs; ++q) ok = ok && (ptrs[q] == nullptr || aligned(ptrs[q], vb));
    if (ok) return vb;
  }
  return 0;
}

// Launches `kernel` on `s` with programmatic stream serialization, so that
// its launch overlaps the tail of the previous kernel (which the kernel
// waits for in await_previous_kernel()). Errors surface through
// cudaGetLastError like a <<<>>> launch.
template <typename... KArgs, typename... Args>
void launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Grid of CTAs for a grid-stride kernel: enough to fill every SM at the
// kernel's occupancy, but no more than `work_ctas`.
template <typename Kernel>
int persistent_grid(Kernel k, int threads, size_t smem, int64_t work_ctas) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) != cudaSuccess || per_sm < 1) {
    (void)cudaGetLastError();
    per_sm = 1;
  }
  int64_t g = (int64_t)per_sm * num_sms();
  if (work_ctas < g) g = work_ctas;
  return (int)(g < 1 ? 1 : g);
}

// Grid for a grid-stride kernel whose warps each take about `items_per_warp`
// items: ceil(work_ctas / items_per_warp) CTAs (work_ctas = CTAs at one item
// per warp), more than fit at once, so the block scheduler hands the later
// CTAs to whichever SMs free up first and uneven item costs even out across
// SMs. items_per_warp <= 0 gives the persistent grid.
template <typename Kernel>
int balanced_grid(Kernel k, int threads, size_t smem, int64_t work_ctas, int items_per_warp) {
  if (items_per_warp <= 0) return persistent_grid(k, threads, smem, work_ctas);
  int64_t g = (work_ctas + items_per_warp - 1) / items_per_warp;
  if (g > 0x7fffffff) g = 0x7fffffff;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace moe
