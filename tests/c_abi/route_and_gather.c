/*
 * A plain C host of the routing library: no Python, no torch. It allocates
 * device memory with the CUDA runtime, runs moe_route_build and then
 * moe_binned_gather / moe_padded_gather / moe_binned_scatter through the C
 * ABI of include/moe_route.h on a seeded problem, then the route build +
 * padded gather in one launch (workspace of
 * moe_route_build_gather_workspace_size bytes, filled with 0xff first so
 * that the test can see the launch wrote its count matrix), and writes the
 * inputs and every output to a binary file for the test to compare with the
 * oracle.
 *
 *   route_and_gather OUT.bin
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "moe_route.h"

#define CHECK_CUDA(x)                                                              \
  do {                                                                             \
    cudaError_t e_ = (x);                                                          \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                      \
      return 2;                                                                    \
    }                                                                              \
  } while (0)
#define CHECK_MOE(x)                                                               \
  do {                                                                             \
    int r_ = (x);                                                                  \
    if (r_ != MOE_OK) {                                                            \
      fprintf(stderr, "%s: %s\n", #x, moe_error_string(r_));                        \
      return 3;                                                                    \
    }                                                                              \
  } while (0)

static uint32_t lcg(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;
  return *s >> 8;
}

static int put(FILE* f, const void* host, size_t bytes) { return fwrite(host, 1, bytes, f) == bytes ? 0 : 1; }

int main(int argc, char** argv) {
  if (argc != 2) return 1;
  const int64_t T = 100, H = 24;
  const int32_t E = 7, K = 3, m = 4, cap = 40;
  const int64_t n = T * K;
  int32_t* te = malloc(n * sizeof(int32_t));
  float* x = malloc(T * H * sizeof(float));
  uint32_t seed = 12345u;
  for (int64_t a = 0; a < n; ++a) te[a] = (int32_t)(lcg(&seed) % (uint32_t)E);
  for (int64_t i = 0; i < T * H; ++i) x[i] = (float)((int32_t)(lcg(&seed) % 2001u) - 1000) / 64.0f;

  int32_t *d_te, *d_idx, *d_bid, *d_bins, *d_pb, *d_pos, *d_status;
  float *d_x, *d_xb, *d_xp, *d_y;
  void* d_ws;
  const size_t ws = moe_route_build_workspace_size(n, E);
  CHECK_CUDA(cudaMalloc((void**)&d_te, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_idx, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_bid, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_pos, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_bins, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_pb, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_status, 4));
  CHECK_CUDA(cudaMalloc(&d_ws, ws));
  CHECK_CUDA(cudaMalloc((void**)&d_x, T * H * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_xb, (size_t)E * cap * H * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_y, T * H * 4));
  CHECK_CUDA(cudaMemcpy(d_te, te, n * 4, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(d_x, x, T * H * 4, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(d_status, 0, 4));
  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreate(&s));

  CHECK_MOE(moe_route_build(d_te, n, E, m, d_idx, d_bid, d_bins, d_pb, d_pos, d_ws, ws, d_status, s));
  /* binned gather without positions (it builds its own), padded gather with the route build's */
  CHECK_MOE(moe_binned_gather(d_x, MOE_F32, d_idx, d_bins, NULL, T, H, E, cap, K, d_xb, d_status, s));
  CHECK_MOE(moe_binned_scatter(d_xb, MOE_F32, d_idx, d_bid, d_bins, NULL, d_pos, T, H, E, cap, K, d_y, NULL, 0,
                               d_status, s));
  int32_t* bins = malloc(E * 4);
  int32_t* pb = malloc(E * 4);
  CHECK_CUDA(cudaMemcpyAsync(pb, d_pb, E * 4, cudaMemcpyDeviceToHost, s));
  CHECK_CUDA(cudaStreamSynchronize(s));
  const int64_t P = pb[E - 1];  /* the caller reads the padded row count back to size the output */
  CHECK_CUDA(cudaMalloc((void**)&d_xp, (P > 0 ? P : 1) * H * 4));
  CHECK_MOE(moe_padded_gather(d_x, MOE_F32, d_idx, d_bins, d_pb, d_pos, T, H, E, K, d_xp, P, d_status, s));
  CHECK_CUDA(cudaStreamSynchronize(s));

  int32_t *idx = malloc(n * 4), *bid = malloc(n * 4), *pos = malloc(n * 4), status = 0;
  float *xb = malloc((size_t)E * cap * H * 4), *xp = malloc((P > 0 ? P : 1) * H * 4), *y = malloc(T * H * 4);
  CHECK_CUDA(cudaMemcpy(idx, d_idx, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(bid, d_bid, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(pos, d_pos, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(bins, d_bins, E * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(xb, d_xb, (size_t)E * cap * H * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(xp, d_xp, P * H * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(y, d_y, T * H * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));

  /* route build + padded gather in one call, sized for the single launch */
  const size_t ws1 = moe_route_build_gather_workspace_size(n, E);
  const int64_t out_rows = n + (int64_t)E * (m - 1); /* the bound: no read-back needed */
  int32_t *d_idx1, *d_bid1, *d_bins1, *d_pb1, *d_pos1;
  float* d_xp1;
  void* d_ws1;
  CHECK_CUDA(cudaMalloc((void**)&d_idx1, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_bid1, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_pos1, n * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_bins1, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_pb1, E * 4));
  CHECK_CUDA(cudaMalloc((void**)&d_xp1, out_rows * H * 4));
  CHECK_CUDA(cudaMalloc(&d_ws1, ws1));
  CHECK_CUDA(cudaMemset(d_ws1, 0xff, ws1));
  CHECK_MOE(moe_route_build_padded_gather(d_te, d_x, MOE_F32, T, H, E, K, m, d_idx1, d_bid1, d_bins1, d_pb1, d_pos1,
                                          d_xp1, out_rows, d_ws1, ws1, d_status, s));
  CHECK_CUDA(cudaStreamSynchronize(s));
  int32_t *idx1 = malloc(n * 4), *bid1 = malloc(n * 4), *pos1 = malloc(n * 4), *bins1 = malloc(E * 4),
          *pb1 = malloc(E * 4), *wsh = malloc(ws1);
  float* xp1 = malloc(out_rows * H * 4);
  CHECK_CUDA(cudaMemcpy(idx1, d_idx1, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(bid1, d_bid1, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(pos1, d_pos1, n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(bins1, d_bins1, E * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(pb1, d_pb1, E * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(xp1, d_xp1, out_rows * H * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(wsh, d_ws1, ws1, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
  int64_t untouched = 0; /* words still 0xffffffff */
  for (size_t i = 0; i < ws1 / 4; ++i) untouched += wsh[i] == -1;

  FILE* f = fopen(argv[1], "wb");
  if (f == NULL) return 4;
  const int64_t header[8] = {T, H, E, K, m, cap, P, status};
  int bad = put(f, header, sizeof(header)) | put(f, te, n * 4) | put(f, x, T * H * 4) | put(f, idx, n * 4) |
            put(f, bid, n * 4) | put(f, bins, E * 4) | put(f, pb, E * 4) | put(f, pos, n * 4) |
            put(f, xb, (size_t)E * cap * H * 4) | put(f, xp, P * H * 4) | put(f, y, T * H * 4);
  const int64_t tail[3] = {out_rows, (int64_t)(ws1 / 4), untouched};
  bad |= put(f, tail, sizeof(tail)) | put(f, idx1, n * 4) | put(f, bid1, n * 4) | put(f, bins1, E * 4) |
         put(f, pb1, E * 4) | put(f, pos1, n * 4) | put(f, xp1, out_rows * H * 4);
  fclose(f);
  printf("moe_version %d, status %d, padded rows %lld\n", moe_version(), status, (long long)P);
  return bad ? 5 : 0;
}
