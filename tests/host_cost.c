/*
 * host_cost.c -- host time of one wq_matmul call, measured from C (no Python
 * or ctypes in the loop).  Allocates the int4 g128 buffers of an M x K x N
 * problem on the current device (contents left as allocated: only the host
 * side is timed), makes one call outside the timing (plans, kernel attributes
 * and tensor maps are then cached), then times `calls` back-to-back calls
 * with clock_gettime, synchronising only at the end.  Prints one JSON line.
 *   host_cost M K N calls
 * Built and run by tests/test_host_cost_gpu.py.
 */
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

#include <cuda_runtime.h>

#include "wq.h"

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

int main(int argc, char **argv) {
  if (argc < 5) {
    fprintf(stderr, "usage: host_cost M K N calls\n");
    return 2;
  }
  const int M = atoi(argv[1]), K = atoi(argv[2]), N = atoi(argv[3]), calls = atoi(argv[4]);
  const int G = K / 128;
  void *x, *w, *s, *z, *y, *ws = NULL;
  if (cudaMalloc(&x, (size_t)M * K * 2) || cudaMalloc(&w, (size_t)K * N / 2) || cudaMalloc(&s, (size_t)G * N * 2) ||
      cudaMalloc(&z, (size_t)((G + 7) / 8) * N * 4) || cudaMalloc(&y, (size_t)M * N * 4)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 1;
  }
  cudaMemset(w, 0, (size_t)K * N / 2);
  cudaMemset(s, 0, (size_t)G * N * 2);
  cudaMemset(z, 0, (size_t)((G + 7) / 8) * N * 4);
  cudaMemset(x, 0, (size_t)M * K * 2);
  const size_t need = wq_workspace_bytes(M, N, K, 4, 128);
  if (need) {
    if (cudaMalloc(&ws, need)) return 1;
    cudaMemset(ws, 0, need);
  }
  cudaStream_t st;
  cudaStreamCreate(&st);
  wq_status r = wq_matmul(x, WQ_BF16, w, s, WQ_BF16, (const int32_t *)z, M, N, K, 4, 128, (float *)y, ws, need, st);
  if (r != WQ_OK) {
    fprintf(stderr, "wq_matmul: %s\n", wq_status_string(r));
    return 1;
  }
  cudaStreamSynchronize(st);
  double best = 1e30, total = 0;
  const double t0 = now_us();
  for (int i = 0; i < calls; ++i) {
    const double a = now_us();
    r = wq_matmul(x, WQ_BF16, w, s, WQ_BF16, (const int32_t *)z, M, N, K, 4, 128, (float *)y, ws, need, st);
    const double b = now_us();
    if (r != WQ_OK) return 1;
    if (b - a < best) best = b - a;
    total += b - a;
  }
  const double t1 = now_us();
  cudaStreamSynchronize(st);
  printf("{\"M\": %d, \"K\": %d, \"N\": %d, \"calls\": %d, \"host_us_mean\": %.3f, \"host_us_min\": %.3f, "
         "\"loop_us_per_call\": %.3f}\n",
         M, K, N, calls, total / calls, best, (t1 - t0) / calls);
  return wq_check_device(st) == WQ_OK ? 0 : 1;
}
