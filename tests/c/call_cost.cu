// Host time of back-to-back calls of the C interface: 400 BF16 512^3
// products enqueued on one stream (the GPU runs each in a few microseconds,
// so the queue never fills and the time measured is the caller's), seven
// repetitions, and for comparison the same count of empty kernel launches.
// Prints "call_us <median>" and "launch_us <median>".
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <vector>

#include "dgt_gemm.h"

__global__ void empty_kernel(int) {}

template <class F>
double median_us_per_call(F f) {
  std::vector<double> reps;
  for (int r = 0; r < 7; ++r) {
    const auto t0 = std::chrono::steady_clock::now();
    for (int i = 0; i < 400; ++i)
      if (!f(i)) return -1.0;
    const auto t1 = std::chrono::steady_clock::now();
    if (cudaDeviceSynchronize() != cudaSuccess) return -1.0;
    reps.push_back(std::chrono::duration<double, std::micro>(t1 - t0).count() / 400);
  }
  std::sort(reps.begin(), reps.end());
  return reps[3];
}

int main() {
  const int n = 512;
  uint16_t *A = nullptr, *B = nullptr, *C = nullptr;
  if (cudaMalloc(&A, n * n * 2) != cudaSuccess || cudaMalloc(&B, n * n * 2) != cudaSuccess ||
      cudaMalloc(&C, n * n * 2) != cudaSuccess)
    return 2;
  cudaMemset(A, 0, n * n * 2);
  cudaMemset(B, 0, n * n * 2);
  cudaStream_t s;
  cudaStreamCreate(&s);
  for (int i = 0; i < 50; ++i)
    if (gemm_bf16(n, n, n, A, n, B, n, C, n, GEMM_B_ROW_MAJOR, s) != GEMM_OK) return 3;
  cudaDeviceSynchronize();
  const double call = median_us_per_call([&](int) { return gemm_bf16(n, n, n, A, n, B, n, C, n, 0, s) == GEMM_OK; });
  const double launch = median_us_per_call([&](int i) {
    empty_kernel<<<1, 32, 0, s>>>(i);
    return cudaGetLastError() == cudaSuccess;
  });
  if (call < 0 || launch < 0) return 4;
  printf("call_us %.3f\nlaunch_us %.3f\n", call, launch);
  return 0;
}
