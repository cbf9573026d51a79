// Internal interface between the C-ABI host code and the per-dtype kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace dgt {

struct LaunchPlan {
  CUtensorMap tmA;  // valid when p.a_tma
  CUtensorMap tmB;  // valid when p.b_tma
  GemmParams p;
  bool b_kmajor;
  int grid;
  int threads;
  cudaStream_t stream;
};

cudaError_t launch_f16(const LaunchPlan& L);
cudaError_t launch_bf16(const LaunchPlan& L);
cudaError_t launch_tf32(const LaunchPlan& L);
cudaError_t launch_fill_zero(void* C, long long ldc, int M, int N, int es, cudaStream_t stream, int sm_count);

// Sets the kernel's dynamic shared-memory limit once per device, then launches.
template <int KIND>
cudaError_t launch_kind(const LaunchPlan& L) {
  static int configured[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (L.b_kmajor) {
    auto kern = gemm_kernel<KIND, true>;
    constexpr int smem = Cfg<KIND, true>::SMEM_BYTES;
    if (dev < 64 && !__atomic_load_n(&configured[1][dev], __ATOMIC_ACQUIRE)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      __atomic_store_n(&configured[1][dev], 1, __ATOMIC_RELEASE);
    }
    kern<<<L.grid, L.threads, smem, L.stream>>>(L.tmA, L.tmB, L.p);
  } else {
    auto kern = gemm_kernel<KIND, false>;
    constexpr int smem = Cfg<KIND, false>::SMEM_BYTES;
    if (dev < 64 && !__atomic_load_n(&configured[0][dev], __ATOMIC_ACQUIRE)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      __atomic_store_n(&configured[0][dev], 1, __ATOMIC_RELEASE);
    }
    kern<<<L.grid, L.threads, smem, L.stream>>>(L.tmA, L.tmB, L.p);
  }
  return cudaGetLastError();
}

}  // namespace dgt
