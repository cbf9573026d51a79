// gemm_bf16_static_scratch: the BF16 product with no allocation at all.
//
// Some callers cannot let a library call cudaMalloc: a serving process that
// hands all device memory to its own pool at start-up (a later cudaMalloc
// fails, or fragments that pool), a host application whose plug-ins must not
// allocate behind its back, or code on a latency budget that cannot absorb
// the device-wide synchronisation cudaFree implies. gemm_bf16 allocates once
// per stream, the first time a shape splits its last round of tiles along K;
// this entry point runs the same kernels and takes that scratch from a fixed
// array in this library's device memory instead.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "dgt_gemm.h"
#include "launch.h"

namespace {

// The fixed scratch: split-tile arrival counters, then fp32 partial tiles.
// Every GPU that loads this library holds it until the process exits.
constexpr size_t kStaticScratchBytes = dgt::kSplitCounterBytes + (size_t(16) << 20);
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct StaticScratch {
  std::atomic<bool> ready{false};  // set up on that device
  void* ptr = nullptr;             // device address of g_static_scratch on that device
};
StaticScratch g_scratch[64];
std::mutex g_scratch_mutex;

// Per device, on the first call with that device current: look up the
// array's device address (the name is only a host-side stand-in) and zero
// the counters. Allocates nothing. A set-up that fails (for instance one
// attempted inside a stream capture, where the synchronisation is not
// allowed) leaves the device not set up, so the next call tries again.
int static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  StaticScratch& s = g_scratch[dev];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!s.ready.load(std::memory_order_relaxed)) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
      if (cudaMemset(p, 0, dgt::kSplitCounterBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
      s.ptr = p;
      s.ready.store(true, std::memory_order_release);
    }
  }
  *out = s.ptr;
  return GEMM_OK;
}

}  // namespace

extern "C" int gemm_bf16_static_scratch(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                        const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc, int layout,
                                        void* stream) {
  void* ptr = nullptr;
  const int st = static_scratch(&ptr);
  if (st != GEMM_OK) return st;
  const dgt::ExternalScratch ext{ptr, kStaticScratchBytes};
  return dgt::run_gemm_external(dgt::KIND_BF16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, &ext);
}
