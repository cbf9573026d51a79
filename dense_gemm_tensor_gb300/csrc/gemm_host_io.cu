// gemm_{tf32,f16,bf16}_host: the product of operands that live in host memory.
//
// Each call copies B and A into device staging buffers, runs the product
// through the device entry point of the same kind, and copies C back into
// host memory, all enqueued asynchronously. A is sent in row blocks so that
// the product of block i runs while block i+1 is still arriving and block
// i-1's rows of C are already on their way back:
//
//   copy-in stream    B | A0 | A1 | A2 | A3
//   caller's stream         P0 | P1 | P2 | P3         (products, after their block arrived)
//   copy-out stream              C0 | C1 | C2 | C3    (after their product)
//
// The staging buffers belong to the library: two slots per (device, stream)
// that consecutive calls take in turn, so one call's uploads may run while
// the previous call's products and downloads finish. A slot's operands are
// overwritten only once the products that read them are done (an event the
// products' stream records), and its C only after the copy-out that read it
// (the caller's stream waits for every call's last download).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "dgt_gemm.h"
#include "launch.h"

namespace {

constexpr int kMaxBlocks = 4;         // row blocks of A per call
constexpr int64_t kBlockRows = 1024;  // at least this many rows per block

struct Slot {
  void* buf = nullptr;
  size_t bytes = 0;
  cudaEvent_t free = nullptr;  // recorded after the last product that read the slot's operands
  bool used = false;
};

struct HostIo {
  std::mutex mu;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t arrived[kMaxBlocks] = {}, computed[kMaxBlocks] = {}, done = nullptr;
  Slot slot[2];
  int next = 0;
  bool ready = false;
};

std::mutex g_mu;
std::unordered_map<uint64_t, HostIo*> g_io;  // (device, stream) -> state; kept until gemm_free_workspaces

HostIo* state_for(int dev, cudaStream_t stream) {
  const uint64_t key = (uint64_t(uint32_t(dev)) << 56) ^ uint64_t(reinterpret_cast<uintptr_t>(stream));
  std::lock_guard<std::mutex> lock(g_mu);
  HostIo*& s = g_io[key];
  if (s == nullptr) s = new HostIo();
  return s;
}

bool init_state(HostIo& s) {
  if (s.ready) return true;
  bool ok = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kMaxBlocks; ++i)
    ok = cudaEventCreateWithFlags(&s.arrived[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s.computed[i], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i) ok = cudaEventCreateWithFlags(&s.slot[i].free, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    // release what was created, so that a later call starts again from nothing
    cudaGetLastError();
    if (s.in) cudaStreamDestroy(s.in);
    if (s.out) cudaStreamDestroy(s.out);
    if (s.done) cudaEventDestroy(s.done);
    for (int i = 0; i < kMaxBlocks; ++i) {
      if (s.arrived[i]) cudaEventDestroy(s.arrived[i]);
      if (s.computed[i]) cudaEventDestroy(s.computed[i]);
      s.arrived[i] = s.computed[i] = nullptr;
    }
    for (int i = 0; i < 2; ++i) {
      if (s.slot[i].free) cudaEventDestroy(s.slot[i].free);
      s.slot[i].free = nullptr;
    }
    s.in = s.out = nullptr;
    s.done = nullptr;
    cudaGetLastError();
    return false;
  }
  s.ready = true;
  return true;
}

// A staging slot of at least `bytes`; a slot that must grow is replaced once
// the products that last used it are done (the only synchronisation here).
void* slot_buffer(Slot& sl, size_t bytes, cudaStream_t out) {
  if (sl.bytes >= bytes) return sl.buf;
  if (sl.buf != nullptr) {
    // the products that read the slot and the copy-out that reads its C are done
    if (sl.used && (cudaEventSynchronize(sl.free) != cudaSuccess || cudaStreamSynchronize(out) != cudaSuccess)) {
      cudaGetLastError();
      return nullptr;
    }
    cudaFree(sl.buf);
    sl.buf = nullptr;
    sl.bytes = 0;
  }
  if (cudaMalloc(&sl.buf, bytes) != cudaSuccess) {
    cudaGetLastError();
    sl.buf = nullptr;
    return nullptr;
  }
  sl.bytes = bytes;
  return sl.buf;
}

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

// Device memory where host memory belongs? (Its copies would be of the wrong
// kind; such a call is refused before anything is enqueued.)
bool is_device_pointer(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

typedef int (*DeviceGemm)(int64_t, int64_t, int64_t, const void*, int64_t, const void*, int64_t, void*, int64_t, int,
                          void*);

int run_host(DeviceGemm fn, int es, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, void* C, int64_t ldc, int layout, void* stream_ptr) {
  const int64_t kLim = (int64_t(1) << 31) - 1;
  if (M < 0 || N < 0 || K < 0 || M > kLim || N > kLim || K > kLim) return GEMM_ERR_INVALID_VALUE;
  if (layout != GEMM_B_ROW_MAJOR && layout != GEMM_B_K_MAJOR) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_VALUE;
  const int64_t b_rows = layout == GEMM_B_ROW_MAJOR ? K : N, b_cols = layout == GEMM_B_ROW_MAJOR ? N : K;
  if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < b_cols)) return GEMM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(C) | (K > 0 ? reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) : 0)) %
          es != 0)
    return GEMM_ERR_MISALIGNED;
  if (is_device_pointer(C) || (K > 0 && (is_device_pointer(A) || is_device_pointer(B)))) return GEMM_ERR_INVALID_VALUE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  HostIo& s = *state_for(dev, stream);
  std::lock_guard<std::mutex> lock(s.mu);
  if (!init_state(s)) return GEMM_ERR_LAUNCH;

  // device copies with rows on 128-byte boundaries (TMA-legal, on whole L2 lines)
  const size_t pa = round_up(size_t(K) * es, 128), pb = round_up(size_t(b_cols) * es, 128);
  const size_t pc = round_up(size_t(N) * es, 128);
  const size_t off_b = round_up(size_t(M) * pa, 256), off_c = off_b + round_up(size_t(b_rows) * pb, 256);
  const size_t need = off_c + size_t(M) * pc;
  Slot& sl = s.slot[s.next];
  s.next ^= 1;
  char* buf = static_cast<char*>(slot_buffer(sl, need, s.out));
  if (buf == nullptr) return GEMM_ERR_LAUNCH;
  char *a_d = buf, *b_d = buf + off_b, *c_d = buf + off_c;

  // the slot's operands may be overwritten once the products that read them are done
  if (sl.used && cudaStreamWaitEvent(s.in, sl.free, 0) != cudaSuccess) return GEMM_ERR_LAUNCH;
  if (K > 0 && cudaMemcpy2DAsync(b_d, pb, B, size_t(ldb) * es, size_t(b_cols) * es, size_t(b_rows),
                                 cudaMemcpyHostToDevice, s.in) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_INVALID_VALUE;  // e.g. B is not host memory
  }
  int nblk = int(M / kBlockRows);
  nblk = nblk < 1 ? 1 : nblk > kMaxBlocks ? kMaxBlocks : nblk;
  for (int i = 0; i < nblk; ++i) {
    const int64_t lo = M * i / nblk, hi = M * (i + 1) / nblk;
    if (K > 0 && cudaMemcpy2DAsync(a_d + size_t(lo) * pa, pa, static_cast<const char*>(A) + size_t(lo) * lda * es,
                                   size_t(lda) * es, size_t(K) * es, size_t(hi - lo), cudaMemcpyHostToDevice,
                                   s.in) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_INVALID_VALUE;
    }
    if (cudaEventRecord(s.arrived[i], s.in) != cudaSuccess || cudaStreamWaitEvent(stream, s.arrived[i], 0) != cudaSuccess)
      return GEMM_ERR_LAUNCH;
    const int st = fn(hi - lo, N, K, a_d + size_t(lo) * pa, int64_t(pa / es), b_d, int64_t(pb / es),
                      c_d + size_t(lo) * pc, int64_t(pc / es), layout, stream);
    if (st != GEMM_OK) return st;
    if (cudaEventRecord(s.computed[i], stream) != cudaSuccess || cudaStreamWaitEvent(s.out, s.computed[i], 0) != cudaSuccess)
      return GEMM_ERR_LAUNCH;
    if (cudaMemcpy2DAsync(static_cast<char*>(C) + size_t(lo) * ldc * es, size_t(ldc) * es, c_d + size_t(lo) * pc, pc,
                          size_t(N) * es, size_t(hi - lo), cudaMemcpyDeviceToHost, s.out) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_INVALID_VALUE;  // e.g. C is not host memory
    }
  }
  // operands free after the last product; the caller's stream waits for the last download
  if (cudaEventRecord(sl.free, stream) != cudaSuccess || cudaEventRecord(s.done, s.out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, s.done, 0) != cudaSuccess)
    return GEMM_ERR_LAUNCH;
  sl.used = true;
  return GEMM_OK;
}

int dev_tf32(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
             int64_t ldc, int layout, void* stream) {
  return gemm_tf32(M, N, K, static_cast<const float*>(A), lda, static_cast<const float*>(B), ldb,
                   static_cast<float*>(C), ldc, layout, stream);
}
int dev_f16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
            int64_t ldc, int layout, void* stream) {
  return gemm_f16(M, N, K, static_cast<const uint16_t*>(A), lda, static_cast<const uint16_t*>(B), ldb,
                  static_cast<uint16_t*>(C), ldc, layout, stream);
}
int dev_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
             int64_t ldc, int layout, void* stream) {
  return gemm_bf16(M, N, K, static_cast<const uint16_t*>(A), lda, static_cast<const uint16_t*>(B), ldb,
                   static_cast<uint16_t*>(C), ldc, layout, stream);
}

}  // namespace

namespace dgt {

// Releases the staging buffers, copy streams and events of the host-memory
// calls (the caller has synchronised the device).
int free_host_buffers() {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& kv : g_io) {
    HostIo* s = kv.second;
    for (Slot& sl : s->slot) {
      if (sl.buf != nullptr) cudaFree(sl.buf);
      if (sl.free != nullptr) cudaEventDestroy(sl.free);
    }
    for (int i = 0; i < kMaxBlocks; ++i) {
      if (s->arrived[i] != nullptr) cudaEventDestroy(s->arrived[i]);
      if (s->computed[i] != nullptr) cudaEventDestroy(s->computed[i]);
    }
    if (s->done != nullptr) cudaEventDestroy(s->done);
    if (s->in != nullptr) cudaStreamDestroy(s->in);
    if (s->out != nullptr) cudaStreamDestroy(s->out);
    delete s;
  }
  g_io.clear();
  return GEMM_OK;
}

}  // namespace dgt

extern "C" int gemm_tf32_host(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                              int64_t ldb, float* C, int64_t ldc, int layout, void* stream) {
  return run_host(dev_tf32, 4, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}

extern "C" int gemm_f16_host(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B,
                             int64_t ldb, uint16_t* C, int64_t ldc, int layout, void* stream) {
  return run_host(dev_f16, 2, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}

extern "C" int gemm_bf16_host(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B,
                              int64_t ldb, uint16_t* C, int64_t ldc, int layout, void* stream) {
  return run_host(dev_bf16, 2, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}
