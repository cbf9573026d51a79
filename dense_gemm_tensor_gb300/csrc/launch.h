// Internal interface between the C-ABI host code and the per-dtype kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "gemm_kernel_pair.cuh"

namespace dgt {

struct LaunchPlan {
  CUtensorMap tmA;  // valid when p.a_tma
  CUtensorMap tmB;  // valid when p.b_tma
  CUtensorMap tmB2; // MN-major B whose tile columns are not whole 128-byte boxes: the last, narrower box
  CUtensorMap tmC;  // valid when p.c_tma
  GemmParams p;
  bool b_kmajor;
  bool pair;  // CTA-pair kernel (cta_group::2)
  bool swap;  // pair kernel on the transposed product (row-major B; OPS_SWAP)
  int pairs;  // pair kernel: CTA pairs per cluster (1, or 2 sharing A by multicast)
  int bn;     // output tile width: one of kTileWidths (single) or kPairTileWidths (pair)
  int grid;
  int threads;
  cudaStream_t stream;
  int dev;  // ordinal of the current device
};

// Kernel launch and co-resident cluster count for one (kind, B layout): the
// single-CTA kernels in gemm_<kind>_<layout>.cu, the CTA-pair kernels in
// gemm_<kind>_<layout>_pair.cu and the two-pair kernels in
// gemm_<kind>_<layout>_quad.cu, so that the units build in parallel. The FP8 kinds exist for K-major B only (a row-major B
// is transposed into scratch first).
#define DGT_DECLARE_VARIANTS(name)                       \
  cudaError_t launch_##name(const LaunchPlan& L);        \
  cudaError_t launch_##name##_pair(const LaunchPlan& L); \
  cudaError_t launch_##name##_quad(const LaunchPlan& L); \
  int pair_clusters_##name(int bn, int pairs);           \
  int quad_clusters_##name(int bn);
DGT_DECLARE_VARIANTS(f16_rm)
DGT_DECLARE_VARIANTS(f16_km)
DGT_DECLARE_VARIANTS(bf16_rm)
DGT_DECLARE_VARIANTS(bf16_km)
DGT_DECLARE_VARIANTS(tf32_rm)
DGT_DECLARE_VARIANTS(tf32_km)
DGT_DECLARE_VARIANTS(e4m3_km)
DGT_DECLARE_VARIANTS(e5m2_km)
#undef DGT_DECLARE_VARIANTS
// The pair kernel on the transposed product (row-major B), one unit per kind.
cudaError_t launch_f16_sw(const LaunchPlan& L);
cudaError_t launch_bf16_sw(const LaunchPlan& L);
cudaError_t launch_tf32_sw(const LaunchPlan& L);
cudaError_t launch_fill_zero(void* C, long long ldc, int M, int N, int es, cudaStream_t stream, int sm_count);
// dst[n][k] = src[k][n] for a rows x cols byte matrix (leading dimensions in bytes).
cudaError_t launch_transpose_bytes(const void* src, int64_t src_ld, void* dst, int64_t dst_ld, int64_t rows,
                                   int64_t cols, cudaStream_t stream, int sm_count);
// The K = 0 product with a fused epilogue (epilogue_only_kernel).
cudaError_t launch_epilogue_only(int kind, void* C, long long ldc, int M, int N, const GemmParams& p,
                                 cudaStream_t stream, int sm_count);
// Copies `rows` rows of `row_bytes` from a source with `gran`-byte-aligned row
// starts to a destination with 16-byte-aligned rows (pack_rows_kernel); up to
// two such copies in one launch.
struct PackSpec {
  const void* src;
  int64_t src_ld_bytes;
  void* dst;
  int64_t dst_ld_bytes;
  int64_t rows;
  int64_t row_bytes;
  int gran;
};
cudaError_t launch_pack(const PackSpec* specs, int n, cudaStream_t stream, int sm_count);

// Split-tail scratch layout: arrival counters (one per CTA of a cluster of up
// to four) for up to 1024 split work tiles, then the fp32 partial tiles.
constexpr size_t kSplitCounterBytes = kSplitCounters * sizeof(unsigned long long);

// Caller-owned scratch for the split tail (instead of the per-stream buffer
// the library allocates): device address and capacity in bytes.
struct ExternalScratch {
  void* ptr;
  size_t bytes;
};

// The C entry points' common body; `ext` non-null: take the split-tail
// scratch from `ext` and refuse plans that need more than it holds.
int run_gemm_external(int kind, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                      int64_t ldb, void* C, int64_t ldc, int layout, void* stream, const ExternalScratch* ext);

// Releases the staging of the host-memory calls (gemm_*_host); the device
// must be idle.
int free_host_buffers();

// Tile widths the kernels are built for (the host picks one per call). The
// single-CTA kernel also takes 64 and 32: a small product then spreads over
// more SMs, each taking in fewer operand bytes per k-slab (512^3 BF16 6.17 ->
// 5.23 us with 32-wide tiles, 1024^3 8.62 -> 8.00 us with 64-wide ones).
constexpr int kTileWidths[] = {256, 224, 192, 128, 64, 32};
constexpr int kPairTileWidths[] = {256, 224, 192, 128};


// Sets the kernel's dynamic shared-memory limit once per device, then launches.
template <int KIND, bool KMAJ, int BN, bool FUSED>
cudaError_t launch_variant(const LaunchPlan& L) {
  static int configured[64] = {};
  const int dev = L.dev;
  cudaError_t e;
  auto kern = gemm_kernel<KIND, KMAJ, BN, FUSED>;
  constexpr int smem = Cfg<KIND, KMAJ, BN>::SMEM_BYTES;
  if (dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pair_variant
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(L.threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmB2, L.tmC, L.p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KIND, bool KMAJ, bool FUSED>
cudaError_t launch_width(const LaunchPlan& L) {
  switch (L.bn) {
    case 256: return launch_variant<KIND, KMAJ, 256, FUSED>(L);
    case 224: return launch_variant<KIND, KMAJ, 224, FUSED>(L);
    case 192: return launch_variant<KIND, KMAJ, 192, FUSED>(L);
    case 128: return launch_variant<KIND, KMAJ, 128, FUSED>(L);
    case 64: return launch_variant<KIND, KMAJ, 64, FUSED>(L);
    case 32: return launch_variant<KIND, KMAJ, 32, FUSED>(L);
    default: return cudaErrorInvalidValue;
  }
}

// The single-CTA kernel, built with the fused epilogue and, for plain
// launches, without it (fewer registers; BF16 512^3 to 2048^3 in CUDA graphs
// on GB300 ran 1-2% faster: 5.05 -> 4.96 us, 14.94 -> 14.63 us).
template <int KIND, bool KMAJ>
cudaError_t launch_layout(const LaunchPlan& L) {
  return L.p.fused ? launch_width<KIND, KMAJ, true>(L) : launch_width<KIND, KMAJ, false>(L);
}


template <int KIND, int OPS, int BN, int PAIRS, bool FUSED>
cudaError_t launch_pair_variant(const LaunchPlan& L) {
  static int configured[64] = {};
  const int dev = L.dev;
  cudaError_t e;
  auto kern = gemm_kernel_pair<KIND, OPS, BN, PAIRS, FUSED>;
  constexpr int smem = PairCfg<KIND, OPS, BN>::SMEM_BYTES;
  if (dev >= 64 || !__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * PAIRS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: the kernel may be scheduled while the
  // previous kernel on the stream finishes; it runs its set-up, then waits
  // (griddepcontrol.wait) for that kernel to complete before touching memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(L.threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmB2, L.tmC, L.p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Co-resident clusters of one pair variant (occupancy query with its launch shape).
template <int KIND, int OPS, int BN, int PAIRS>
int pair_clusters_variant() {
  auto kern = gemm_kernel_pair<KIND, OPS, BN, PAIRS, true>;
  constexpr int smem = PairCfg<KIND, OPS, BN>::SMEM_BYTES;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * PAIRS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * PAIRS, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int KIND, int OPS, int PAIRS, bool FUSED = true>
cudaError_t launch_pair_width(const LaunchPlan& L) {
  switch (L.bn) {
    case 256: return launch_pair_variant<KIND, OPS, 256, PAIRS, FUSED>(L);
    case 224: return launch_pair_variant<KIND, OPS, 224, PAIRS, FUSED>(L);
    case 192: return launch_pair_variant<KIND, OPS, 192, PAIRS, FUSED>(L);
    case 128: return launch_pair_variant<KIND, OPS, 128, PAIRS, FUSED>(L);
    default: return cudaErrorInvalidValue;
  }
}

// One CTA pair per cluster: built with the fused epilogue and, for plain
// launches, without it (its registers then hold nothing for the fused terms:
// no spills); two pairs sharing A (their own unit): with it only.
template <int KIND, int OPS>
cudaError_t launch_pair_layout(const LaunchPlan& L) {
  if (L.pairs != 1) return cudaErrorInvalidValue;
  return L.p.fused ? launch_pair_width<KIND, OPS, 1, true>(L) : launch_pair_width<KIND, OPS, 1, false>(L);
}

template <int KIND, int OPS, int PAIRS>
int pair_clusters_width(int bn) {
  switch (bn) {
    case 256: return pair_clusters_variant<KIND, OPS, 256, PAIRS>();
    case 224: return pair_clusters_variant<KIND, OPS, 224, PAIRS>();
    case 192: return pair_clusters_variant<KIND, OPS, 192, PAIRS>();
    case 128: return pair_clusters_variant<KIND, OPS, 128, PAIRS>();
    default: return 0;
  }
}

// Body of one gemm_<kind>_<layout>.cu: the single-CTA kernels of that kind
// and B layout, each tile width; pair plans go to launch_<name>_pair.
#define DGT_DEFINE_VARIANTS(name, KIND, KMAJ)                                                  \
  cudaError_t launch_##name(const LaunchPlan& L) {                                             \
    if (L.b_kmajor != (KMAJ) || L.swap) return cudaErrorInvalidValue;                          \
    return L.pair ? launch_##name##_pair(L) : launch_layout<KIND, KMAJ>(L);                    \
  }

// Body of one gemm_<kind>_<layout>_pair.cu: the CTA-pair kernels of that
// kind and B layout, each tile width, with and without the fused epilogue;
// two-pair plans go to launch_<name>_quad.
#define DGT_DEFINE_PAIR_VARIANTS(name, KIND, KMAJ)                                             \
  cudaError_t launch_##name##_pair(const LaunchPlan& L) {                                      \
    if (L.b_kmajor != (KMAJ) || L.swap || !L.pair) return cudaErrorInvalidValue;               \
    if (L.pairs == 2) return launch_##name##_quad(L);                                          \
    return launch_pair_layout<KIND, (KMAJ) ? OPS_B_K : OPS_B_MN>(L);                           \
  }                                                                                            \
  int pair_clusters_##name(int bn, int pairs) {                                                \
    if (pairs == 1) return pair_clusters_width<KIND, (KMAJ) ? OPS_B_K : OPS_B_MN, 1>(bn);      \
    if (pairs == 2) return quad_clusters_##name(bn);                                           \
    return 0;                                                                                  \
  }

// Body of one gemm_<kind>_<layout>_quad.cu: the two-pair kernels (two CTA
// pairs sharing A by TMA multicast), each tile width; a build without
// multicast defines the same two calls without them (DGT_DEFINE_NO_QUAD).
#define DGT_DEFINE_QUAD_VARIANTS(name, KIND, KMAJ)                                             \
  cudaError_t launch_##name##_quad(const LaunchPlan& L) {                                      \
    if (L.b_kmajor != (KMAJ) || L.swap || !L.pair || L.pairs != 2) return cudaErrorInvalidValue; \
    return launch_pair_width<KIND, (KMAJ) ? OPS_B_K : OPS_B_MN, 2>(L);                         \
  }                                                                                            \
  int quad_clusters_##name(int bn) { return pair_clusters_width<KIND, (KMAJ) ? OPS_B_K : OPS_B_MN, 2>(bn); }
#define DGT_DEFINE_NO_QUAD(name)                                                               \
  cudaError_t launch_##name##_quad(const LaunchPlan&) { return cudaErrorInvalidValue; }        \
  int quad_clusters_##name(int) { return 0; }

// Body of one gemm_<kind>_sw.cu: the pair kernel on the transposed product,
// each width, built twice: with the fused epilogue, and without it for plain
// launches (no registers held for the fused terms: measured 0.1-0.6% faster).
#define DGT_DEFINE_SWAP_VARIANTS(name, KIND)                                   \
  cudaError_t launch_##name(const LaunchPlan& L) {                             \
    if (L.b_kmajor || !L.pair || !L.swap || L.pairs != 1) return cudaErrorInvalidValue; \
    return L.p.fused ? launch_pair_width<KIND, OPS_SWAP, 1, true>(L)           \
                     : launch_pair_width<KIND, OPS_SWAP, 1, false>(L);         \
  }

}  // namespace dgt
