// C-ABI entry points: argument checks, device checks, TMA tensor-map encoding,
// variant selection and the persistent-grid launch. No allocation per call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "dgt_gemm.h"
#include "launch.h"

namespace dgt {

// Device status words: [0] first recorded failure (sticky), [1] epoch of the
// most recently aborted launch. One copy per device that loads the library.
__device__ uint32_t g_status_words[2];

// Row packing: copies rows x row_bytes matrices from sources whose row
// starts are only `gran`-byte aligned (gran in {1, 2, 4, 8, 16}) to
// destinations with 16-byte aligned rows of dst_ld bytes; bytes of a row's
// last 16-byte chunk beyond row_bytes are zero. One launch takes both
// operands of a product. The unit of work is a warp task: kPackSegChunks
// consecutive 16-byte chunks of one row, each lane loading its kPackUnroll
// chunks before it stores any (so every lane keeps that many loads in
// flight); tasks are strided over the grid's warps.
//
// L2 priorities: the source is read with evict_first and the packed copy is
// written with evict_last, so that the copy, which the product reads next,
// stays in L2 in preference to the source it came from. The product's own
// (default-priority) reads of the copy return its lines to normal priority.
// On GB300 this took the 4000 x 4100 x 4104 BF16 product (both operands
// packed) from 101.5 to 96.2 us; the 8-byte loads keep L1 allocation, since
// a chunk's two halves come from the same sectors (without it that operand's
// copy ran 3.5 us slower).
constexpr int kPackUnroll = 4;
constexpr int kPackSegChunks = 32 * kPackUnroll;

struct PackJob {
  const uint8_t* src;
  long long src_ld;  // bytes
  uint8_t* dst;
  long long dst_ld;  // bytes, a multiple of 16
  long long row_bytes;
  long long segs_per_row;  // warp tasks per row
  int gran;
};

// One 16-byte chunk of a source row whose start is G-byte aligned; `valid`
// bytes of it belong to the row (< 16 only for the row's last chunk).
template <int G>
__device__ __forceinline__ uint4 pack_load(const uint8_t* s, long long valid, uint64_t pol) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (valid >= 16) {
    if constexpr (G == 16) {
      asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "l"(s), "l"(pol));
    } else if constexpr (G == 8) {
      asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(s), "l"(pol));
      asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                   : "=r"(v.z), "=r"(v.w)
                   : "l"(s + 8), "l"(pol));
    } else if constexpr (G == 4) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(s);
      v = make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
    } else if constexpr (G == 2) {
      const uint16_t* h = reinterpret_cast<const uint16_t*>(s);
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = uint32_t(__ldg(h + 2 * q)) | (uint32_t(__ldg(h + 2 * q + 1)) << 16);
      v = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int q = 0; q < 16; ++q) w[q >> 2] |= uint32_t(__ldg(s + q)) << (8 * (q & 3));
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (valid > 0) {
    // the row's ragged end, byte by byte
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int q = 0; q < 16; ++q)
      if (q < valid) w[q >> 2] |= uint32_t(__ldg(s + q)) << (8 * (q & 3));
    v = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return v;
}

template <int G>
__device__ __forceinline__ void pack_task(const PackJob& j, long long row, long long seg, int lane, uint64_t pol_src,
                                          uint64_t pol_dst) {
  const uint8_t* s = j.src + row * j.src_ld;
  uint8_t* d = j.dst + row * j.dst_ld;
  const long long b0 = (seg * kPackSegChunks + lane) * 16;
  uint4 v[kPackUnroll];
#pragma unroll
  for (int u = 0; u < kPackUnroll; ++u) {
    const long long b = b0 + u * 32 * 16;
    v[u] = pack_load<G>(s + b, j.row_bytes - b, pol_src);
  }
#pragma unroll
  for (int u = 0; u < kPackUnroll; ++u) {
    const long long b = b0 + u * 32 * 16;
    if (b < j.row_bytes)
      asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(d + b), "r"(v[u].x),
                   "r"(v[u].y), "r"(v[u].z), "r"(v[u].w), "l"(pol_dst)
                   : "memory");
  }
}

// Launched as a programmatic dependent of the previous kernel on the stream
// (which may still be reading this stream's scratch): it waits for that
// kernel before touching memory, and lets the kernel after it be scheduled
// once its own copies are done. Tasks [0, tasks0) belong to j0, the rest to j1.
__global__ void __launch_bounds__(256, 4) pack_rows_kernel(PackJob j0, PackJob j1, long long tasks0,
                                                           long long tasks) {
  grid_dependency_wait();
  uint64_t pol_src, pol_dst;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_src));
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_dst));
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long t = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < tasks;
       t += warps) {
    const bool first = t < tasks0;
    const PackJob j = first ? j0 : j1;
    const long long tt = first ? t : t - tasks0;
    const long long row = tt / j.segs_per_row, seg = tt - row * j.segs_per_row;
    switch (j.gran) {
      case 16: pack_task<16>(j, row, seg, lane, pol_src, pol_dst); break;
      case 8: pack_task<8>(j, row, seg, lane, pol_src, pol_dst); break;
      case 4: pack_task<4>(j, row, seg, lane, pol_src, pol_dst); break;
      case 2: pack_task<2>(j, row, seg, lane, pol_src, pol_dst); break;
      default: pack_task<1>(j, row, seg, lane, pol_src, pol_dst); break;
    }
  }
  grid_launch_dependents();
}

// dst[n][k] = src[k][n] for a rows x cols byte matrix (rows = K, cols = N):
// a row-major K x N FP8 B becomes the K-major N x K operand the FP8 kernels
// read. 64 x 64-byte tiles through shared memory: 256 threads read the tile's
// rows as 4-byte words (bytes at a ragged or unaligned edge), and write the
// transposed rows as 4-byte words gathered from four tile rows. The tiles are
// strided over the grid. dst_ld is a multiple of 64 no smaller than rows
// rounded up to 64, so the words past `rows` land in the row's padding.
__global__ void __launch_bounds__(256) transpose_bytes_kernel(const uint8_t* __restrict__ src, long long src_ld,
                                                              uint8_t* __restrict__ dst, long long dst_ld,
                                                              int rows, int cols, int src_words) {
  __shared__ __align__(16) uint8_t tile[64][68];
  const int tiles_c = (cols + 63) / 64;
  const long long ntiles = static_cast<long long>((rows + 63) / 64) * tiles_c;
  const int t = threadIdx.x;
  for (long long tt = blockIdx.x; tt < ntiles; tt += gridDim.x) {
    const int r0 = static_cast<int>(tt / tiles_c) * 64, c0 = static_cast<int>(tt % tiles_c) * 64;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (t >> 4) + 16 * i, w = t & 15;  // tile row, word
      const int gr = r0 + r, gc = c0 + 4 * w;
      uint32_t v = 0;
      if (gr < rows) {
        const uint8_t* p = src + static_cast<long long>(gr) * src_ld + gc;
        if (src_words && gc + 3 < cols) {
          v = *reinterpret_cast<const uint32_t*>(p);
        } else {
          for (int j = 0; j < 4; ++j)
            if (gc + j < cols) v |= uint32_t(p[j]) << (8 * j);
        }
      }
      *reinterpret_cast<uint32_t*>(&tile[r][4 * w]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = (t >> 4) + 16 * i, w = t & 15;  // dst row (tile column), word
      if (c0 + c < cols) {
        const uint32_t v = uint32_t(tile[4 * w][c]) | (uint32_t(tile[4 * w + 1][c]) << 8) |
                           (uint32_t(tile[4 * w + 2][c]) << 16) | (uint32_t(tile[4 * w + 3][c]) << 24);
        *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(c0 + c) * dst_ld + r0 + 4 * w) = v;
      }
    }
    __syncthreads();
  }
}

namespace {

constexpr int kMaxDevices = 64;
// Default bound of every wait inside the kernels: far above any wait of a
// launch that makes progress (a 16384^3 product takes a few milliseconds), so
// that a launch slowed by other work sharing the GPU does not give up and
// leave C unspecified, yet a launch that can never finish still ends.
constexpr uint64_t kDefaultWaitLimitNs = 10000000000ull;  // 10 s

struct DeviceInfo {
  int status;  // GEMM_OK or the reason this device cannot run the kernels
  int sm_count;
  uint32_t* status_words;
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
std::atomic<uint32_t> g_epoch{1};
std::atomic<uint64_t> g_launches{0};
std::atomic<uint32_t> g_debug_flags{0};
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
// The plan of the calling thread's last successful launch (see gemm_last_plan).
thread_local int32_t t_last_plan[8] = {0, 0, 0, 0, 0, 0, 0, 0};
std::atomic<int> g_force_variant{0};
std::atomic<int> g_force_bn{0};
std::atomic<int> g_force_raster{0};
std::atomic<int> g_force_split{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Looks up (once per device) whether the current device is an sm_103 part,
// its SM count and the device address of the status words; `dev_out` (if
// given) receives the device's ordinal.
int current_device(const DeviceInfo** out, int* dev_out = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::call_once(g_dev_once[dev], [dev] {
    DeviceInfo& d = g_dev[dev];
    int major = 0, minor = 0;
    d.status = GEMM_ERR_UNSUPPORTED_DEVICE;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) return;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_words) != cudaSuccess) {
      cudaGetLastError();
      d.status = GEMM_ERR_LAUNCH;
      return;
    }
    d.status_words = static_cast<uint32_t*>(p);
    d.status = GEMM_OK;
  });
  *out = &g_dev[dev];
  if (dev_out != nullptr) *dev_out = dev;
  return g_dev[dev].status;
}

PFN_cuPointerGetAttributes_v7000 g_ptr_attrs = nullptr;
std::once_flag g_ptr_attrs_once;

// Device (or managed) memory of device `dev` (the current one)? One driver
// query of three attributes (about half the cost of the runtime's query).
bool is_device_memory(const void* ptr, int dev) {
  std::call_once(g_ptr_attrs_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &fn, 7000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ptr_attrs = reinterpret_cast<PFN_cuPointerGetAttributes_v7000>(fn);
  });
  if (g_ptr_attrs != nullptr) {
    unsigned int type = 0, managed = 0;
    int ordinal = -1;
    CUpointer_attribute at[3] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_IS_MANAGED,
                                 CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL};
    void* data[3] = {&type, &managed, &ordinal};
    // unknown pointers come back as success with zeroed attributes
    if (g_ptr_attrs(3, at, data, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS) return false;
    if (managed) return true;
    return type == CU_MEMORYTYPE_DEVICE && ordinal == dev;
  }
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  if (a.type != cudaMemoryTypeDevice) return false;
  return a.device == dev;
}

// Byte range [lo, hi) touched by a rows x cols matrix with row pitch ld.
void extent(const void* p, int64_t rows, int64_t cols, int64_t ld, int es, uintptr_t* lo, uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * es);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Largest power-of-two granularity in [es, 16] that divides the address and
// the row pitch in bytes.
int granularity(const void* p, int64_t ld, int es) {
  const uint64_t v = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(p)) | static_cast<uint64_t>(ld * es);
  int g = 16;
  while (g > es && (v % g) != 0) g >>= 1;
  return g;
}

// A few entries of host-side work per calling thread, keyed by the plain
// numbers it was computed from (no device state enters it), so an entry can
// never go stale: the same key always yields the same value. Calls that repeat
// a shape on the same buffers -- the common case in a loop -- skip the work.
template <int NK, class Val, int N>
struct TinyCache {
  uint64_t keys[N][NK];
  Val vals[N];
  bool used[N] = {};
  int next = 0;
  const Val* find(const uint64_t (&k)[NK]) const {
    for (int i = 0; i < N; ++i)
      if (used[i] && memcmp(keys[i], k, sizeof(k)) == 0) return &vals[i];
    return nullptr;
  }
  void put(const uint64_t (&k)[NK], const Val& v) {
    memcpy(keys[next], k, sizeof(k));
    vals[next] = v;
    used[next] = true;
    next = (next + 1) % N;
  }
};

// 3-D tiled tensor map: x innermost (contiguous), y rows `row_bytes` apart, z
// matrices of a batch `mat_bytes` apart (depth 1 for one product, whose z is
// always 0). Boxes are box_inner x box_outer x 1. Encoded maps are cached per
// thread (a map is a pure function of these arguments).
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint64_t depth, uint64_t mat_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  thread_local TinyCache<9, CUtensorMap, 16> cache;
  if (depth == 1) mat_bytes = row_bytes * outer;  // never stepped; a stride that spans the matrix
  if (mat_bytes == 0 || mat_bytes % 16 != 0 || mat_bytes >= (uint64_t(1) << 40)) return false;
  const uint64_t key[9] = {uint64_t(dt), uint64_t(reinterpret_cast<uintptr_t>(base)), inner, outer, row_bytes,
                           depth, mat_bytes, (uint64_t(box_inner) << 32) | box_outer, uint64_t(swizzle)};
  if (const CUtensorMap* hit = cache.find(key)) {
    *m = *hit;
    return true;
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, outer, depth};
  cuuint64_t strides[2] = {row_bytes, mat_bytes};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.put(key, *m);
  return true;
}

// The kernel of two CTA pairs sharing A loads it with a cluster-multicast TMA
// copy. The library runs it only in a process that sees exactly one CUDA
// device (and never in a build with DGT_NO_MULTICAST): every multicast copy
// then reads the memory of the one GPU in use. `dev` < 0 (a plan query
// without a device) asks about such a one-GPU process.
bool multicast_allowed(int dev) {
  if (DGT_NO_MULTICAST) return false;
  if (dev < 0) return true;
  static const bool one_device = [] {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return n == 1;
  }();
  return one_device;
}

// Co-resident CTA pairs of each pair-kernel variant, per device (-1 = not queried yet).
std::atomic<int> g_pair_clusters[kMaxDevices][5][2][4][2];
std::once_flag g_pair_once;

int pair_clusters(int dev, int kind, bool kmajor, int bn, int pairs) {
  std::call_once(g_pair_once, [] {
    for (auto& a : g_pair_clusters)
      for (auto& b : a)
        for (auto& c : b)
          for (auto& d : c)
            for (auto& e : d) e.store(-1);
  });
  const int wi = bn == 256 ? 0 : bn == 224 ? 1 : bn == 192 ? 2 : 3;
  std::atomic<int>& slot = g_pair_clusters[dev][kind][kmajor ? 1 : 0][wi][pairs - 1];
  int n = slot.load(std::memory_order_acquire);
  if (n < 0) {
    switch (kind) {
      case KIND_TF32: n = kmajor ? pair_clusters_tf32_km(bn, pairs) : pair_clusters_tf32_rm(bn, pairs); break;
      case KIND_BF16: n = kmajor ? pair_clusters_bf16_km(bn, pairs) : pair_clusters_bf16_rm(bn, pairs); break;
      case KIND_F16: n = kmajor ? pair_clusters_f16_km(bn, pairs) : pair_clusters_f16_rm(bn, pairs); break;
      case KIND_E4M3: n = kmajor ? pair_clusters_e4m3_km(bn, pairs) : 0; break;
      case KIND_E5M2: n = kmajor ? pair_clusters_e5m2_km(bn, pairs) : 0; break;
      default: n = 0;
    }
    slot.store(n, std::memory_order_release);
  }
  return n;
}

// ---------------------------------------------------------------- workspace
// Scratch for the split tail of the pair kernel: arrival counters (first
// kCounterBytes) followed by fp32 partial tiles. One buffer per (device,
// stream), allocated on first need and grown (never shrunk) when a larger plan
// needs it, so calls on one stream reuse it and calls on different streams
// never share it. The counters carry the launch epoch, so they are zeroed once
// at allocation and never reset between calls.
constexpr int kMaxTailSegs = 4;
constexpr int kMinSegmentSlabs = 16;         // k-slabs per segment below which splitting does not pay
// ~4 us at 2 GHz per segment for publishing and reading back a partial tile
// (from measured splits that lost: TF32 2560^3 in three segments 55.6 us
// against 48.8 unsplit on 192-wide tiles; BF16 12288 x 4096 x 4096 in four
// 228.7 against 222.9)
constexpr double kSplitPublishCycles = 8000;
constexpr double kPairLaunchCycles = 8000;    // extra fixed cost of the pair kernel's launch and set-up
// The two-pair kernel (clusters of four) costs about 1.2 us more per launch
// than the plain pair where both run the same rounds (GB300, CUDA graphs:
// BF16 3072^3 35.2 against 34.1 us, 2048 x 2048 x 8192 44.5 against 43.2,
// TF32 2048^3 26.8 against 25.8); where its 36 clusters fit the work in whole
// rounds and the plain pair's 76 pairs do not, it wins (BF16 6144^3, eight
// rounds either way, 241.5 against 252.5 us).
constexpr double kTwoPairLaunchCycles = 2500;
constexpr size_t kCounterBytes = kSplitCounterBytes;  // up to 1024 split tiles

// `ctas`: CTAs per cluster, each publishing its own 128 x bn partial
size_t workspace_bytes(int split_tiles, int segs, int bn, int ctas) {
  return kCounterBytes + size_t(split_tiles) * size_t(segs) * size_t(ctas) * 128u * size_t(bn) * sizeof(float);
}

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mutex;
std::unordered_map<uint64_t, Workspace> g_ws;

void* stream_workspace(int dev, cudaStream_t stream, size_t bytes) {
  const uint64_t key = (uint64_t(uint32_t(dev)) << 56) ^ uint64_t(reinterpret_cast<uintptr_t>(stream));
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace& w = g_ws[key];
  if (w.bytes >= bytes) return w.ptr;
  if (w.ptr != nullptr) {
    cudaFree(w.ptr);  // waits for the device: no kernel can still be using it
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaMemset(p, 0, kCounterBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p);
    return nullptr;
  }
  w.ptr = p;
  w.bytes = bytes;
  return p;
}

void free_workspaces() {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (auto& kv : g_ws)
    if (kv.second.ptr != nullptr) cudaFree(kv.second.ptr);
  g_ws.clear();
}

struct TilePlan {
  bool pair;
  int pairs;  // pair kernel: CTA pairs per cluster (2: the pairs share A and take two adjacent tiles)
  int bn;
  int raster;
  int grid;   // CTAs
  int segs;   // pair kernel: k-slab segments per tile of the last partial round (1 = no split)
  int conc;   // tiles in flight at once (SMs, or co-resident CTA pairs)
  bool swap;  // pair kernel on the transposed product C^T = B^T A^T (row-major B)
};

// Cycles one SM spends per 128-byte k-slab of a tile in the steady state of
// the k-loop, by kernel (single CTA, CTA pair, two pairs sharing A) and tile
// width 256/224/192/128/64/32, measured on GB300 at 4096^3 (bf16; tf32 takes
// the same time per slab). The single CTA's 64- and 32-wide entries follow
// its operand bytes per slab at the SM's intake rate (24 and 20 KB against
// 32 KB at 128 wide); the pair kernels are not built that narrow. The dense MMA rate alone would give 2 x width; the
// rest is time the MMA issuer waits for operands. Sharing A between two pairs
// halves the A bytes each SM fetches from L2 but measured no faster per slab
// at this size, and its clusters of four leave a few SMs idle.
constexpr double kSlabCycles[3][6] = {
    {672.0, 640.0, 605.0, 570.0, 455.0, 380.0},  // single CTA, 128 x width tiles
    {564.0, 504.0, 499.0, 464.0, 0.0, 0.0},      // CTA pair, 256 x width tiles
    {560.0, 503.0, 500.0, 470.0, 0.0, 0.0},      // two pairs sharing A, two 256 x width tiles
};
// TF32 with row-major B fetches B in 32-column boxes, twice as many as the
// 16-bit kinds; its pair and shared-A slabs measured 564/542/495/476 cycles,
// the 224-wide one since recalibrated against the 256-wide one by their times
// at 4096^3 (158.2 and 157.2 us with K walked in alternating directions).
constexpr double kSlabCyclesTf32Mn[4] = {564.0, 512.0, 495.0, 476.0};
// The pair kernel on the transposed product (row-major B as the MMA's A
// operand, in whole 128-byte boxes): its stages hold no unused columns, so
// widths 224 and 192 keep seven stages, which outweighs its costlier
// epilogue (a transpose on the way to shared memory) at 224 and not at 256.
// Scaled from the plain pair's table by the times measured at 4096^3
// (16-bit: 224-wide 82.6 against 84.4 us, 256-wide 89.6 against 87.3 us,
// 192-wide 97.0 us over five rounds; TF32: 154.9 against 158.2 us, 160.6
// against 157.2 us, 192-wide 177.5 us); the 128-wide entries (not measured)
// are the plain pair's with the 256-wide penalty.
constexpr double kSlabCyclesSwap[4] = {579.0, 493.0, 467.0, 476.0};
constexpr double kSlabCyclesSwapTf32[4] = {576.0, 501.0, 461.0, 488.0};
// Its epilogue (the transpose) also costs more per tile, which shows once the
// k-loop is short: 4096 x 4096 x 1024 BF16 ran 34.4 us against 33.6 us.
constexpr double kSwapTileCycles = 600.0;
// The single-CTA kernel with TF32 and row-major B fetches B in eight
// 32-column boxes per stage at width 256: at 2048^3 it ran 38.6 us where the
// CTA pair ran 33.4 (BF16: 22.7 and 23.6 us), about 807 cycles per slab
// against the 16-bit kernel's 672 once the fixed costs are taken out.
constexpr double kSlabCyclesTf32MnSingle[6] = {807.0, 768.0, 726.0, 684.0, 560.0, 470.0};

// Cycles per k-slab of a tile for a kernel family and tile width (wi: index
// into kTileWidths / kPairTileWidths).
double slab_cycles(int kind, bool kmajor, bool pair, int pairs, bool swap, int wi) {
  if (swap) return kind == KIND_TF32 ? kSlabCyclesSwapTf32[wi] : kSlabCyclesSwap[wi];
  if (kind == KIND_TF32 && !kmajor) return pair ? kSlabCyclesTf32Mn[wi] : kSlabCyclesTf32MnSingle[wi];
  return kSlabCycles[pair ? pairs : 0][wi];
}

// Band height of the tile order, in tile rows of `rows` rows each (before
// clamping to the tile rows there are). `nb_ext`: the extent of the other side
// of the tile grid (N, or M for the transposed product).
int band_rows(bool pair, bool swap, int64_t K, int64_t nb_ext, int es, int64_t rows) {
  // the transposed product: bands 16 tile rows high (at 4096^3 that is every
  // 256-column block of C, so consecutive tiles share one block of A's rows)
  // ran about 1.7% faster than 2 (16-bit) or 9 (TF32)
  if (swap) return 16;
  // 2 pair rows / 8 single-CTA rows (measured best at 4096^3) while B stays
  // resident in L2; for a larger B, which is re-read once per band, as many
  // rows as keep the band's A rows within ~40 MB of L2
  const int band_min = pair ? 2 : 8;
  if (double(K) * double(nb_ext) * es <= 64.0e6) return band_min;
  const int band = int(40.0e6 / (double(rows) * double(K) * es));
  return band < band_min ? band_min : band > 16 ? 16 : band;
}

// Picks the kernel (single CTA, CTA pair, two pairs sharing A, or a CTA pair
// on the transposed product), the tile width and the tile order.
//
// Cost model: a tile takes (k-slabs x kSlabCycles) cycles; the grid holds one
// CTA per SM, so a product of T work tiles takes ceil(T / concurrent tiles)
// rounds, the last partial round possibly split along K; the plan with the
// least total time wins. The band height keeps a band's A rows and the B tiles
// in flight inside L2. A call with a fused epilogue (`fused`) does not take
// the transposed product unless forced: its epilogue is the costlier one there
// (4096^3 with beta * C: 100.2 against 97.4 us for BF16, 181.8 against
// 176.8 us for TF32).
//
// pair_conc / quad_conc > 0 give the co-resident CTA pairs / clusters of two
// pairs instead of the occupancy query (gemm_plan_query, without a device).
TilePlan choose_plan_uncached(int dev, int kind, int64_t M, int64_t N, int64_t K, int es, bool kmajor, bool all_tma,
                              int sms, int64_t nbat, bool fused, int pair_conc, int quad_conc, int fv, int fb, int fr,
                              int fs) {
  const int64_t kslabs = (K * es + 127) / 128;
  TilePlan best{false, 1, 256, 8, sms, 1, sms, false};
  double best_cost = -1.0;
  // the transposed product: C's columns take the 256-row side of the pair's tile
  const bool swap_ok = !kmajor && (kind == KIND_TF32 || kind == KIND_F16 || kind == KIND_BF16);
  auto consider = [&](bool pair, int pairs, int bn, bool swap) {
    if (fv == 1 && pair) return;
    if (fv == 2 && !(pair && pairs == 1 && !swap)) return;
    if (fv == 3 && !(pair && pairs == 2)) return;
    if (fv == 4 && !swap) return;
    if (fb && fb != bn) return;
    if (pair && !all_tma) return;
    if (swap && !(swap_ok && pair && pairs == 1)) return;
    if (swap && fused && fv != 4) return;
    if (pairs == 2 && !multicast_allowed(dev)) return;
    // extents of the tile grid: the MMA's A side (256-row pair tiles) and its B side (bn wide)
    const int64_t ma = swap ? N : M, nb_ext = swap ? M : N;
    int conc;  // work tiles in flight
    if (pair) {
      // (the transposed product's kernel has the same cluster shape and one CTA per SM)
      const int given = pairs == 1 ? pair_conc : quad_conc;
      conc = given > 0 ? given : pair_clusters(dev, kind, kmajor, bn, pairs);
      if (conc <= 0) return;
    } else {
      conc = sms;
    }
    const int wi = bn == 256 ? 0 : bn == 224 ? 1 : bn == 192 ? 2 : bn == 128 ? 3 : bn == 64 ? 4 : 5;
    const double slab = slab_cycles(kind, kmajor, pair, pairs, swap, wi);
    const int64_t rows = pair ? 256 : 128;
    const int64_t tiles_n = (nb_ext + bn - 1) / bn;
    const int64_t tiles = nbat * ((ma + rows - 1) / rows) * ((tiles_n + pairs - 1) / pairs);
    const int64_t full = tiles / conc, rest = tiles % conc;
    // pair kernel: the tiles of the last partial round may be split along K
    // into `segs` pieces run by different pairs (fp32 partials summed at the end)
    int segs = 1;
    if (pair && rest > 0 && fs != 1) {
      segs = int(conc / rest);
      if (segs > kMaxTailSegs) segs = kMaxTailSegs;
      while (segs > 1 && kslabs / segs < kMinSegmentSlabs) --segs;
      if (segs < 1) segs = 1;
    }
    const double tile_cost = double(kslabs) * slab + 600.0 + (swap ? kSwapTileCycles : 0.0);
    // a cluster launch with pair set-up costs ~4 us more than a plain one (measured)
    double cost = double(full) * tile_cost + (pair ? kPairLaunchCycles : 0.0) + (pairs == 2 ? kTwoPairLaunchCycles : 0.0);
    if (rest > 0) {
      // a split tile also publishes a 128 KiB fp32 partial per CTA and its last
      // segment reads the other segments' partials back (kSplitPublishCycles each)
      const double split_cost = tile_cost / segs + kSplitPublishCycles * segs;
      if (segs > 1 && split_cost >= tile_cost && fs != 2) segs = 1;  // (2: split wherever possible)
      cost += segs > 1 ? split_cost : tile_cost;
    }
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      const int64_t tiles_m = (ma + rows - 1) / rows;
      const int64_t work = tiles + (segs - 1) * rest;
      const int64_t grid_tiles = work < conc ? work : conc;
      const int band = band_rows(pair, swap, K, nb_ext, es, rows);
      best = TilePlan{pair, pairs, bn, int(tiles_m < band ? tiles_m : band),
                      int(pair ? 2 * pairs * grid_tiles : grid_tiles), segs, conc, swap};
    }
  };
  for (int bn : kPairTileWidths) consider(true, 2, bn, false);
  for (int bn : kPairTileWidths) consider(true, 1, bn, false);
  for (int bn : kPairTileWidths) consider(true, 1, bn, true);
  for (int bn : kTileWidths) consider(false, 1, bn, false);
  if (best_cost < 0) {  // a forced combination that does not apply: fall back to the single-CTA default
    const int64_t tiles = nbat * ((M + 127) / 128) * ((N + 255) / 256);
    best = TilePlan{false, 1, 256, 8, int(tiles < sms ? tiles : sms), 1, sms, false};
  }
  if (fr) best.raster = fr;
  return best;
}

// choose_plan_uncached with the tuning hook's settings, cached per thread (the
// plan is a pure function of the shape, the device's SM and cluster counts and
// those settings).
TilePlan choose_plan(int dev, int kind, int64_t M, int64_t N, int64_t K, int es, bool kmajor, bool all_tma, int sms,
                     int64_t nbat, bool fused, int pair_conc = 0, int quad_conc = 0) {
  const int fv = g_force_variant.load(std::memory_order_relaxed);
  const int fb = g_force_bn.load(std::memory_order_relaxed);
  const int fr = g_force_raster.load(std::memory_order_relaxed);
  const int fs = g_force_split.load(std::memory_order_relaxed);
  thread_local TinyCache<13, TilePlan, 8> cache;
  const uint64_t key[13] = {uint64_t(int64_t(dev)), uint64_t(kind), uint64_t(M), uint64_t(N), uint64_t(K),
                            uint64_t(es) | (uint64_t(kmajor) << 8) | (uint64_t(all_tma) << 9) | (uint64_t(fused) << 10),
                            uint64_t(sms), uint64_t(nbat), uint64_t(pair_conc), uint64_t(quad_conc),
                            (uint64_t(uint32_t(fv)) << 32) | uint32_t(fb), (uint64_t(uint32_t(fr)) << 32) | uint32_t(fs),
                            0};
  if (const TilePlan* hit = cache.find(key)) return *hit;
  const TilePlan plan = choose_plan_uncached(dev, kind, M, N, K, es, kmajor, all_tma, sms, nbat, fused, pair_conc,
                                             quad_conc, fv, fb, fr, fs);
  cache.put(key, plan);
  return plan;
}

// Strided batch of products (batch = 1: one product; strides in elements).
struct Batch {
  int64_t count = 1, stride_a = 0, stride_b = 0, stride_c = 0;
};

// One call of the C interface, with the quantities derived from its kind.
struct Call {
  int kind;
  bool fp8;
  int es;        // operand element size in bytes
  int eo;        // output element size (FP8 writes bfloat16)
  int out_kind;  // kind whose output type C has
  int64_t M, N, K;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  int layout;
  Batch bat;
  const gemm_epilogue_t* epi;
  bool fused;        // the epilogue is not the identity
  const void* bias;  // fused ? epi->bias : nullptr
  cudaStream_t stream;
  const ExternalScratch* ext;
};

// Argument rules of the C interface that need no device (sizes, leading
// dimensions, batch strides, epilogue code, element alignment).
int check_arguments(const Call& c) {
  const int64_t kLim = (int64_t(1) << 31) - 1;
  const int64_t M = c.M, N = c.N, K = c.K;
  if (M < 0 || N < 0 || K < 0 || M > kLim || N > kLim || K > kLim) return GEMM_ERR_INVALID_VALUE;
  if (c.layout != GEMM_B_ROW_MAJOR && c.layout != GEMM_B_K_MAJOR) return GEMM_ERR_INVALID_VALUE;
  const Batch& bat = c.bat;
  if (bat.count < 0 || bat.stride_a < 0 || bat.stride_b < 0 || bat.stride_c < 0) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0 || bat.count == 0) return GEMM_OK;
  if (c.C == nullptr || c.ldc < N) return GEMM_ERR_INVALID_VALUE;
  if (bat.count > 1) {
    // the C matrices must not overlap one another; A and B may repeat (stride 0) but not overlap partly
    if (bat.stride_c < (M - 1) * c.ldc + N) return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && bat.stride_a != 0 && bat.stride_a < (M - 1) * c.lda + K) return GEMM_ERR_INVALID_VALUE;
    const int64_t b_ext = c.layout == GEMM_B_ROW_MAJOR ? (K - 1) * c.ldb + N : (N - 1) * c.ldb + K;
    if (K > 0 && bat.stride_b != 0 && bat.stride_b < b_ext) return GEMM_ERR_INVALID_VALUE;
    if (bat.stride_a > (int64_t(1) << 40) || bat.stride_b > (int64_t(1) << 40) || bat.stride_c > (int64_t(1) << 40))
      return GEMM_ERR_INVALID_VALUE;
    if (bat.count > kLim) return GEMM_ERR_INVALID_VALUE;
    // FP8 B is read K-major; a batch is not transposed
    if (c.fp8 && c.layout != GEMM_B_K_MAJOR) return GEMM_ERR_INVALID_VALUE;
  }
  if (K > 0) {
    if (c.A == nullptr || c.B == nullptr || c.lda < K) return GEMM_ERR_INVALID_VALUE;
    if (c.ldb < (c.layout == GEMM_B_ROW_MAJOR ? N : K)) return GEMM_ERR_INVALID_VALUE;
    if (c.lda > (int64_t(1) << 40) / c.es || c.ldb > (int64_t(1) << 40) / c.es) return GEMM_ERR_INVALID_VALUE;
  }
  if (c.ldc > (int64_t(1) << 40) / c.eo) return GEMM_ERR_INVALID_VALUE;
  if (((M + 127) / 128) * ((N + 127) / 128) > kLim / bat.count) return GEMM_ERR_INVALID_VALUE;
  if (c.epi != nullptr && (c.epi->activation < GEMM_ACT_NONE || c.epi->activation > GEMM_ACT_GELU_TANH))
    return GEMM_ERR_INVALID_VALUE;
  auto mis = [](const void* p, int size) { return (reinterpret_cast<uintptr_t>(p) % size) != 0; };
  if (mis(c.C, c.eo) || (K > 0 && (mis(c.A, c.es) || mis(c.B, c.es))) || (c.bias != nullptr && mis(c.bias, c.eo)))
    return GEMM_ERR_MISALIGNED;
  return GEMM_OK;
}

// Memory rules that need the device: every pointer is device memory, and C
// overlaps neither an operand of the batch nor the bias.
int check_memory(const Call& c, int dev) {
  const int64_t nbat = c.bat.count;
  uintptr_t c0, c1;
  extent(c.C, c.M, c.N, c.ldc, c.eo, &c0, &c1);
  c1 += static_cast<uintptr_t>((nbat - 1) * c.bat.stride_c * c.eo);  // every matrix of the batch
  if (!is_device_memory(c.C, dev)) return GEMM_ERR_NOT_DEVICE_MEMORY;
  if (c.bias != nullptr) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(c.bias), s1 = s0 + uintptr_t(c.N) * c.eo;
    if (overlaps(c0, c1, s0, s1)) return GEMM_ERR_INVALID_VALUE;
    if (!is_device_memory(c.bias, dev)) return GEMM_ERR_NOT_DEVICE_MEMORY;
  }
  if (c.K == 0) return GEMM_OK;
  uintptr_t a0, a1, b0, b1;
  extent(c.A, c.M, c.K, c.lda, c.es, &a0, &a1);
  if (c.layout == GEMM_B_ROW_MAJOR)
    extent(c.B, c.K, c.N, c.ldb, c.es, &b0, &b1);
  else
    extent(c.B, c.N, c.K, c.ldb, c.es, &b0, &b1);
  a1 += static_cast<uintptr_t>((nbat - 1) * c.bat.stride_a * c.es);
  b1 += static_cast<uintptr_t>((nbat - 1) * c.bat.stride_b * c.es);
  if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return GEMM_ERR_INVALID_VALUE;
  if (!is_device_memory(c.A, dev) || !is_device_memory(c.B, dev)) return GEMM_ERR_NOT_DEVICE_MEMORY;
  return GEMM_OK;
}

// K = 0: C = 0, or act(beta C + bias) with a fused epilogue, matrix by matrix.
int run_k_zero(const Call& c, const DeviceInfo* dev) {
  for (int64_t z = 0; z < c.bat.count; ++z) {
    void* Cz = static_cast<char*>(c.C) + z * c.bat.stride_c * c.eo;
    cudaError_t e;
    if (c.fused) {
      GemmParams ep;
      memset(&ep, 0, sizeof(ep));
      ep.alpha = c.epi->alpha;
      ep.beta = c.epi->beta;
      ep.bias = c.bias;
      ep.act = c.epi->activation;
      e = launch_epilogue_only(c.out_kind, Cz, c.ldc, int(c.M), int(c.N), ep, c.stream, dev->sm_count);
    } else {
      e = launch_fill_zero(Cz, c.ldc, int(c.M), int(c.N), c.eo, c.stream, dev->sm_count);
    }
    if (e != cudaSuccess) return GEMM_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return GEMM_OK;
}

// Threads of a launch. Pair kernels: 192 (TMA operands only). Single-CTA
// kernel: 320 when warps 6-9 are needed, to copy operand rows TMA cannot
// load or, for tiles of four or more 32-column chunks, to drain the
// accumulator as a second set of epilogue warps (GB300, BF16, CUDA graphs:
// 2048^3 15.03 -> 14.81 us, a batch of 512 products of 256^3 41.6 -> 39.6 us;
// narrower tiles ran slower with the extra warps: 512^3 5.04 -> 5.25 us).
int launch_threads(bool pair, bool all_tma, int bn) {
  if (pair) return 192;
  return (!all_tma || bn >= 128) ? 320 : 192;
}

// Operands as the kernel reads them, after any packing or transposition.
struct Operands {
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  int ga, gb;   // row granularity (16: TMA-addressable)
  bool kmajor;  // B K-major as read by the kernel
};

// Chooses the plan, sets up the stream's scratch ([counters][split partials]
// [packed A][packed B]), launches the packing / transposition copies, and
// fills the work-decomposition fields of p. Returns a status.
int prepare(const Call& c, const DeviceInfo* dev, int dev_id, TilePlan& plan, Operands& op, GemmParams& p) {
  const int es = c.es;
  const int64_t M = c.M, N = c.N, K = c.K, nbat = c.bat.count;
  op = Operands{c.A, c.lda, c.B, c.ldb, granularity(c.A, c.lda, es), granularity(c.B, c.ldb, es), false};
  if (nbat > 1) {
    // a batch is streamed by TMA in place: rows and matrix strides on 16-byte boundaries
    if (op.ga < 16 || op.gb < 16 || (c.bat.stride_a * es) % 16 != 0 || (c.bat.stride_b * es) % 16 != 0)
      return GEMM_ERR_MISALIGNED;
  }
  // The FP8 kernels read B K-major only: a row-major FP8 B is transposed into
  // the stream's scratch first (the packed-B slot), and from then on it is K-major.
  const bool transpose_b = c.fp8 && c.layout == GEMM_B_ROW_MAJOR;
  op.kmajor = c.layout == GEMM_B_K_MAJOR || transpose_b;
  // Operands whose rows TMA cannot address (row starts not 16-byte aligned)
  // are packed into 128-byte-aligned rows in the stream's scratch first (a
  // bandwidth-bound copy), so that the TMA kernels run; without scratch the
  // kernel's copy warps read them in place. In a large product an operand is
  // also packed when its rows are TMA-legal but do not start on 128-byte
  // boundaries: each 128-byte row of its boxes then straddles two L2 lines,
  // and the k-loop ran about a third slower (4000 x 4100 x 4104 on GB300). The
  // copy pays for itself once the other output dimension is a few thousand.
  // FP8 operands always go through TMA (the copy warps do not handle 1-byte
  // granules), so they are packed whenever they need it.
  const bool may_pack = nbat == 1 && c.ext == nullptr &&
                        (c.fp8 || !(g_debug_flags.load(std::memory_order_relaxed) & DEBUG_NO_PACK));
  auto off_line = [es](const void* ptr, int64_t ld) {
    return ((reinterpret_cast<uintptr_t>(ptr) | static_cast<uintptr_t>(ld * es)) % 128) != 0;
  };
  const bool big = 2.0 * double(M) * double(N) * double(K) >= 1.6e10;
  const bool pack_a = may_pack && (op.ga < 16 || (big && N >= 2048 && off_line(c.A, c.lda)));
  const bool pack_b = may_pack && (transpose_b || op.gb < 16 || (big && M >= 2048 && off_line(c.B, c.ldb)));
  plan = choose_plan(dev_id, c.kind, M, N, K, es, op.kmajor, (op.ga == 16 || pack_a) && (op.gb == 16 || pack_b),
                     dev->sm_count, nbat, c.fused);
  const int64_t lda_p = pack_a ? (K * es + 127) / 128 * 128 / es : c.lda;
  const int64_t b_rows = op.kmajor ? N : K, b_cols = op.kmajor ? K : N;  // of the operand the kernel reads
  const int64_t ldb_p = pack_b ? (b_cols * es + 127) / 128 * 128 / es : c.ldb;
  auto split_tiles = [&](const TilePlan& pl) {
    const int64_t ma = pl.swap ? N : M, nb_ext = pl.swap ? M : N;
    const int64_t tm = (ma + (pl.pair ? 255 : 127)) / (pl.pair ? 256 : 128);
    const int64_t tn = ((nb_ext + pl.bn - 1) / pl.bn + pl.pairs - 1) / pl.pairs;
    const int64_t r = (pl.pair && pl.segs > 1) ? (nbat * tm * tn) % pl.conc : 0;
    return (r > 0 && r <= 1024) ? int(r) : 0;
  };
  int rest = split_tiles(plan);
  const size_t split_bytes = rest ? workspace_bytes(rest, plan.segs, plan.bn, 2 * plan.pairs) : 0;
  const size_t off_a = (split_bytes + 255) / 256 * 256;
  const size_t off_b = off_a + (pack_a ? (size_t(M) * size_t(lda_p) * es + 255) / 256 * 256 : 0);
  const size_t total = off_b + (pack_b ? size_t(b_rows) * size_t(ldb_p) * es : 0);
  char* ws = nullptr;
  if (c.ext != nullptr) {
    if (rest) {
      if (split_bytes > c.ext->bytes) return GEMM_ERR_SCRATCH_LIMIT;
      ws = static_cast<char*>(c.ext->ptr);
    }
  } else if (total > 0) {
    ws = static_cast<char*>(stream_workspace(dev_id, c.stream, total < kCounterBytes ? kCounterBytes : total));
    if (ws == nullptr) {
      // no scratch: no split tail, and unaligned operands are read in place by the copy warps
      if (c.fp8 && (pack_a || pack_b)) return GEMM_ERR_LAUNCH;  // FP8 cannot do without the packed copy
      if (pack_a || pack_b)
        plan = choose_plan(dev_id, c.kind, M, N, K, es, op.kmajor, op.ga == 16 && op.gb == 16, dev->sm_count, nbat,
                           c.fused);
      rest = 0;
    }
  }
  // work decomposition: tiles along N count pairs of adjacent tiles for the
  // shared-A kernel (the second past the last column when the count is odd:
  // computed, not stored); the transposed product tiles C^T (N x M)
  const int64_t ma = plan.swap ? N : M, nb_ext = plan.swap ? M : N;
  const int64_t tiles_m = (ma + (plan.pair ? 255 : 127)) / (plan.pair ? 256 : 128);
  const int64_t tiles_n = ((nb_ext + plan.bn - 1) / plan.bn + plan.pairs - 1) / plan.pairs;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.tiles_m = int(tiles_m);
  p.tiles_n = int(tiles_n);
  p.batch = int(nbat);
  p.tiles_per_batch = int(tiles_m * tiles_n);
  p.num_tiles = int(nbat * tiles_m * tiles_n);
  p.stride_a = nbat > 1 ? c.bat.stride_a : 0;
  p.stride_b = nbat > 1 ? c.bat.stride_b : 0;
  p.stride_c = nbat > 1 ? c.bat.stride_c : 0;
  p.num_kb = int((K * es + 127) / 128);
  p.raster = plan.raster;
  p.tail_start = p.num_tiles;
  p.tail_segs = 1;
  p.num_work = p.num_tiles;
  if (ws != nullptr && rest > 0) {
    p.tail_segs = plan.segs;
    p.tail_start = p.num_tiles - rest;
    p.num_work = p.tail_start + rest * plan.segs;
    p.ws_ctr = reinterpret_cast<unsigned long long*>(ws);
    p.ws = reinterpret_cast<float*>(ws + kCounterBytes);
    p.ws_slots = static_cast<long long>(rest) * plan.segs * 2 * plan.pairs;
  }
  if (ws != nullptr && (pack_a || pack_b)) {
    // one launch packs both operands (a row-major FP8 B is transposed instead)
    PackSpec spec[2];
    int n = 0;
    if (pack_a) spec[n++] = PackSpec{c.A, c.lda * es, ws + off_a, lda_p * es, M, K * es, op.ga};
    if (pack_b && !transpose_b) spec[n++] = PackSpec{c.B, c.ldb * es, ws + off_b, ldb_p * es, b_rows, b_cols * es, op.gb};
    if (n > 0 && launch_pack(spec, n, c.stream, dev->sm_count) != cudaSuccess) return GEMM_ERR_LAUNCH;
    if (pack_b && transpose_b &&
        launch_transpose_bytes(c.B, c.ldb, ws + off_b, ldb_p, K, N, c.stream, dev->sm_count) != cudaSuccess)
      return GEMM_ERR_LAUNCH;
    if (pack_a) {
      op.A = ws + off_a;
      op.lda = lda_p;
      op.ga = 16;
    }
    if (pack_b) {
      op.B = ws + off_b;
      op.ldb = ldb_p;
      op.gb = 16;
    }
  }
  if (plan.pair && !(op.ga == 16 && op.gb == 16)) return GEMM_ERR_LAUNCH;  // the pair kernel needs TMA operands
  return GEMM_OK;
}

// The tensor maps of A, B (and the last, narrower B box) and C.
int encode_maps(const Call& c, const TilePlan& plan, const Operands& op, LaunchPlan& L) {
  const GemmParams& p = L.p;
  const int es = c.es, eo = c.eo, bn = plan.bn;
  const uint64_t nbat = uint64_t(c.bat.count);
  const CUtensorMapDataType dt = c.kind == KIND_TF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : c.kind == KIND_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : c.kind == KIND_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType dt_out = c.fp8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : dt;
  const uint32_t bk = 128 / es;  // K elements per 128-byte row
  const uint64_t za = p.stride_a ? nbat : 1, zb = p.stride_b ? nbat : 1;
  const uint64_t M = uint64_t(c.M), N = uint64_t(c.N), K = uint64_t(c.K);
  // A box: 128 rows, or 64 where two pairs each load half a CTA's rows for
  // both, or (transposed product) the bn / 2 rows of C a CTA computes
  const uint32_t a_rows = plan.swap ? uint32_t(bn / 2) : (plan.pair && plan.pairs == 2) ? 64u : 128u;
  if (p.a_tma && !encode_3d(&L.tmA, dt, op.A, K, M, uint64_t(op.lda) * es, za, uint64_t(p.stride_a) * es, bk, a_rows))
    return GEMM_ERR_DRIVER;
  if (p.b_tma) {
    bool ok;
    if (plan.swap) {
      // B^T as the MMA's MN-major A operand: whole 128-byte boxes of 128 / es columns
      const CUtensorMapSwizzle swz = es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
      ok = encode_3d(&L.tmB, dt, op.B, N, K, uint64_t(op.ldb) * es, zb, uint64_t(p.stride_b) * es, 128 / es, bk, swz);
    } else if (op.kmajor) {
      ok = encode_3d(&L.tmB, dt, op.B, K, N, uint64_t(op.ldb) * es, zb, uint64_t(p.stride_b) * es, bk,
                     uint32_t(plan.pair ? bn / 2 : bn));
    } else {
      const CUtensorMapSwizzle swz = es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
      ok = encode_3d(&L.tmB, dt, op.B, N, K, uint64_t(op.ldb) * es, zb, uint64_t(p.stride_b) * es, 128 / es, bk, swz);
      // the last box of a tile whose columns per CTA are not whole 128-byte boxes
      const int cols = plan.pair ? bn / 2 : bn, boxn = 128 / es;
      const int lastn = cols - (cols + boxn - 1) / boxn * boxn + boxn;
      if (ok && lastn != boxn)
        ok = encode_3d(&L.tmB2, dt, op.B, N, K, uint64_t(op.ldb) * es, zb, uint64_t(p.stride_b) * es,
                       uint32_t(lastn), bk, swz);
    }
    if (!ok) return GEMM_ERR_DRIVER;
  }
  // C box: 32 rows x 64 bytes, the staging tile of one epilogue warp (64-byte swizzle)
  if (p.c_tma && !encode_3d(&L.tmC, dt_out, c.C, N, M, uint64_t(c.ldc) * eo, p.stride_c ? nbat : 1,
                            uint64_t(p.stride_c) * eo, uint32_t(64 / eo), 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return GEMM_ERR_DRIVER;
  return GEMM_OK;
}

int run_gemm(int kind, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
             void* C, int64_t ldc, int layout, void* stream_ptr, const ExternalScratch* ext = nullptr,
             const gemm_epilogue_t* epi = nullptr, const Batch& bat = Batch()) {
  Call c;
  c.kind = kind;
  c.fp8 = kind == KIND_E4M3 || kind == KIND_E5M2;
  c.es = (kind == KIND_TF32) ? 4 : c.fp8 ? 1 : 2;
  c.eo = (kind == KIND_TF32) ? 4 : 2;
  c.out_kind = c.fp8 ? int(KIND_BF16) : kind;
  c.M = M;
  c.N = N;
  c.K = K;
  c.A = A;
  c.lda = lda;
  c.B = B;
  c.ldb = ldb;
  c.C = C;
  c.ldc = ldc;
  c.layout = layout;
  c.bat = bat;
  c.epi = epi;
  c.fused = epi != nullptr && !(epi->alpha == 1.0f && epi->beta == 0.0f && epi->bias == nullptr &&
                                epi->activation == GEMM_ACT_NONE);
  c.bias = c.fused ? epi->bias : nullptr;
  c.stream = static_cast<cudaStream_t>(stream_ptr);
  c.ext = ext;

  int st = check_arguments(c);
  if (st != GEMM_OK || M == 0 || N == 0 || bat.count == 0) return st;
  const DeviceInfo* dev = nullptr;
  int dev_id = 0;
  st = current_device(&dev, &dev_id);
  if (st != GEMM_OK) return st;
  st = check_memory(c, dev_id);
  if (st != GEMM_OK) return st;
  if (K == 0) return run_k_zero(c, dev);

  LaunchPlan L;
  memset(&L, 0, sizeof(L));
  GemmParams& p = L.p;
  TilePlan plan;
  Operands op;
  st = prepare(c, dev, dev_id, plan, op, p);
  if (st != GEMM_OK) return st;
  p.A = op.A;
  p.lda = op.lda;
  p.B = op.B;
  p.ldb = op.ldb;
  p.C = C;
  p.ldc = ldc;
  p.a_tma = op.ga == 16;
  p.b_tma = op.gb == 16;
  p.copy_bytes = 16;
  if (!p.a_tma) p.copy_bytes = op.ga;
  if (!p.b_tma && op.gb < p.copy_bytes) p.copy_bytes = op.gb;
  // widest access that every C element's address allows: base, row pitch and
  // (in a batch) the matrix stride, which offsets every matrix after the first
  p.c_gran = granularity(C, ldc, c.eo);
  if (p.stride_c != 0) {
    const int gs = granularity(nullptr, p.stride_c, c.eo);
    if (gs < p.c_gran) p.c_gran = gs;
  }
  // TMA stores of C need 16-byte rows, base and (in a batch) matrix stride; else row stores
  p.c_tma = p.c_gran == 16;
  p.status = dev->status_words;
  uint32_t ep = g_epoch.fetch_add(1, std::memory_order_relaxed);
  if (ep == 0) ep = g_epoch.fetch_add(1, std::memory_order_relaxed);
  p.epoch = ep;
  p.debug = g_debug_flags.load(std::memory_order_relaxed);
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.fused = c.fused ? 1 : 0;
  if (c.fused) {
    p.alpha = epi->alpha;
    p.beta = epi->beta;
    p.bias = c.bias;
    p.act = epi->activation;
  }
  st = encode_maps(c, plan, op, L);
  if (st != GEMM_OK) return st;
  L.b_kmajor = op.kmajor;
  L.pair = plan.pair;
  L.swap = plan.swap;
  L.pairs = plan.pairs;
  L.bn = plan.bn;
  L.grid = plan.grid;
  L.threads = launch_threads(plan.pair, p.a_tma && p.b_tma, plan.bn);
  L.stream = c.stream;
  L.dev = dev_id;

  // internal consistency of the derived launch parameters (a violation is a library bug)
  if (p.raster < 1 || p.num_kb < 1 || p.num_tiles < 1 || p.num_work < p.num_tiles || p.tail_segs < 1 ||
      p.tail_segs > kMaxTailSegs || L.grid < 1 || (L.pair && (L.grid % (2 * L.pairs) != 0)) || p.tiles_n < 1 ||
      p.tiles_m < 1 || (L.pair && L.pairs != 1 && L.pairs != 2) || (!L.pair && L.pairs != 1) ||
      (L.pair && L.threads != 192))
    return GEMM_ERR_LAUNCH;
  if (c.fp8 && !(p.a_tma && p.b_tma && op.kmajor)) return GEMM_ERR_LAUNCH;  // guaranteed by prepare()
  if (L.swap && !(L.pair && L.pairs == 1 && !op.kmajor && !c.fp8)) return GEMM_ERR_LAUNCH;  // choose_plan's rule
  cudaError_t e;
  switch (kind) {
    case KIND_TF32: e = L.swap ? launch_tf32_sw(L) : op.kmajor ? launch_tf32_km(L) : launch_tf32_rm(L); break;
    case KIND_BF16: e = L.swap ? launch_bf16_sw(L) : op.kmajor ? launch_bf16_km(L) : launch_bf16_rm(L); break;
    case KIND_F16: e = L.swap ? launch_f16_sw(L) : op.kmajor ? launch_f16_km(L) : launch_f16_rm(L); break;
    case KIND_E4M3: e = launch_e4m3_km(L); break;
    default: e = launch_e5m2_km(L); break;
  }
  if (e != cudaSuccess) return GEMM_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  const int32_t info[8] = {plan.swap ? 3 : plan.pair ? 2 * plan.pairs : 1, plan.bn, p.raster, L.grid, p.tail_segs,
                           plan.conc,
                           p.tail_start, p.num_work};
  memcpy(t_last_plan, info, sizeof(info));
  return GEMM_OK;
}

}  // namespace

cudaError_t launch_pack(const PackSpec* specs, int n, cudaStream_t stream, int sm_count) {
  PackJob job[2] = {};
  long long tasks[2] = {0, 0};
  for (int i = 0; i < n && i < 2; ++i) {
    const PackSpec& q = specs[i];
    const long long chunks = (q.row_bytes + 15) / 16;
    job[i] = PackJob{static_cast<const uint8_t*>(q.src), (long long)q.src_ld_bytes, static_cast<uint8_t*>(q.dst),
                     (long long)q.dst_ld_bytes, (long long)q.row_bytes,
                     (chunks + kPackSegChunks - 1) / kPackSegChunks, q.gran};
    tasks[i] = job[i].segs_per_row * q.rows;
  }
  if (n < 2) job[1] = job[0];
  const long long total = tasks[0] + tasks[1];
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 7) / 8;  // eight warps (tasks) per block, four blocks per SM
  if (blocks > 4LL * sm_count) blocks = 4LL * sm_count;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(unsigned(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pack_rows_kernel, job[0], job[1], tasks[0], total);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

int run_gemm_external(int kind, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                      int64_t ldb, void* C, int64_t ldc, int layout, void* stream, const ExternalScratch* ext) {
  return run_gemm(kind, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, ext);
}

cudaError_t launch_epilogue_only(int kind, void* C, long long ldc, int M, int N, const GemmParams& p,
                                 cudaStream_t stream, int sm_count) {
  const long long total = static_cast<long long>(M) * N;
  long long blocks = (total + 255) / 256;
  if (blocks > 4LL * sm_count) blocks = 4LL * sm_count;
  if (kind == KIND_TF32)
    epilogue_only_kernel<KIND_TF32><<<int(blocks), 256, 0, stream>>>(C, ldc, M, N, p.alpha, p.beta, p.bias, p.act);
  else if (kind == KIND_BF16)
    epilogue_only_kernel<KIND_BF16><<<int(blocks), 256, 0, stream>>>(C, ldc, M, N, p.alpha, p.beta, p.bias, p.act);
  else
    epilogue_only_kernel<KIND_F16><<<int(blocks), 256, 0, stream>>>(C, ldc, M, N, p.alpha, p.beta, p.bias, p.act);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bytes(const void* src, int64_t src_ld, void* dst, int64_t dst_ld, int64_t rows,
                                   int64_t cols, cudaStream_t stream, int sm_count) {
  const long long tiles = ((rows + 63) / 64) * ((cols + 63) / 64);
  long long blocks = tiles < 8LL * sm_count ? tiles : 8LL * sm_count;
  // 4-byte source words where every row start is 4-byte aligned
  const int words = ((reinterpret_cast<uintptr_t>(src) | static_cast<uintptr_t>(src_ld)) % 4) == 0;
  transpose_bytes_kernel<<<int(blocks), 256, 0, stream>>>(static_cast<const uint8_t*>(src), src_ld,
                                                          static_cast<uint8_t*>(dst), dst_ld, int(rows), int(cols),
                                                          words);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

cudaError_t launch_fill_zero(void* C, long long ldc, int M, int N, int es, cudaStream_t stream, int sm_count) {
  const long long total = static_cast<long long>(M) * N;
  long long blocks = (total + 255) / 256;
  if (blocks > 4LL * sm_count) blocks = 4LL * sm_count;
  if (es == 4)
    fill_zero_kernel<4><<<int(blocks), 256, 0, stream>>>(C, ldc, M, N);
  else
    fill_zero_kernel<2><<<int(blocks), 256, 0, stream>>>(C, ldc, M, N);
  return cudaGetLastError();
}

}  // namespace dgt

extern "C" {

int gemm_tf32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
              int64_t ldc, int layout, void* stream) {
  return dgt::run_gemm(dgt::KIND_TF32, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}

int gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
             uint16_t* C, int64_t ldc, int layout, void* stream) {
  return dgt::run_gemm(dgt::KIND_F16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}

int gemm_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, void* stream) {
  return dgt::run_gemm(dgt::KIND_BF16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream);
}

int gemm_tf32_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                              int64_t stride_a, const float* B, int64_t ldb, int64_t stride_b, float* C, int64_t ldc,
                              int64_t stride_c, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  const dgt::Batch b{batch, stride_a, stride_b, stride_c};
  return dgt::run_gemm(dgt::KIND_TF32, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue, b);
}

int gemm_f16_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                             int64_t stride_a, const uint16_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                             int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                             void* stream) {
  const dgt::Batch b{batch, stride_a, stride_b, stride_c};
  return dgt::run_gemm(dgt::KIND_F16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue, b);
}

int gemm_bf16_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                              int64_t stride_a, const uint16_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream) {
  const dgt::Batch b{batch, stride_a, stride_b, stride_c};
  return dgt::run_gemm(dgt::KIND_BF16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue, b);
}

int gemm_e4m3_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                              int64_t stride_a, const uint8_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream) {
  const dgt::Batch b{batch, stride_a, stride_b, stride_c};
  return dgt::run_gemm(dgt::KIND_E4M3, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue, b);
}

int gemm_e5m2_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                              int64_t stride_a, const uint8_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream) {
  const dgt::Batch b{batch, stride_a, stride_b, stride_c};
  return dgt::run_gemm(dgt::KIND_E5M2, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue, b);
}

int gemm_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  return dgt::run_gemm(dgt::KIND_E4M3, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue);
}

int gemm_e5m2(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  return dgt::run_gemm(dgt::KIND_E5M2, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue);
}

int gemm_tf32_ex(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
                 int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  return dgt::run_gemm(dgt::KIND_TF32, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue);
}

int gemm_f16_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  return dgt::run_gemm(dgt::KIND_F16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue);
}

int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                 uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream) {
  return dgt::run_gemm(dgt::KIND_BF16, M, N, K, A, lda, B, ldb, C, ldc, layout, stream, nullptr, epilogue);
}

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_VALUE: return "invalid argument (size, leading dimension, layout, NULL or overlap)";
    case GEMM_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103)";
    case GEMM_ERR_LAUNCH: return "CUDA launch or synchronisation failed";
    case GEMM_ERR_NOT_DEVICE_MEMORY: return "pointer is not device memory of the current device";
    case GEMM_ERR_DRIVER: return "tensor-map encoding failed in the CUDA driver";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a kernel exceeded its wait time limit and gave up";
    case GEMM_ERR_SCRATCH_LIMIT: return "the shape needs more scratch than the fixed scratch array holds";
    default: return "unknown status";
  }
}

int gemm_get_device_status(void* stream, uint32_t* out) {
  if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
  const dgt::DeviceInfo* dev = nullptr;
  int st = dgt::current_device(&dev);
  if (st != GEMM_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_LAUNCH;
  uint32_t w[2] = {0, 0};
  if (cudaMemcpy(w, dev->status_words, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_LAUNCH;
  *out = w[0];
  return w[0] ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}

int gemm_reset_device_status(void) {
  const dgt::DeviceInfo* dev = nullptr;
  int st = dgt::current_device(&dev);
  if (st != GEMM_OK) return st;
  if (cudaMemset(dev->status_words, 0, 2 * sizeof(uint32_t)) != cudaSuccess) return GEMM_ERR_LAUNCH;
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}

int gemm_set_debug(uint32_t flags, uint64_t wait_limit_ns) {
  dgt::g_debug_flags.store(flags);
  dgt::g_wait_limit_ns.store(wait_limit_ns ? wait_limit_ns : dgt::kDefaultWaitLimitNs);
  return GEMM_OK;
}

uint64_t gemm_launch_count(void) { return dgt::g_launches.load(); }

int gemm_free_workspaces(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_LAUNCH;
  dgt::free_workspaces();
  return dgt::free_host_buffers();
}

int gemm_last_plan(int32_t* out) {
  if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
  memcpy(out, dgt::t_last_plan, sizeof(dgt::t_last_plan));
  return GEMM_OK;
}

int gemm_plan_query(int kind, int64_t M, int64_t N, int64_t K, int layout, int64_t batch, int fused, int sms,
                    int pair_clusters, int quad_clusters, int32_t* out) {
  if (out == nullptr || kind < dgt::KIND_F16 || kind > dgt::KIND_E5M2 || M < 1 || N < 1 || K < 1 || batch < 1 ||
      (layout != GEMM_B_ROW_MAJOR && layout != GEMM_B_K_MAJOR) || sms < 2 || pair_clusters < 1 || quad_clusters < 1)
    return GEMM_ERR_INVALID_VALUE;
  const bool fp8 = kind == dgt::KIND_E4M3 || kind == dgt::KIND_E5M2;
  const int es = kind == dgt::KIND_TF32 ? 4 : fp8 ? 1 : 2;
  const bool kmajor = layout == GEMM_B_K_MAJOR || fp8;  // a row-major FP8 B is transposed first
  const dgt::TilePlan plan = dgt::choose_plan(-1, kind, M, N, K, es, kmajor, true, sms, batch, fused != 0,
                                              pair_clusters, quad_clusters);
  const int32_t info[6] = {plan.swap ? 3 : plan.pair ? 2 * plan.pairs : 1, plan.bn, plan.raster, plan.grid,
                           plan.segs, plan.conc};
  memcpy(out, info, sizeof(info));
  return GEMM_OK;
}

int gemm_set_tuning(int variant, int tile_n, int raster, int tail_split) {
  if (variant < 0 || variant > 4 || raster < 0 || tail_split < 0 || tail_split > 2) return GEMM_ERR_INVALID_VALUE;
  if (tile_n != 0) {
    bool ok = false;
    if (variant < 2)
      for (int w : dgt::kTileWidths) ok = ok || (w == tile_n);
    if (variant != 1)
      for (int w : dgt::kPairTileWidths) ok = ok || (w == tile_n);
    if (!ok) return GEMM_ERR_INVALID_VALUE;
  }
  dgt::g_force_variant.store(variant);
  dgt::g_force_bn.store(tile_n);
  dgt::g_force_raster.store(raster);
  dgt::g_force_split.store(tail_split);
  return GEMM_OK;
}

}  // extern "C"
