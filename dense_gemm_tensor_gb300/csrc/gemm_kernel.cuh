// Persistent, warp-specialised dense GEMM for sm_103a:  C (M x N) = A (M x K) . B (K x N).
//
// The method is the dense matrix product of the TF32 and FP16/BF16 GEMM pages
// ("sgemm tf32 - beating cuBLAS" and "hgemm - beating cuBLAS"): block tiling
// with operands staged through shared memory, a pipelined k-loop, tensor-core
// MMA with fp32 accumulation, grid-swizzled tile order for L2 reuse, and an
// epilogue that converts the fp32 accumulator to the output type with
// round-to-nearest-even. Here each of those steps is a Blackwell unit; this
// file holds the single-CTA kernel and what both kernels share (the CTA-pair
// kernel is in gemm_kernel_pair.cuh):
//
//   * one CTA per SM loops over output tiles of BM x BN = 128 x (256, 224,
//     192 or 128) in a banded order (the pages' grid swizzle, generalised to
//     ragged grids and to strided batches of products);
//   * warp 4 streams A and B boxes with TMA (3-D tensor maps: the batch's
//     matrix is the outer coordinate) into a ring of 128-byte-swizzled
//     shared-memory stages (the hardware swizzle replaces the pages'
//     hand-derived XOR layouts); for an operand whose rows TMA cannot address
//     (row pitch not a multiple of 16 bytes) and that was not packed, warps
//     6-9 copy it with cp.async into the same swizzled image;
//   * warp 5 issues tcgen05.mma 128 x BN x (32 bytes of K) -- kind::f16,
//     kind::tf32 or kind::f8f6f4 -- into one of two accumulators in tensor
//     memory, so the epilogue of one tile overlaps the k-loop of the next;
//   * warps 0-3 read the accumulator with tcgen05.ld (warp w owns TMEM lanes
//     32w..32w+31 = tile rows), apply the optional fused epilogue, convert,
//     stage 32 x 64-byte pieces in shared memory and store them with TMA.
//
// Every wait on an mbarrier is bounded: past the launch's time limit the
// waiting thread records a timeout in the device status word and the CTA
// winds down (in-flight copies and MMAs are drained, TMEM is freed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "ptx.cuh"

// A checked build (-DDGT_CHECKED=1) tests, before each shared-memory, tensor
// memory, TMA-coordinate and scratch access the kernels compute, that it lies
// in its range; a failing access is skipped and recorded in the device status
// word (kind 3, the site in bits 4-11), where compute-sanitizer cannot run.
// The default build compiles every check away.
#ifndef DGT_CHECKED
#define DGT_CHECKED 0
#endif

// Geometry of the 32-byte-atom swizzle (MN-major 32-bit operands): stride
// between K-row groups in the descriptor, and which row bits select the
// XOR pattern of the 32-byte chunks.
#ifndef DGT_ATOM32_SBO
#define DGT_ATOM32_SBO 512
#endif
#ifndef DGT_ATOM32_ROWSHIFT
#define DGT_ATOM32_ROWSHIFT 0
#endif

namespace dgt {

// Operand kinds. The FP8 kinds (OCP E4M3 and E5M2 bytes) accumulate in fp32
// like the others and write a bfloat16 C.
enum Kind : int { KIND_F16 = 0, KIND_BF16 = 1, KIND_TF32 = 2, KIND_E4M3 = 3, KIND_E5M2 = 4 };

template <int KIND>
struct KindTraits;
template <>
struct KindTraits<KIND_F16> {
  using T = __half;
  static constexpr uint32_t fmt = 0;  // instruction-descriptor operand format F16 (kind::f16)
  static constexpr int out = KIND_F16;
};
template <>
struct KindTraits<KIND_BF16> {
  using T = __nv_bfloat16;
  static constexpr uint32_t fmt = 1;  // BF16 (kind::f16)
  static constexpr int out = KIND_BF16;
};
template <>
struct KindTraits<KIND_TF32> {
  using T = float;
  static constexpr uint32_t fmt = 2;  // TF32 (kind::tf32)
  static constexpr int out = KIND_TF32;
};
template <>
struct KindTraits<KIND_E4M3> {
  using T = uint8_t;
  static constexpr uint32_t fmt = 0;  // E4M3 (kind::f8f6f4)
  static constexpr int out = KIND_BF16;
};
template <>
struct KindTraits<KIND_E5M2> {
  using T = uint8_t;
  static constexpr uint32_t fmt = 1;  // E5M2 (kind::f8f6f4)
  static constexpr int out = KIND_BF16;
};

// One tcgen05.mma of the kind's instruction family (single CTA / CTA pair).
template <int KIND>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (KIND == KIND_TF32)
    mma_tf32(d, a, b, idesc, acc);
  else if constexpr (KIND == KIND_E4M3 || KIND == KIND_E5M2)
    mma_f8f6f4(d, a, b, idesc, acc);
  else
    mma_f16(d, a, b, idesc, acc);
}
template <int KIND>
__device__ __forceinline__ void mma_issue_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (KIND == KIND_TF32)
    mma_tf32_pair(d, a, b, idesc, acc);
  else if constexpr (KIND == KIND_E4M3 || KIND == KIND_E5M2)
    mma_f8f6f4_pair(d, a, b, idesc, acc);
  else
    mma_f16_pair(d, a, b, idesc, acc);
}

// Status word codes (device status[0]); status[1] holds the epoch of the last aborted launch.
enum : uint32_t {
  STATUS_TIMEOUT = 1u,
  STATUS_OUT_OF_RANGE = 3u,  // a checked build skipped an access outside its range
  ROLE_PRODUCER = 1u << 4,
  ROLE_MMA = 2u << 4,
  ROLE_EPILOGUE = 3u << 4,
  ROLE_COPY = 4u << 4,
  ROLE_TEARDOWN = 5u << 4,
};
enum : uint32_t {
  DEBUG_STALL_PRODUCER = 1u,
  DEBUG_NO_PACK = 2u,  // host: copy unaligned operands with the kernel's copy warps instead of packing them
};

struct GemmParams {
  int M, N, K;
  // Strided batch: matrix z of A, B, C starts stride_{a,b,c} elements after
  // matrix z-1 (a stride of 0 repeats one matrix); batch = 1 for one product.
  // Work tiles run batch by batch: tile t belongs to matrix t / tiles_per_batch.
  int batch, tiles_per_batch;
  long long stride_a, stride_b, stride_c;
  int tiles_m, tiles_n, num_tiles, num_kb;
  int raster;  // band height (in tiles along M) of the tile order
  // Work items: tiles [0, tail_start) in tile order, whole; each tile from
  // tail_start on is split into tail_segs ranges of k-slabs (the last partial
  // round of tiles spread over more SMs). num_work counts the items. The
  // segments' fp32 partial tiles meet in `ws`; `ws_ctr` holds one arrival
  // counter per (split tile, CTA of the pair), tagged with the launch epoch.
  int tail_start, tail_segs, num_work;
  float* ws;
  unsigned long long* ws_ctr;
  const void* A;
  long long lda;
  const void* B;
  long long ldb;
  void* C;
  long long ldc;
  int a_tma, b_tma;  // operand loaded by TMA (1) or by the copy warps (0)
  int copy_bytes;    // copy-warp granularity in bytes: 16, 8, 4 or 2
  int c_tma;         // C written by TMA stores (base and row pitch are 16-byte multiples)
  int c_gran;        // widest store (bytes: 16, 8, 4 or 2) the C base and row pitch allow
  uint32_t* status;  // device status words [2]
  uint32_t epoch;    // unique per launch
  uint32_t debug;
  unsigned long long wait_limit_ns;
  // Fused epilogue (fused != 0): C = act(alpha * A.B + beta * C + bias[col]),
  // evaluated in fp32; beta == 0 leaves C unread; bias (N elements of the
  // output type) may be null; act is a GEMM_ACT_* code.
  int fused;
  int act;
  float alpha, beta;
  const void* bias;
  long long ws_slots;  // fp32 partial tiles the split-tail scratch holds (range checks of a checked build)
};

// Arrival counters of split tiles the scratch holds: one per CTA of a cluster
// of up to four, for up to 1024 split work tiles.
constexpr int kSplitCounters = 1024 * 4;

// Sites of the checked build's range checks (status bits 4-11).
enum : uint32_t {
  CHECK_A_STAGE = 1u,     // TMA destination of an A box inside its stage
  CHECK_B_STAGE = 2u,     // TMA destination of a B box inside its stage
  CHECK_TMA_X = 3u,       // innermost TMA coordinate on a 16-byte boundary
  CHECK_ACC_COLS = 4u,    // accumulator columns inside the allocated tensor memory
  CHECK_DESC = 5u,        // MMA operand descriptors inside the stage
  CHECK_STAGING = 6u,     // epilogue staging tile inside the warp's ring
  CHECK_TMEM_LD = 7u,     // tensor-memory columns the epilogue reads
  CHECK_SPLIT_SLOT = 8u,  // fp32 partial tile inside the scratch
  CHECK_SPLIT_CTR = 9u,   // arrival counter inside the scratch
};

// Output staging in shared memory (see epi_chunk_addr): each epilogue warp
// has a ring of 1-4 tiles of 2 KB (EPI_BYTES = one tile for each of the four
// warps); the shared memory the operand stages leave over sets the count.
constexpr int EPI_WARP_BYTES = 32 * 64;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;

// Staging tiles needed per warp, given what a kernel's stages leave of `limit`.
constexpr int epi_bufs_for(int limit, int used) {
  return (limit - used) / EPI_BYTES >= 4 ? 4 : (limit - used) / EPI_BYTES < 1 ? 1 : (limit - used) / EPI_BYTES;
}

// A warp's staging ring: round i writes tile i mod bufs.
struct EpiRing {
  uint32_t base;  // this warp's first tile
  int bufs;
  int next;
  uint32_t end;   // end of the staging area (range checks of a checked build)
};

template <int KIND, bool B_KMAJOR, int BN_>
struct Cfg {
  using T = typename KindTraits<KIND>::T;
  static constexpr int ES = sizeof(T);
  static constexpr int BM = 128;
  static constexpr int BN = BN_;            // output tile width (multiple of 32, <= 256)
  static constexpr int BK = 128 / ES;       // one 128-byte swizzle row of K per stage
  static constexpr int UK = 32 / ES;        // K of one tcgen05.mma (16 for 16-bit, 8 for tf32)
  static constexpr int KSTEPS = BK / UK;    // MMAs per stage
  static constexpr int A_BYTES = BM * 128;  // 16 KB
  static constexpr int BOXN = 128 / ES;     // MN-major B: N elements per 128-byte box row
  static constexpr int NBOX = (BN + BOXN - 1) / BOXN;  // MN-major B: boxes per stage (last may be partly used)
  static constexpr int BOX_BYTES = BK * 128;
  static constexpr int B_BYTES = B_KMAJOR ? BN * 128 : NBOX * BOX_BYTES;
  // MN-major B: the last box carries only the tile's columns (see the pair kernel)
  static constexpr int LASTN = BN - (NBOX - 1) * BOXN;
  static constexpr int B_TX = B_KMAJOR ? B_BYTES : (NBOX - 1) * BOX_BYTES + LASTN * BK * ES;
  // MN-major B of 32-bit elements uses the 128-byte swizzle with 32-byte
  // atoms (16-bit MN-major and every K-major tile use 16-byte atoms).
  static constexpr bool B_ATOM32 = (ES == 4) && !B_KMAJOR;
  static constexpr uint32_t B_SWZ = B_ATOM32 ? SWZ_128B_ATOM32 : SWZ_128B;
  static constexpr uint32_t B_SBO = B_ATOM32 ? DGT_ATOM32_SBO : 1024;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM_LIMIT = 232448;  // opt-in dynamic shared memory per block
  static constexpr int STAGES_FIT = (SMEM_LIMIT - (1024 + EPI_BYTES + 256)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int EPI_BUFS = epi_bufs_for(SMEM_LIMIT, 1024 + 256 + STAGES * STAGE_BYTES);
  static constexpr int RESERVED = 1024 /*align slack*/ + EPI_BUFS * EPI_BYTES /*output staging*/ + 256 /*barriers*/;
  static constexpr int ACC_COLS = BN;       // fp32 accumulator columns of one buffer
  static constexpr int TMEM_COLS = (2 * BN <= 256) ? 256 : 512;  // power of two >= 2 * BN
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + RESERVED;
  static constexpr int COPY_LAG = 2;        // stages a copy warp keeps in flight before signalling
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(NUM_BARS * 8 + 16 <= 256, "barrier area");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");

  // Instruction descriptor: D fp32, A/B format, A K-major, B K- or MN-major, N, M.
  static constexpr uint32_t IDESC = (1u << 4) | (KindTraits<KIND>::fmt << 7) | (KindTraits<KIND>::fmt << 10) |
                                    ((B_KMAJOR ? 0u : 1u) << 16) | (uint32_t(BN >> 3) << 17) |
                                    (uint32_t(BM >> 4) << 24);
};

// Linear work id -> output tile (mb, nb) of matrix bz of the batch. Within a
// matrix, tiles go in bands of `raster` tile-rows: down the band's rows
// first, then across N, band after band. A band's B tiles and its A
// row-tiles stay in L2 while the band is worked on.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb, int& bz) {
  bz = t / p.tiles_per_batch;
  t -= bz * p.tiles_per_batch;
  const int band = p.raster * p.tiles_n;
  const int g = t / band;
  const int first_m = g * p.raster;
  const int rows = min(p.raster, p.tiles_m - first_m);
  const int r = t - g * band;
  mb = first_m + r % rows;
  nb = r / rows;
}

static __device__ __noinline__ void record_out_of_range(const GemmParams& p, uint32_t site) {
  atomicCAS(p.status, 0u, STATUS_OUT_OF_RANGE | ((site & 0xFFu) << 4) | ((blockIdx.x & 0xFFFFu) << 16));
  atomicExch(p.status + 1, p.epoch);  // the launch winds down like one that timed out
  __threadfence();
}

// true when the access may go ahead; in a checked build a false `ok` is recorded.
__device__ __forceinline__ bool in_range(const GemmParams& p, bool ok, uint32_t site) {
  if constexpr (DGT_CHECKED != 0) {
    if (!ok) record_out_of_range(p, site);
    return ok;
  } else {
    return true;
  }
}

static __device__ __noinline__ void record_timeout(const GemmParams& p, uint32_t code) {
  atomicCAS(p.status, 0u, code | STATUS_TIMEOUT | ((blockIdx.x & 0xFFFFu) << 16));
  atomicExch(p.status + 1, p.epoch);
  __threadfence();
}

// Bounded wait for the phase of `bar` with `parity`. Returns false when this
// launch has been aborted (by this thread's own time limit or another's).
__device__ __forceinline__ bool wait_phase(const GemmParams& p, uint32_t bar, uint32_t parity, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (ld_volatile_u32(p.status + 1) == p.epoch) return false;
      if (globaltimer_ns() - t0 > p.wait_limit_ns) {
        record_timeout(p, code);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ bool wait_phase_drain(const GemmParams& p, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > p.wait_limit_ns) {
      record_timeout(p, ROLE_TEARDOWN);
      return false;
    }
  }
  return true;
}

// Warp-uniform version: lane 0 waits, the outcome is broadcast.
__device__ __forceinline__ bool warp_wait_phase(const GemmParams& p, uint32_t bar, uint32_t parity, uint32_t code) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_phase(p, bar, parity, code) ? 1u : 0u;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// ------------------------------------------------------------------ copy warps
// Copy one G-byte piece (G = 16, 8, 4: cp.async; 2: a plain load and store)
// from global to a swizzled shared-memory position; `valid` bytes come from
// memory, the rest are zero.
template <int G>
__device__ __forceinline__ void copy_chunk(uint32_t dst, const uint8_t* src, int valid) {
  if constexpr (G == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid) : "memory");
  } else if constexpr (G == 8) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(valid) : "memory");
  } else if constexpr (G == 4) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid) : "memory");
  } else {
    uint16_t v = 0;
    if (valid >= 2) v = *reinterpret_cast<const uint16_t*>(src);
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(dst), "h"(v) : "memory");
  }
}

// Byte position of `byte` (0..127) of row `k` inside a 128-byte-swizzled
// tile: 16-byte chunks XOR (k mod 8), or 32-byte chunks XOR the row bits the
// 32-byte-atom mode uses.
template <bool ATOM32>
__device__ __forceinline__ uint32_t swz_pos(int k, int byte) {
  if constexpr (ATOM32)
    return (((byte >> 5) ^ ((k >> DGT_ATOM32_ROWSHIFT) & 3)) << 5) | (byte & 31);
  else
    return (((byte >> 4) ^ (k & 7)) << 4) | (byte & 15);
}

// `n` 128-byte rows of a swizzled tile (row r of the tile at sdst + r * 128)
// from global rows grow0 + r, bytes [colb, colb + 128) of each: rows at or
// past grow_lim and bytes at or past col_lim read as zero. The 128 copy
// threads each keep one G-byte column of the rows (128 / G threads to a row,
// G rows a pass for G = 16... 2 per pass), so a thread's column offset and
// its zero-fill at the right edge are worked out once, and each further row
// costs an address step and one copy.
template <int G, bool ATOM32>
__device__ __forceinline__ void copy_rows(uint32_t sdst, int n, const uint8_t* base, long long ld_bytes, int grow0,
                                          int grow_lim, long long colb, long long col_lim, int tid) {
  constexpr int TPR = 128 / G;   // threads per row
  constexpr int RPP = 128 / TPR; // rows per pass
  const int r0 = tid / TPR;
  const int byte = (tid % TPR) * G;
  const long long cb = colb + byte;
  const int valid_c = cb >= col_lim ? 0 : (col_lim - cb < G ? static_cast<int>(col_lim - cb) : G);
  const uint8_t* src = base + static_cast<long long>(grow0 + r0) * ld_bytes + cb;
  const long long step = static_cast<long long>(RPP) * ld_bytes;
#pragma unroll 2
  for (int r = r0; r < n; r += RPP, src += step) {
    const int valid = grow0 + r < grow_lim ? valid_c : 0;
    copy_chunk<G>(sdst + r * 128 + swz_pos<ATOM32>(r, byte), valid ? src : base, valid);
  }
}

// One K-major operand tile: `rows` rows (M or N) of 128 bytes along K.
// Row r of the tile is global row (row0 + r), bytes from k0 * ES.
template <int G, int ES>
__device__ __forceinline__ void copy_kmajor_tile(uint32_t sdst, const uint8_t* base, long long ld_bytes, int rows,
                                                 int row0, int row_lim, int k0, int K, int tid) {
  copy_rows<G, false>(sdst, rows, base, ld_bytes, row0, row_lim, static_cast<long long>(k0) * ES,
                      static_cast<long long>(K) * ES, tid);
}

// One MN-major B tile: NBOX boxes, each BK rows (K) of 128 bytes along N.
template <int G, int ES, int BK, int NBOX, int BOX_BYTES, bool ATOM32>
__device__ __forceinline__ void copy_mnmajor_tile(uint32_t sdst, const uint8_t* base, long long ld_bytes, int n0,
                                                  int N, int k0, int K, int tid) {
#pragma unroll 1
  for (int box = 0; box < NBOX; ++box)
    copy_rows<G, ATOM32>(sdst + box * BOX_BYTES, BK, base, ld_bytes, k0, K,
                         static_cast<long long>(n0) * ES + box * 128, static_cast<long long>(N) * ES, tid);
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Generic-proxy writes to shared memory become visible to tcgen05.mma (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ epilogue helpers
template <int KIND>
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
  const float a = __uint_as_float(lo), b = __uint_as_float(hi);
  if constexpr (KIND == KIND_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Each epilogue warp owns a 32-row x 64-byte tile of shared memory in the
// layout of TMA's 64-byte swizzle: 16-byte chunk j of row r sits at
// r * 64 + ((j ^ ((r >> 1) & 3)) * 16), so both the lanes' row writes (lane =
// row) and the row-wise accesses below are free of bank conflicts. One round
// stages 64 bytes of each of the warp's 32 rows -- 32 columns of a 16-bit C,
// 16 of an fp32 C -- and writes them to C[row0 .., col0 ..]: by one TMA store
// of the 32 x 64-byte box when C's base and row pitch are 16-byte multiples
// and the box ends at or before column N (TMA leaves out the rows past M; a
// box that crosses column N wrote whole 16-byte pieces past it on GB300, so
// that last round of a row goes the other way), otherwise by coalesced stores:
// where C's addresses are 8-byte multiples and the round's 64 bytes of a row
// lie inside column N, 8 lanes to a row and four rows a step, 8 bytes a lane;
// else 16 lanes to a row and two rows a step, 4 bytes a lane where C's
// alignment allows and 2 where it does not.
__device__ __forceinline__ uint32_t epi_chunk_addr(uint32_t stage, int r, int j) {
  return stage + static_cast<uint32_t>(r * 64) + (static_cast<uint32_t>(j ^ ((r >> 1) & 3)) << 4);
}

// The next tile of the warp's ring, once the TMA store that last used it has
// read it (only lane 0 has stores in flight; up to bufs - 1 younger ones may
// still be reading their tiles).
__device__ __forceinline__ uint32_t epi_acquire(const GemmParams& p, int lane, EpiRing& ring) {
  uint32_t stage = ring.base + static_cast<uint32_t>(ring.next % ring.bufs) * EPI_WARP_BYTES;
  ++ring.next;
  if (!in_range(p, stage >= ring.base && stage + EPI_WARP_BYTES <= ring.end, CHECK_STAGING)) stage = ring.base;
  if (p.c_tma && lane == 0) {
    switch (ring.bufs) {
      case 1: bulk_wait_read<0>(); break;
      case 2: bulk_wait_read<1>(); break;
      case 3: bulk_wait_read<2>(); break;
      default: bulk_wait_read<3>(); break;
    }
  }
  __syncwarp();
  return stage;
}

__device__ __forceinline__ void epi_put_row(uint32_t stage, int lane, const uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(epi_chunk_addr(stage, lane, j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

__device__ __forceinline__ void epi_get_row(uint32_t stage, int lane, uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a = epi_chunk_addr(stage, lane, j);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4 * j]), "=r"(w[4 * j + 1]), "=r"(w[4 * j + 2]), "=r"(w[4 * j + 3])
                 : "r"(a)
                 : "memory");
  }
}

// Writes the staged tile to C[row0 .., col0 ..] (see above).
template <int KIND>
__device__ __forceinline__ void epi_flush(const GemmParams& p, const CUtensorMap* tmC, uint32_t stage, int lane,
                                          int row0, int col0, int bz) {
  constexpr int ROUND_COLS = KIND == KIND_TF32 ? 16 : 32;
  if (p.c_tma && col0 + ROUND_COLS <= p.N) {
    fence_proxy_async_smem();  // make the tile visible to the TMA unit
    __syncwarp();
    if (lane == 0 && row0 < p.M && col0 < p.N) {
      tma_store_3d(tmC, stage, col0, row0, bz);
      bulk_commit_group();
    }
  } else if (p.c_gran >= 8 && col0 + ROUND_COLS <= p.N) {
    __syncwarp();
    constexpr int ES = KIND == KIND_TF32 ? 4 : 2;
    const int l = lane & 7;  // the lane's 8-byte piece of the row's 64 bytes
    uint8_t* dst0 = reinterpret_cast<uint8_t*>(p.C) + (bz * p.stride_c + col0) * ES + l * 8;
#pragma unroll
    for (int rr = 0; rr < 32; rr += 4) {
      const int r = rr + (lane >> 3);
      const int row = row0 + r;
      uint32_t lo, hi;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                   : "=r"(lo), "=r"(hi)
                   : "r"(epi_chunk_addr(stage, r, l >> 1) + ((l & 1) << 3))
                   : "memory");
      if (row < p.M) *reinterpret_cast<uint2*>(dst0 + static_cast<long long>(row) * p.ldc * ES) = make_uint2(lo, hi);
    }
    __syncwarp();
  } else {
    __syncwarp();
    constexpr int ES = KIND == KIND_TF32 ? 4 : 2;
    const int l = lane & 15;
    const int col = col0 + l * (4 / ES);
#pragma unroll 4
    for (int rr = 0; rr < 32; rr += 2) {
      const int r = rr + (lane >> 4);
      const int row = row0 + r;
      const uint32_t v = ld_shared_u32(epi_chunk_addr(stage, r, l >> 2) + ((l & 3) << 2));
      if (row < p.M && col < p.N) {
        uint8_t* dst = reinterpret_cast<uint8_t*>(p.C) + (bz * p.stride_c + static_cast<long long>(row) * p.ldc + col) * ES;
        if (ES == 4 || (p.c_gran >= 4 && col + 1 < p.N)) {
          *reinterpret_cast<uint32_t*>(dst) = v;
        } else {
          reinterpret_cast<uint16_t*>(dst)[0] = static_cast<uint16_t>(v & 0xFFFFu);
          if (col + 1 < p.N) reinterpret_cast<uint16_t*>(dst)[1] = static_cast<uint16_t>(v >> 16);
        }
      }
    }
    __syncwarp();
  }
}

// Loads C's current 32 x 64-byte block at (row0, col0) into the tile with
// coalesced loads (the mirror of the row-wise stores); zeros outside M x N.
template <int KIND>
__device__ __forceinline__ void epi_load_c(const GemmParams& p, uint32_t stage, int lane, int row0, int col0,
                                           int bz) {
  constexpr int ES = KIND == KIND_TF32 ? 4 : 2;
  const int l = lane & 15;
  const int col = col0 + l * (4 / ES);
  // all 16 loads of the lane first (in flight together: the tile costs one
  // memory latency, not one per load), then the shared-memory stores
  uint32_t v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int row = row0 + 2 * i + (lane >> 4);
    v[i] = 0;
    if (row < p.M && col < p.N) {
      const uint8_t* src =
          reinterpret_cast<const uint8_t*>(p.C) + (bz * p.stride_c + static_cast<long long>(row) * p.ldc + col) * ES;
      if (ES == 4 || (p.c_gran >= 4 && col + 1 < p.N)) {
        v[i] = *reinterpret_cast<const uint32_t*>(src);
      } else {
        v[i] = reinterpret_cast<const uint16_t*>(src)[0];
        if (col + 1 < p.N) v[i] |= static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(src)[1]) << 16;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i)
    st_shared_u32(epi_chunk_addr(stage, 2 * i + (lane >> 4), l >> 2) + ((l & 3) << 2), v[i]);
  __syncwarp();
}

// Element k (0 .. 64 / ES - 1) of a staged row, as float.
template <int KIND>
__device__ __forceinline__ float epi_elem(const uint32_t (&w)[16], int k) {
  if constexpr (KIND == KIND_TF32) {
    return __uint_as_float(w[k]);
  } else {
    const uint32_t h = (k & 1) ? (w[k >> 1] >> 16) : (w[k >> 1] & 0xFFFFu);
    if constexpr (KIND == KIND_BF16)
      return __uint_as_float(h << 16);
    else
      return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  }
}

// Activation of the fused epilogue (GEMM_ACT_* of the C interface).
__device__ __forceinline__ float epi_activation(float v, int act) {
  if (act == 1) return v < 0.0f ? 0.0f : v;                                   // ReLU
  if (act == 2) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));   // GELU, x * Phi(x)
  if (act == 3) {                                                             // GELU, tanh form
    const float u = 0.79788456080286536f * (v + 0.044715f * v * v * v);
    return 0.5f * v * (1.0f + tanhf(u));
  }
  return v;
}

// The activation applied to every element of v, the choice taken once (each
// activation is one straight loop, so a plain epilogue runs no per-element
// branches).
template <int NV>
__device__ __forceinline__ void epi_activate(float (&v)[NV], int act) {
  switch (act) {
    case 1:
#pragma unroll
      for (int k = 0; k < NV; ++k) v[k] = epi_activation(v[k], 1);
      break;
    case 2:
#pragma unroll
      for (int k = 0; k < NV; ++k) v[k] = epi_activation(v[k], 2);
      break;
    case 3:
#pragma unroll
      for (int k = 0; k < NV; ++k) v[k] = epi_activation(v[k], 3);
      break;
    default:
      break;
  }
}

// One round with the fused epilogue: out = act(alpha * acc + beta * C + bias[col]),
// in fp32, then rounded to the output type. The round's accumulator columns
// are r[OFF .. OFF + 63 / ES] (32 for 16-bit C, 16 for fp32 C).
template <int KIND, int OFF>
__device__ __forceinline__ void epi_round_fused(const GemmParams& p, const CUtensorMap* tmC, EpiRing& ring,
                                                int lane, int row0, int col0, int bz, const uint32_t (&r)[32]) {
  constexpr int RC = KIND == KIND_TF32 ? 16 : 32;
  using T = typename KindTraits<KIND>::T;
  const uint32_t stage = epi_acquire(p, lane, ring);
  float v[RC];
#pragma unroll
  for (int k = 0; k < RC; ++k) v[k] = p.alpha * __uint_as_float(r[OFF + k]);
  if (p.beta != 0.0f) {
    epi_load_c<KIND>(p, stage, lane, row0, col0, bz);
    uint32_t w[16];
    epi_get_row(stage, lane, w);
#pragma unroll
    for (int k = 0; k < RC; ++k) v[k] += p.beta * epi_elem<KIND>(w, k);
    __syncwarp();  // every lane has read its row before the tile is overwritten
  }
  if (p.bias != nullptr) {
    // one load per lane (lane k holds bias[col0 + k]), handed to every lane by shuffles
    const T* bias = static_cast<const T*>(p.bias);
    float b = 0.0f;
    if (lane < RC && col0 + lane < p.N) {
      if constexpr (KIND == KIND_TF32)
        b = bias[col0 + lane];
      else if constexpr (KIND == KIND_BF16)
        b = __bfloat162float(bias[col0 + lane]);
      else
        b = __half2float(bias[col0 + lane]);
    }
#pragma unroll
    for (int k = 0; k < RC; ++k) {
      const float bk = __shfl_sync(0xFFFFFFFFu, b, k);
      if (col0 + k < p.N) v[k] += bk;
    }
  }
  epi_activate(v, p.act);
  uint32_t w[16];
  if constexpr (KIND == KIND_TF32) {
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(v[k]);
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = pack2<KIND>(__float_as_uint(v[2 * k]), __float_as_uint(v[2 * k + 1]));
  }
  epi_put_row(stage, lane, w);
  epi_flush<KIND>(p, tmC, stage, lane, row0, col0, bz);
}

// Converts 32 accumulator columns of the warp's 32 rows (lane = row, values
// in r) to the output type and writes them to C[row0 .., col0 .. col0+31] of
// matrix bz, through the fused epilogue when the launch has one (FUSED =
// false: a kernel built for plain launches only, without that code).
// Warp-collective.
template <int KIND, bool FUSED = true>
__device__ __forceinline__ void emit_chunk(const GemmParams& p, const CUtensorMap* tmC, EpiRing& ring, int lane,
                                           int row0, int col0, int bz, const uint32_t (&r)[32]) {
  if (FUSED && p.fused) {
    epi_round_fused<KIND, 0>(p, tmC, ring, lane, row0, col0, bz, r);
    if (KIND == KIND_TF32 && col0 + 16 < p.N) epi_round_fused<KIND, 16>(p, tmC, ring, lane, row0, col0 + 16, bz, r);
    return;
  }
  if constexpr (KIND == KIND_TF32) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (col0 + 16 * h >= p.N) break;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = r[16 * h + j];
      const uint32_t stage = epi_acquire(p, lane, ring);
      epi_put_row(stage, lane, w);
      epi_flush<KIND>(p, tmC, stage, lane, row0, col0 + 16 * h, bz);
    }
  } else {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack2<KIND>(r[2 * j], r[2 * j + 1]);
    const uint32_t stage = epi_acquire(p, lane, ring);
    epi_put_row(stage, lane, w);
    epi_flush<KIND>(p, tmC, stage, lane, row0, col0, bz);
  }
}

// Address of the element at byte `byte` (0 .. 63) of row r of a staging tile.
__device__ __forceinline__ uint32_t epi_elem_addr(uint32_t stage, int r, int byte) {
  return epi_chunk_addr(stage, r, byte >> 4) + static_cast<uint32_t>(byte & 15);
}

// A staged element of the output type, as float.
template <int KIND>
__device__ __forceinline__ float epi_load_elem(uint32_t addr) {
  if constexpr (KIND == KIND_TF32) {
    return __uint_as_float(ld_shared_u32(addr));
  } else if constexpr (KIND == KIND_BF16) {
    return __uint_as_float(ld_shared_u16(addr) << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(ld_shared_u16(addr))));
  }
}

// Stores one staging tile of a C^T chunk (see emit_chunk_t): x[j] holds
// C[row0 + j][col0 + lane] as fp32 bits. Neighbouring lanes trade a value so
// that each stores whole 32-bit words, a pair of rows per step (one lane row
// j, its partner row j + 1), 128 bytes a step for the warp, free of bank
// conflicts. 16-bit C (one tile of 32 columns): lanes 2i and 2i+1 hold
// columns 2i and 2i+1 and write that column pair's word in rows j and j+1
// (rounded to the output type here). fp32 C (tile h of two, 16 columns
// each): lanes l and l ^ 16 trade their row-(j+1) values, so in the tile of
// the lower 16 columns lanes 0-15 write row j and lanes 16-31 row j + 1, and
// the other way round in the upper tile.
template <int KIND>
__device__ __forceinline__ void epi_put_cols(uint32_t stage, int lane, int h, const uint32_t (&x)[32]) {
  if constexpr (KIND == KIND_TF32) {
    const int k = (lane & 15) * 4;      // byte of this lane's column within a tile
    const bool own = (lane >> 4) == h;  // this lane's column lies in tile h
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x[2 * i + 1], 16);  // partner's row 2i+1
      st_shared_u32(epi_elem_addr(stage, 2 * i + (own ? 0 : 1), k), own ? x[2 * i] : y);
    }
  } else {
    const bool odd = lane & 1;
    const int k = (lane >> 1) * 4;  // byte of this lane's column pair within the tile
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t t = odd ? x[2 * i] : x[2 * i + 1];
      const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, t, 1);
      const uint32_t w = odd ? pack2<KIND>(y, x[2 * i + 1]) : pack2<KIND>(x[2 * i], y);
      st_shared_u32(epi_elem_addr(stage, 2 * i + (odd ? 1 : 0), k), w);
    }
  }
}

// emit_chunk for an accumulator that holds a tile of C^T: lane l has
// C[row0 + j][col0 + l] in r[j], j = 0..31 (32 rows of one column of C per
// lane). Each staging tile is a 32-row box of C (16-bit C: one tile of 32
// columns; fp32 C: two of 16), filled by epi_put_cols and written out as in
// emit_chunk. With the fused epilogue each lane first computes its column's
// values in fp32 in the order of epi_round_fused (alpha * acc, + beta * C,
// read from the staged box of C, + bias[col], activation). FUSED = false
// leaves the fused code out (a kernel built for plain launches: its
// registers then hold no fused-epilogue values). Warp-collective.
template <int KIND, bool FUSED = true>
__device__ __forceinline__ void emit_chunk_t(const GemmParams& p, const CUtensorMap* tmC, EpiRing& ring, int lane,
                                             int row0, int col0, int bz, const uint32_t (&r)[32]) {
  constexpr int NT = KIND == KIND_TF32 ? 2 : 1;  // staging tiles per chunk
  constexpr int RC = 32 / NT;                    // columns per staging tile
  constexpr int ES = KIND == KIND_TF32 ? 4 : 2;
#pragma unroll
  for (int h = 0; h < NT; ++h) {
    const int cb = col0 + h * RC;
    if (cb >= p.N) break;
    const uint32_t stage = epi_acquire(p, lane, ring);
    if (FUSED && p.fused) {
      using T = typename KindTraits<KIND>::T;
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
      if (p.beta != 0.0f) {
        epi_load_c<KIND>(p, stage, lane, row0, cb, bz);
        // this lane's column of the staged box (lanes of the other fp32 tile read
        // a column of this one; their values are not stored)
        const int byte = (lane % RC) * ES;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += p.beta * epi_load_elem<KIND>(epi_elem_addr(stage, j, byte));
        __syncwarp();  // every lane has read the box before the tile is overwritten
      }
      if (p.bias != nullptr && col0 + lane < p.N) {
        const T b = static_cast<const T*>(p.bias)[col0 + lane];
        float bias;
        if constexpr (KIND == KIND_TF32)
          bias = b;
        else if constexpr (KIND == KIND_BF16)
          bias = __bfloat162float(b);
        else
          bias = __half2float(b);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bias;
      }
      epi_activate(v, p.act);
      uint32_t x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(v[j]);
      epi_put_cols<KIND>(stage, lane, h, x);
    } else {
      epi_put_cols<KIND>(stage, lane, h, r);
    }
    epi_flush<KIND>(p, tmC, stage, lane, row0, cb, bz);
  }
}

// Reads `nchunks` 32-column chunks of this warp's 32 accumulator rows from
// tensor memory and hands each to `use(c, r)`, keeping the next chunk's load
// in flight while the current one is used. Warp-collective.
template <typename Use>
__device__ __forceinline__ void for_each_acc_chunk(uint32_t taddr, int nchunks, Use use) {
  uint32_t ra[32], rb[32];
  __syncwarp();
  tmem_ld_32x32b_x32(taddr, ra);
  tmem_wait_ld_into(ra);
#pragma unroll 1
  for (int c = 0; c < nchunks; c += 2) {
    __syncwarp();
    if (c + 1 < nchunks) tmem_ld_32x32b_x32(taddr + (c + 1) * 32, rb);
    use(c, ra);
    __syncwarp();
    tmem_wait_ld_into(rb);
    if (c + 1 < nchunks) {
      __syncwarp();
      if (c + 2 < nchunks) tmem_ld_32x32b_x32(taddr + (c + 2) * 32, ra);
      use(c + 1, rb);
      __syncwarp();
      tmem_wait_ld_into(ra);
    }
  }
}

// for_each_acc_chunk over the chunks first, first + step, ... of a warp's
// accumulator rows (the single-CTA kernel's two sets of epilogue warps take
// alternate chunks). Warp-collective.
template <typename Use>
__device__ __forceinline__ void for_each_acc_chunk_strided(uint32_t taddr, int nchunks, int first, int step, Use use) {
  if (first >= nchunks) return;
  uint32_t ra[32], rb[32];
  __syncwarp();
  tmem_ld_32x32b_x32(taddr + first * 32, ra);
  tmem_wait_ld_into(ra);
#pragma unroll 1
  for (int c = first; c < nchunks; c += 2 * step) {
    const int c1 = c + step, c2 = c + 2 * step;
    __syncwarp();
    if (c1 < nchunks) tmem_ld_32x32b_x32(taddr + c1 * 32, rb);
    use(c, ra);
    __syncwarp();
    tmem_wait_ld_into(rb);
    if (c1 < nchunks) {
      __syncwarp();
      if (c2 < nchunks) tmem_ld_32x32b_x32(taddr + c2 * 32, ra);
      use(c1, rb);
      __syncwarp();
      tmem_wait_ld_into(ra);
    }
  }
}

// ------------------------------------------------------------------ the kernel
// FUSED = false: built for launches without a fused epilogue (p.fused == 0),
// with that code left out.
template <int KIND, bool B_KMAJOR, int BN, bool FUSED>
__global__ void __launch_bounds__(320, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                const GemmParams p) {
  using Cf = Cfg<KIND, B_KMAJOR, BN>;
  constexpr int S = Cf::STAGES;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + S * Cf::A_BYTES;
  const uint32_t sE = sbase + S * (Cf::A_BYTES + Cf::B_BYTES);  // output staging, EPI_BUFS x EPI_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(sptr + S * (Cf::A_BYTES + Cf::B_BYTES) + Cf::EPI_BUFS * EPI_BYTES);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain_bar = acce0 + 16;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + Cf::NUM_BARS);
  volatile int* issued_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 1;
  volatile int* consumed_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool has_copy = !(p.a_tma && p.b_tma);
  const uint32_t full_count = 1u + (has_copy ? 4u : 0u);
  // Warps 0-3 drain the accumulator; for tiles of four or more 32-column
  // chunks, where TMA loads every operand and the launch has warps 6-9 (the
  // copy warps' slots), those are a second set of epilogue warps taking every
  // other chunk. (Narrower tiles keep the plain epilogue: with the second set
  // in their code, 512^3 and 1024^3 ran 2% slower.)
  constexpr bool kTwoSets = BN >= 128;
  const int epi_warps = (kTwoSets && !has_copy && blockDim.x >= 320) ? 8 : 4;

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, full_count);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, epi_warps);
    }
    mbar_init(drain_bar, 1);
    *issued_slot = 0;
    *consumed_slot = 0;
    fence_mbar_init();
    if (p.a_tma) tma_prefetch_desc(&tmA);
    if (p.b_tma) tma_prefetch_desc(&tmB);
    if (p.b_tma && !B_KMAJOR && Cf::LASTN != Cf::BOXN) tma_prefetch_desc(&tmB2);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), Cf::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up done; from here on A, B, C and the scratch are read or written
  grid_dependency_wait();

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && !(p.debug & DEBUG_STALL_PRODUCER)) {
      const uint32_t tx = (p.a_tma ? Cf::A_BYTES : 0) + (p.b_tma ? Cf::B_TX : 0);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb, bz;
        tile_coords(p, t, mb, nb, bz);
        const int za = p.stride_a ? bz : 0, zb = p.stride_b ? bz : 0;  // a stride of 0 repeats matrix 0
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!wait_phase(p, empty0 + 8 * s, ph ^ 1, ROLE_PRODUCER | (s << 8))) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * s;
          mbar_arrive_expect_tx(fb, tx);
          const bool kx = in_range(p, (kb * Cf::BK * Cf::ES) % 16 == 0, CHECK_TMA_X);
          if (p.a_tma && kx && in_range(p, s < S && sA + (s + 1) * Cf::A_BYTES <= sB, CHECK_A_STAGE))
            tma_load_3d(sA + s * Cf::A_BYTES, &tmA, fb, kb * Cf::BK, mb * Cf::BM, za);
          if (p.b_tma && in_range(p, s < S && sB + (s + 1) * Cf::B_BYTES <= sE, CHECK_B_STAGE)) {
            if constexpr (B_KMAJOR) {
              if (kx) tma_load_3d(sB + s * Cf::B_BYTES, &tmB, fb, kb * Cf::BK, nb * Cf::BN, zb);
            } else {
#pragma unroll
              for (int j = 0; j < Cf::NBOX; ++j)
                if (in_range(p, ((nb * Cf::BN + j * Cf::BOXN) * Cf::ES) % 16 == 0, CHECK_TMA_X))
                  tma_load_3d(sB + s * Cf::B_BYTES + j * Cf::BOX_BYTES,
                              (j == Cf::NBOX - 1 && Cf::LASTN != Cf::BOXN) ? &tmB2 : &tmB, fb,
                              nb * Cf::BN + j * Cf::BOXN, kb * Cf::BK, zb);
            }
          }
        }
      }
      *issued_slot = it;
    }
    grid_launch_dependents();  // this CTA's last operand load is issued
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++tc) {
        const int b = tc & 1;
        const uint32_t use = (tc >> 1) & 1;
        if (!wait_phase(p, acce0 + 8 * b, use ^ 1, ROLE_MMA | (0x80u << 8))) break;
        tc_fence_after();
        const uint32_t d = tmem + b * Cf::ACC_COLS;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!wait_phase(p, full0 + 8 * s, ph, ROLE_MMA | (s << 8))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sA + s * Cf::A_BYTES;
          const uint32_t b_addr = sB + s * Cf::B_BYTES;
          const bool mma_ok =
              in_range(p, a_addr + Cf::A_BYTES <= sB && b_addr + Cf::B_BYTES <= sE, CHECK_DESC) &&
              in_range(p, (d & 0xFFFFu) - (tmem & 0xFFFFu) + Cf::BN <= uint32_t(Cf::TMEM_COLS), CHECK_ACC_COLS);
#pragma unroll
          for (int kk = 0; kk < Cf::KSTEPS && mma_ok; ++kk) {
            const uint64_t ad = sdesc(a_addr + kk * 32, 16, 1024, SWZ_128B);
            uint64_t bd;
            if constexpr (B_KMAJOR)
              bd = sdesc(b_addr + kk * 32, 16, 1024, SWZ_128B);
            else
              bd = sdesc(b_addr + kk * Cf::UK * 128, Cf::BOX_BYTES, Cf::B_SBO, Cf::B_SWZ);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_issue<KIND>(d, ad, bd, Cf::IDESC, acc);
          }
          mma_commit(empty0 + 8 * s);  // frees the stage once these MMAs have read it
        }
        if (!ok) break;
        mma_commit(accf0 + 8 * b);  // accumulator ready for the epilogue
      }
      *consumed_slot = it;
      // wait for every MMA this thread issued (normally already complete)
      mma_commit(drain_bar);
      wait_phase_drain(p, drain_bar, 0);
    }
  } else if (warp < 4 || (kTwoSets && epi_warps == 8)) {
    // ---------------------------------------------------------------- epilogue
    // epilogue warp e (0..epi_warps-1) reads tensor-memory lane quadrant q
    // (warp w may access lanes 32 * (w % 4) ..) and takes chunks set, set +
    // nsets, ...; its ring of staging tiles is its share of the staging area
    const int e = kTwoSets ? (warp < 4 ? warp : warp - 2) : warp;
    const int q = kTwoSets ? (warp & 3) : warp;
    const int set = kTwoSets ? (warp < 4 ? 0 : 1) : 0;
    const int nsets = kTwoSets ? epi_warps / 4 : 1;
    const int bufs = (kTwoSets && epi_warps == 8) ? (Cf::EPI_BUFS >= 2 ? Cf::EPI_BUFS / 2 : 1) : Cf::EPI_BUFS;
    int tc = 0;
    EpiRing ring{sE + static_cast<uint32_t>(e * bufs * EPI_WARP_BYTES), bufs, 0,
                 sE + static_cast<uint32_t>(Cf::EPI_BUFS * EPI_BYTES)};
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tc) {
      int mb, nb, bz;
      tile_coords(p, t, mb, nb, bz);
      const int b = tc & 1;
      const uint32_t use = (tc >> 1) & 1;
      if (!warp_wait_phase(p, accf0 + 8 * b, use, ROLE_EPILOGUE | (b << 8))) break;
      tc_fence_after();
      const int row0 = mb * Cf::BM + q * 32;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * Cf::ACC_COLS;
      int ncols = min(Cf::BN, p.N - nb * Cf::BN);
      if (!in_range(p, b * Cf::ACC_COLS + ((ncols + 31) / 32) * 32 <= Cf::TMEM_COLS, CHECK_TMEM_LD)) ncols = 0;
      auto emit = [&](int c, const uint32_t(&r)[32]) {
        emit_chunk<KindTraits<KIND>::out, FUSED>(p, &tmC, ring, lane, row0, nb * Cf::BN + c * 32, bz, r);
      };
      if constexpr (kTwoSets)
        for_each_acc_chunk_strided(taddr, (ncols + 31) / 32, set, nsets, emit);
      else
        for_each_acc_chunk(taddr, (ncols + 31) / 32, emit);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
    }
    // this warp's TMA stores of C have read their staging tiles (the shared
    // memory may be released; the grid's completion covers their writes)
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- copy warps (6-9)
    const int ctid = threadIdx.x - 6 * 32;  // 0..127
    const long long lda_b = p.lda * Cf::ES, ldb_b = p.ldb * Cf::ES;
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      int mb, nb, bz;
      tile_coords(p, t, mb, nb, bz);
      const uint8_t* Ab = static_cast<const uint8_t*>(p.A) + bz * p.stride_a * Cf::ES;
      const uint8_t* Bb = static_cast<const uint8_t*>(p.B) + bz * p.stride_b * Cf::ES;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!warp_wait_phase(p, empty0 + 8 * s, ph ^ 1, ROLE_COPY | (s << 8))) {
          ok = false;
          break;
        }
        auto copy_stage = [&](auto g) {
          constexpr int G = decltype(g)::value;
          if (!p.a_tma)
            copy_kmajor_tile<G, Cf::ES>(sA + s * Cf::A_BYTES, Ab, lda_b, Cf::BM, mb * Cf::BM, p.M, kb * Cf::BK, p.K,
                                        ctid);
          if (!p.b_tma) {
            if constexpr (B_KMAJOR)
              copy_kmajor_tile<G, Cf::ES>(sB + s * Cf::B_BYTES, Bb, ldb_b, Cf::BN, nb * Cf::BN, p.N, kb * Cf::BK,
                                          p.K, ctid);
            else
              copy_mnmajor_tile<G, Cf::ES, Cf::BK, Cf::NBOX, Cf::BOX_BYTES, Cf::B_ATOM32>(
                  sB + s * Cf::B_BYTES, Bb, ldb_b, nb * Cf::BN, p.N, kb * Cf::BK, p.K, ctid);
          }
        };
        // the copy granularity is the same for every stage of the launch
        switch (p.copy_bytes) {
          case 16: copy_stage(std::integral_constant<int, 16>{}); break;
          case 8: copy_stage(std::integral_constant<int, 8>{}); break;
          case 4: copy_stage(std::integral_constant<int, 4>{}); break;
          default:
            if constexpr (Cf::ES == 2) copy_stage(std::integral_constant<int, 2>{});
            break;
        }
        cp_async_commit();
        if (it >= Cf::COPY_LAG) {
          // the copies of stage (it - LAG) have landed: publish them to the MMA
          cp_async_wait<Cf::COPY_LAG>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full0 + 8 * ((it - Cf::COPY_LAG) % S));
        }
      }
    }
    // publish the last stages (also on abort: nothing may stay in flight)
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (ok && lane == 0) {
      for (int j = max(0, it - Cf::COPY_LAG); j < it; ++j) mbar_arrive(full0 + 8 * (j % S));
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // Loads issued but not consumed exist only when the launch was aborted: let
  // them land first. (Comparing the two counts in shared memory keeps the
  // global abort word, one L2 round trip, off every CTA's exit.)
  if (threadIdx.x == 0 && *consumed_slot < *issued_slot) {
    const int issued = *issued_slot, consumed = *consumed_slot;
    if (p.a_tma || p.b_tma)
      for (int j = consumed; j < issued; ++j)
        if (!wait_phase_drain(p, full0 + 8 * (j % S), (j / S) & 1)) break;
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Cf::TMEM_COLS);
  }
}

// Writes C = 0 (the K = 0 product) for any layout.
template <int ES>
__global__ void fill_zero_kernel(void* C, long long ldc, int M, int N) {
  const long long total = static_cast<long long>(M) * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / N, c = i - r * N;
    if constexpr (ES == 4)
      reinterpret_cast<uint32_t*>(C)[r * ldc + c] = 0u;
    else
      reinterpret_cast<uint16_t*>(C)[r * ldc + c] = 0;
  }
}

// K = 0 with the fused epilogue: C = act(alpha * 0 + beta * C + bias[col]),
// in fp32, rounded to the output type.
template <int KIND>
__global__ void epilogue_only_kernel(void* C, long long ldc, int M, int N, float alpha, float beta,
                                     const void* bias, int act) {
  using T = typename KindTraits<KIND>::T;
  const long long total = static_cast<long long>(M) * N;
  T* c = static_cast<T*>(C);
  const T* b = static_cast<const T*>(bias);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / N, col = i - r * N;
    T* e = c + r * ldc + col;
    float v = alpha * 0.0f;
    if constexpr (KIND == KIND_TF32) {
      if (beta != 0.0f) v += beta * *e;
      if (b != nullptr) v += b[col];
      *e = epi_activation(v, act);
    } else if constexpr (KIND == KIND_BF16) {
      if (beta != 0.0f) v += beta * __bfloat162float(*e);
      if (b != nullptr) v += __bfloat162float(b[col]);
      *e = __float2bfloat16_rn(epi_activation(v, act));
    } else {
      if (beta != 0.0f) v += beta * __half2float(*e);
      if (b != nullptr) v += __half2float(b[col]);
      *e = __float2half_rn(epi_activation(v, act));
    }
  }
}

}  // namespace dgt
