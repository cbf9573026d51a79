// CTA-pair variant of the GEMM kernel (cluster of 2 CTAs on two SMs):
// the pair computes a 256 x BN output tile with tcgen05.mma.cta_group::2.
//
// Each CTA streams only its own half of the operands -- A rows 128r..128r+127
// and B columns [r*BN/2, (r+1)*BN/2) of the tile for CTA rank r -- so an SM
// receives 16 KB of A and BN/2 x 128 bytes of B per 128-byte k-slab instead
// of 16 KB + BN x 128 bytes: the same tile FLOPs for two thirds of the bytes
// at BN = 256. The MMA, issued by one thread of the leader CTA (rank 0), reads
// both CTAs' shared memory at the same offsets and leaves rows 0-127 of the
// accumulator in the leader's tensor memory and rows 128-255 in the peer's.
//
// OPS (operand arrangement, see OPS_B_MN / OPS_B_K / OPS_SWAP below): with
// OPS_SWAP the pair computes a tile of C^T = B^T A^T instead -- the rows above
// are columns of C and the tile's BN columns are rows of C -- and the
// epilogue transposes each accumulator chunk on its way to shared memory.
//
// PAIRS = 2: a cluster of four CTAs holds two pairs (ranks 0-1 and 2-3) that
// compute two adjacent tiles of one 256-row band. CTAs of the same half (ranks
// r and r + 2) need the same 128 rows of A, so each loads 64 of them and TMA
// multicasts them into both; a stage is refilled only once both pairs' MMAs
// have read it. A work tile is then two 256 x BN tiles; when the number of tile
// columns is odd the second pair's last tile lies past N and is not stored.
//
// Tail: when the tiles do not fill a whole number of rounds of the grid, each
// tile of the last partial round is split into `tail_segs` ranges of k-slabs
// run by different pairs, so the round takes 1/tail_segs of a tile's time.
// Every segment writes its fp32 partial tile to the workspace and bumps an
// arrival counter; the last to arrive sums the segments in segment order
// (its own from tensor memory) and stores C. No CTA waits for another, and
// the sum does not depend on the arrival order.
//
// Synchronisation (per pair; "leader" = the pair's even rank):
//   full[s]   leader only; 1 arrival (leader producer, expecting the bytes that
//             land in both CTAs of the pair, which all complete on this barrier)
//   empty[s]  every CTA; PAIRS arrivals, one commit from each pair's leader
//             (multicast to every CTA of the cluster)
//   accf[b]   both CTAs of the pair; 1 arrival from the leader's commit (multicast)
//   acce[b]   leader only; 8 arrivals (4 epilogue warps of each CTA of the pair)
// Every wait is bounded as in the single-CTA kernel.
#pragma once

#include "gemm_kernel.cuh"

namespace dgt {

// Operand arrangements of the pair kernel (its OPS parameter).
enum : int {
  OPS_B_MN = 0,  // A K-major (row-major M x K), B MN-major (row-major K x N)
  OPS_B_K = 1,   // A and B K-major (B given as N x K)
  // The transposed product C^T = B^T A^T for a row-major B: the MMA's A operand
  // is B^T, MN-major, 128 of C's columns per CTA in whole 128-byte boxes; its B
  // operand is A, K-major, BN / 2 of C's rows per CTA; the accumulator holds
  // a tile of C^T (tensor-memory lane = column of C, column = row of C). A tile
  // width that is not whole 128-byte boxes of B (224, 192) then costs no
  // unused shared memory, and the 224-wide tile gets a seventh stage.
  OPS_SWAP = 2,
};

template <int KIND, int OPS, int BN_>
struct PairCfg {
  using T = typename KindTraits<KIND>::T;
  static constexpr bool B_KMAJOR = OPS == OPS_B_K;
  static constexpr bool SWAP = OPS == OPS_SWAP;
  static constexpr int ES = sizeof(T);
  static constexpr int BM = 128;   // rows of the MMA's A operand per CTA (of C^T when SWAP)
  static constexpr int BMP = 256;  // per pair
  static constexpr int BN = BN_;   // tile width (columns of the pair's accumulator; rows of C when SWAP)
  static constexpr int BNH = BN / 2;
  static constexpr int BK = 128 / ES;
  static constexpr int UK = 32 / ES;
  static constexpr int KSTEPS = BK / UK;
  // MN-major boxes (B, or B^T as the MMA's A operand when SWAP): 128-byte rows along M/N
  static constexpr int BOXN = 128 / ES;
  static constexpr int BOX_BYTES = BK * 128;
  static constexpr bool MN_ATOM32 = ES == 4;  // fp32 MN-major: 128-byte swizzle of 32-byte chunks
  static constexpr uint32_t MN_SWZ = MN_ATOM32 ? SWZ_128B_ATOM32 : SWZ_128B;
  static constexpr uint32_t MN_SBO = MN_ATOM32 ? DGT_ATOM32_SBO : 1024;
  static constexpr int A_BYTES = BM * 128;  // 128 K-major rows, or (SWAP) 128 / BOXN MN-major boxes
  static constexpr int NABOX = SWAP ? BM / BOXN : 0;
  static constexpr int NBOX = (BNH + BOXN - 1) / BOXN;  // MN-major B: boxes per CTA (last may be partly used)
  static constexpr int B_BYTES = (B_KMAJOR || SWAP) ? BNH * 128 : NBOX * BOX_BYTES;
  // MN-major B: the last box carries only the columns the tile uses (a
  // narrower box still lands in 128-byte swizzled rows), so a stage moves
  // B_TX bytes of B while taking B_BYTES of shared memory.
  static constexpr int LASTN = BNH - (NBOX - 1) * BOXN;
  static constexpr bool B_MN = OPS == OPS_B_MN;
  static constexpr int B_TX = B_MN ? (NBOX - 1) * BOX_BYTES + LASTN * BK * ES : B_BYTES;
  static constexpr uint32_t B_SWZ = MN_SWZ;
  static constexpr uint32_t B_SBO = MN_SBO;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGE_TX = A_BYTES + B_TX;  // bytes the TMA loads of one CTA's stage deliver
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - (1024 + EPI_BYTES + 256)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int EPI_BUFS = epi_bufs_for(SMEM_LIMIT, 1024 + 256 + STAGES * STAGE_BYTES);
  static constexpr int RESERVED = 1024 /*align slack*/ + EPI_BUFS * EPI_BYTES /*output staging*/ + 256 /*barriers*/;
  static constexpr int ACC_BUFS = 2;  // the epilogue of one tile overlaps the next tile's k-loop
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = (ACC_BUFS * BN <= 256) ? 256 : 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + RESERVED;
  static constexpr int PARTIAL_FLOATS = BM * BN;  // one CTA's fp32 partial tile
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
  static_assert(BNH % 16 == 0, "each CTA's B half is whole 16-column groups");
  static_assert(!SWAP || BM % BOXN == 0, "B^T comes in whole boxes");
  static_assert(ACC_BUFS * BN <= 512, "tensor memory");
  static_assert(NUM_BARS * 8 + 32 <= 256, "barrier area");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
  // bit 15: A MN-major (SWAP), bit 16: B MN-major (row-major B, not swapped)
  static constexpr uint32_t IDESC = (1u << 4) | (KindTraits<KIND>::fmt << 7) | (KindTraits<KIND>::fmt << 10) |
                                    ((SWAP ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
                                    (uint32_t(BN >> 3) << 17) | (uint32_t(BMP >> 4) << 24);
};

// Work item w of the pair kernel -> tile, k-slab range and (for split tiles)
// the tail index f and segment.
struct PairWork {
  int mb, nb, bz, kb0, kb1, f, seg;
};
__device__ __forceinline__ PairWork pair_work(const GemmParams& p, int w) {
  PairWork r;
  int t = w;
  r.f = -1;
  r.seg = 0;
  r.kb0 = 0;
  r.kb1 = p.num_kb;
  if (w >= p.tail_start) {
    const int j = w - p.tail_start;
    r.f = j / p.tail_segs;
    r.seg = j - r.f * p.tail_segs;
    t = p.tail_start + r.f;
    r.kb0 = static_cast<int>((static_cast<long long>(p.num_kb) * r.seg) / p.tail_segs);
    r.kb1 = static_cast<int>((static_cast<long long>(p.num_kb) * (r.seg + 1)) / p.tail_segs);
  }
  tile_coords(p, t, r.mb, r.nb, r.bz);
  return r;
}

// Registers an arrival on a split tile's counter and returns the arrival
// index (0-based) within this launch. The counter holds (epoch << 32) | count,
// so a value left by an earlier launch reads as zero arrivals.
__device__ __forceinline__ int arrive_split(const GemmParams& p, unsigned long long* ctr) {
  const unsigned long long tag = static_cast<unsigned long long>(p.epoch) << 32;
  unsigned long long cur = atomicAdd(ctr, 0ull);
  for (int guard = 0; guard < (1 << 20); ++guard) {
    const unsigned long long cnt = ((cur & 0xFFFFFFFF00000000ull) == tag) ? (cur & 0xFFFFFFFFull) : 0ull;
    const unsigned long long seen = atomicCAS(ctr, cur, tag | (cnt + 1));
    if (seen == cur) return static_cast<int>(cnt);
    cur = seen;
  }
  record_timeout(p, ROLE_EPILOGUE | (0xF0u << 8));
  return 0;
}

// k-slab taken at step i of a work item in the pair's round `round`. Rounds
// alternate direction, so each round starts on the slabs that the previous
// round (whose tiles ran in step with this one's) read last, while they are
// still in L2.
__device__ __forceinline__ int pair_kb(const PairWork& wk, int i, int round) {
  return (round & 1) ? wk.kb1 - 1 - i : wk.kb0 + i;
}

__device__ __forceinline__ void epilogue_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// FUSED = false: built for launches without a fused epilogue (p.fused == 0),
// with that code left out.
template <int KIND, int OPS, int BN, int PAIRS, bool FUSED>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                     const GemmParams p) {
  using Cf = PairCfg<KIND, OPS, BN>;
  constexpr bool B_KMAJOR = Cf::B_KMAJOR;
  constexpr int S = Cf::STAGES;
  constexpr int NB = Cf::ACC_BUFS;
  constexpr int CL = 2 * PAIRS;  // CTAs per cluster
  static_assert(PAIRS == 1 || PAIRS == 2, "one pair, or two pairs sharing A");
  static_assert(PAIRS == 1 || !DGT_NO_MULTICAST, "two pairs share A through a multicast load");
  static_assert(PAIRS == 1 || !Cf::SWAP, "the transposed product runs as single pairs");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + S * Cf::A_BYTES;
  const uint32_t sE = sbase + S * Cf::STAGE_BYTES;  // output staging, EPI_BUFS x EPI_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(sptr + S * Cf::STAGE_BYTES + Cf::EPI_BUFS * EPI_BYTES);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 8 * NB;
  const uint32_t drain_bar = acce0 + 8 * NB;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + Cf::NUM_BARS);
  volatile int* issued_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 1;
  volatile int* consumed_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 2;
  volatile int* last_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 3;
  volatile int* ok_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 4;  // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 .. CL-1
  const uint32_t half = rank & 1u;           // which half of the pair's 256 rows
  const uint32_t lead = rank & ~1u;          // rank of this pair's leader
  const int q = int(rank >> 1);              // which pair of the cluster
  const bool leader = half == 0;
  const int pair = blockIdx.x / CL;          // the cluster's index in the work stream
  const int npairs = gridDim.x / CL;

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, PAIRS);  // one commit from each pair that reads stage s's A
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 8);
    }
    mbar_init(drain_bar, 1);
    *issued_slot = 0;
    *consumed_slot = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Cf::B_MN && Cf::LASTN != Cf::BOXN) tma_prefetch_desc(&tmB2);
  }
  if (warp == 5) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), Cf::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up done; from here on A, B, C and the scratch are read or written
  grid_dependency_wait();

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    // The whole warp walks the loop (so addresses and coordinates stay
    // warp-uniform); one elected lane issues.
    if (!(p.debug & DEBUG_STALL_PRODUCER)) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int w = pair; ok && w < p.num_work; w += npairs, ++tc) {
        const PairWork wk = pair_work(p, w);
        // rows of the MMA's A operand (SWAP: columns of C) and columns of its B operand (SWAP: rows of C)
        const int row0 = wk.mb * Cf::BMP + int(half) * Cf::BM;
        const int col0 = (wk.nb * PAIRS + q) * BN + int(half) * Cf::BNH;
        const int za = p.stride_a ? wk.bz : 0, zb = p.stride_b ? wk.bz : 0;  // a stride of 0 repeats matrix 0
        for (int i = 0; i < wk.kb1 - wk.kb0; ++i, ++it) {
          const int kb = pair_kb(wk, i, tc);
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!warp_wait_phase(p, empty0 + 8 * s, ph ^ 1, ROLE_PRODUCER | (s << 8))) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full0 + 8 * s, lead);
          const uint32_t a_dst = sA + s * Cf::A_BYTES;
          const uint32_t b_dst = sB + s * Cf::B_BYTES;
          const bool ld_ok = in_range(p, s < S && a_dst + Cf::A_BYTES <= sB, CHECK_A_STAGE) &&
                             in_range(p, b_dst + Cf::B_BYTES <= sE, CHECK_B_STAGE) &&
                             in_range(p, (kb * Cf::BK * Cf::ES) % 16 == 0 && ((Cf::SWAP ? row0 : col0) * Cf::ES) % 16 == 0,
                                      CHECK_TMA_X);
          if (ld_ok && elect_one()) {
            if (leader) mbar_arrive_expect_tx(full0 + 8 * s, 2 * Cf::STAGE_TX);
            if constexpr (Cf::SWAP) {
              // B^T: this CTA's 128 columns of C in MN-major boxes; A: its BN / 2 rows of C, K-major
#pragma unroll
              for (int j = 0; j < Cf::NABOX; ++j)
                tma_load_3d_pair(a_dst + j * Cf::BOX_BYTES, &tmB, fb, row0 + j * Cf::BOXN, kb * Cf::BK, zb);
              tma_load_3d_pair(b_dst, &tmA, fb, kb * Cf::BK, col0, za);
            } else {
              if constexpr (PAIRS == 1) {
                tma_load_3d_pair(a_dst, &tmA, fb, kb * Cf::BK, row0, za);
              } else {
#if !DGT_NO_MULTICAST
                // both pairs need these 128 rows of A: each loads 64 of them into
                // the same place in its own and the other pair's CTA of this half
                tma_load_3d_pair_mc(a_dst + q * (Cf::A_BYTES / 2), &tmA, fb, kb * Cf::BK, row0 + q * (Cf::BM / 2),
                                    za, uint16_t(0x5u << half));
#endif
              }
              if constexpr (B_KMAJOR) {
                tma_load_3d_pair(b_dst, &tmB, fb, kb * Cf::BK, col0, zb);
              } else {
#pragma unroll
                for (int j = 0; j < Cf::NBOX; ++j)
                  tma_load_3d_pair(b_dst + j * Cf::BOX_BYTES,
                                   (j == Cf::NBOX - 1 && Cf::LASTN != Cf::BOXN) ? &tmB2 : &tmB, fb,
                                   col0 + j * Cf::BOXN, kb * Cf::BK, zb);
              }
            }
          }
          __syncwarp();
        }
      }
      if (lane == 0) *issued_slot = it;
    }
    grid_launch_dependents();  // this CTA's last operand load is issued
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer (leader only)
    // The whole warp walks the loop and builds the descriptors (warp-uniform);
    // one elected lane -- the same lane every time -- issues the MMAs and commits.
    if (leader) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int w = pair; ok && w < p.num_work; w += npairs, ++tc) {
        const PairWork wk = pair_work(p, w);
        const int b = tc % NB;
        const uint32_t use = (tc / NB) & 1;
        if (!warp_wait_phase(p, acce0 + 8 * b, use ^ 1, ROLE_MMA | (0x80u << 8))) break;
        tc_fence_after();
        const uint32_t d = tmem + b * Cf::ACC_COLS;
        for (int i = 0; i < wk.kb1 - wk.kb0; ++i, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!warp_wait_phase(p, full0 + 8 * s, ph, ROLE_MMA | (s << 8))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sA + s * Cf::A_BYTES;
          const uint32_t b_addr = sB + s * Cf::B_BYTES;
          const bool mma_ok =
              in_range(p, a_addr + Cf::A_BYTES <= sB && b_addr + Cf::B_BYTES <= sE, CHECK_DESC) &&
              in_range(p, (d & 0xFFFFu) - (tmem & 0xFFFFu) + BN <= uint32_t(Cf::TMEM_COLS), CHECK_ACC_COLS);
          uint64_t ad[Cf::KSTEPS], bd[Cf::KSTEPS];
#pragma unroll
          for (int kk = 0; kk < Cf::KSTEPS; ++kk) {
            if constexpr (Cf::SWAP)
              ad[kk] = sdesc(a_addr + kk * Cf::UK * 128, Cf::BOX_BYTES, Cf::MN_SBO, Cf::MN_SWZ);
            else
              ad[kk] = sdesc(a_addr + kk * 32, 16, 1024, SWZ_128B);
            if constexpr (B_KMAJOR || Cf::SWAP)
              bd[kk] = sdesc(b_addr + kk * 32, 16, 1024, SWZ_128B);
            else
              bd[kk] = sdesc(b_addr + kk * Cf::UK * 128, Cf::BOX_BYTES, Cf::B_SBO, Cf::B_SWZ);
          }
          const uint32_t first = (i == 0) ? 0u : 1u;  // the accumulator restarts at a work item's first step
          if (mma_ok && elect_one()) {
#pragma unroll
            for (int kk = 0; kk < Cf::KSTEPS; ++kk) {
              const uint32_t acc = kk > 0 ? 1u : first;
              mma_issue_pair<KIND>(d, ad[kk], bd[kk], Cf::IDESC, acc);
            }
            // every CTA whose loads land in stage s may refill it once all pairs are done with it
            mma_commit_pair(empty0 + 8 * s, uint16_t((1u << CL) - 1u));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) mma_commit_pair(accf0 + 8 * b, uint16_t(0x3u << lead));  // both halves of the accumulator ready
        __syncwarp();
      }
      if (lane == 0) *consumed_slot = it;
      if (elect_one()) mma_commit_pair(drain_bar, uint16_t(1u << lead));
      __syncwarp();
      if (lane == 0) wait_phase_drain(p, drain_bar, 0);
      __syncwarp();
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    // The four warps take every decision together (thread 0 waits, the named
    // barrier publishes the outcome), so the barriers below always see all 128.
    const int tid = threadIdx.x;  // 0..127
    int tc = 0;
    EpiRing ring{sE + static_cast<uint32_t>(warp * Cf::EPI_BUFS * EPI_WARP_BYTES), Cf::EPI_BUFS, 0,
                 sE + static_cast<uint32_t>(Cf::EPI_BUFS * EPI_BYTES)};
    for (int w = pair; w < p.num_work; w += npairs, ++tc) {
      const PairWork wk = pair_work(p, w);
      const int b = tc % NB;
      const uint32_t use = (tc / NB) & 1;
      if (tid == 0) ok_slot[tc & 1] = wait_phase(p, accf0 + 8 * b, use, ROLE_EPILOGUE | (b << 8)) ? 1 : 0;
      epilogue_barrier();
      if (!ok_slot[tc & 1]) break;
      tc_fence_after();
      const int nbt = wk.nb * PAIRS + q;  // this pair's tile column (past the last one: nothing to store)
      // first of this warp's 32 accumulator rows (SWAP: columns of C), and the
      // tile's first accumulator column (SWAP: row of C)
      const int row0 = wk.mb * Cf::BMP + int(half) * Cf::BM + warp * 32;
      const int col0 = nbt * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + b * Cf::ACC_COLS;
      const int ncols = min(BN, (Cf::SWAP ? p.M : p.N) - col0);
      int nchunks = ncols > 0 ? (ncols + 31) / 32 : 0;
      if (!in_range(p, b * Cf::ACC_COLS + nchunks * 32 <= Cf::TMEM_COLS, CHECK_TMEM_LD)) nchunks = 0;
      // accumulator chunk c (32 columns) of the warp's 32 rows, as output
      auto emit = [&](int c, const uint32_t(&v)[32]) {
        if constexpr (Cf::SWAP)
          emit_chunk_t<KindTraits<KIND>::out, FUSED>(p, &tmC, ring, lane, col0 + c * 32, row0, wk.bz, v);
        else
          emit_chunk<KindTraits<KIND>::out, FUSED>(p, &tmC, ring, lane, row0, col0 + c * 32, wk.bz, v);
      };
      if (wk.f < 0) {
        for_each_acc_chunk(taddr, nchunks, emit);
      } else {
        // split tile: publish this segment's partial, then find out whether it is the last
        // (every slot this tile's segments use, and its counters, lie in the scratch)
        const bool slots_ok =
            in_range(p, static_cast<long long>(wk.f + 1) * p.tail_segs * CL <= p.ws_slots, CHECK_SPLIT_SLOT) &&
            in_range(p, (wk.f + 1) * CL <= kSplitCounters, CHECK_SPLIT_CTR);
        if (!slots_ok) nchunks = 0;
        float4* mine = reinterpret_cast<float4*>(
            p.ws + (static_cast<long long>(wk.f * p.tail_segs + wk.seg) * CL + rank) * Cf::PARTIAL_FLOATS);
        for_each_acc_chunk(taddr, nchunks, [&](int c, const uint32_t(&r)[32]) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            __stcg(mine + (c * 8 + q) * 128 + tid,
                   make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                               __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
        });
        __threadfence();
        epilogue_barrier();
        if (tid == 0) {
          const int arrival = slots_ok ? arrive_split(p, p.ws_ctr + wk.f * CL + rank) : 0;
          *last_slot = (arrival + 1 == p.tail_segs) ? 1 : 0;
        }
        epilogue_barrier();
        const bool last = *last_slot != 0;
        __threadfence();
        if (last && p.tail_segs == 2) {
          // C = own + other: fp32 addition commutes, so which segment arrives last does not matter
          const float4* other = reinterpret_cast<const float4*>(
              p.ws + (static_cast<long long>(wk.f * 2 + (1 - wk.seg)) * CL + rank) * Cf::PARTIAL_FLOATS);
          float4 nxt[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) nxt[q] = __ldcg(other + q * 128 + tid);
          for_each_acc_chunk(taddr, nchunks, [&](int c, const uint32_t(&r)[32]) {
            float4 cur[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) cur[q] = nxt[q];
            if (c + 1 < nchunks) {
#pragma unroll
              for (int q = 0; q < 8; ++q) nxt[q] = __ldcg(other + ((c + 1) * 8 + q) * 128 + tid);
            }
            uint32_t sum[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              sum[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + cur[q].x);
              sum[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + cur[q].y);
              sum[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + cur[q].z);
              sum[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + cur[q].w);
            }
            emit(c, sum);
          });
        } else if (last) {
          // three or four segments: add them in segment order; this CTA's own one comes from tensor memory
          for_each_acc_chunk(taddr, nchunks, [&](int c, const uint32_t(&r)[32]) {
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
            for (int sg = 0; sg < p.tail_segs; ++sg) {
              if (sg == wk.seg) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  acc[j] = (sg == 0) ? __uint_as_float(r[j]) : acc[j] + __uint_as_float(r[j]);
              } else {
                const float4* part = reinterpret_cast<const float4*>(
                    p.ws + (static_cast<long long>(wk.f * p.tail_segs + sg) * CL + rank) * Cf::PARTIAL_FLOATS);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float4 v = __ldcg(part + (c * 8 + q) * 128 + tid);
                  acc[4 * q] = (sg == 0) ? v.x : acc[4 * q] + v.x;
                  acc[4 * q + 1] = (sg == 0) ? v.y : acc[4 * q + 1] + v.y;
                  acc[4 * q + 2] = (sg == 0) ? v.z : acc[4 * q + 2] + v.z;
                  acc[4 * q + 3] = (sg == 0) ? v.w : acc[4 * q + 3] + v.w;
                }
              }
            }
            uint32_t out[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) out[j] = __float_as_uint(acc[j]);
            emit(c, out);
          });
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce0 + 8 * b, lead));
    }
    // this warp's TMA stores of C have read their staging tiles (the shared
    // memory may be released; the grid's completion covers their writes)
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // loads issued but not consumed exist only when the launch was aborted
  // (shared-memory counts: no global read on the normal exit path)
  if (leader && threadIdx.x == 0 && *consumed_slot < *issued_slot) {
    const int issued = *issued_slot, consumed = *consumed_slot;
    for (int j = consumed; j < issued; ++j)
      if (!wait_phase_drain(p, full0 + 8 * (j % S), (j / S) & 1)) break;
  }
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Cf::TMEM_COLS);
  }
}

}  // namespace dgt
