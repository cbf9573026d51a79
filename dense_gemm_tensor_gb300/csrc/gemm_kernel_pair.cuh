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
// Synchronisation:
//   full[s]   leader only; 1 arrival (leader producer, expecting the bytes of
//             both CTAs' TMA loads, which all complete on this barrier)
//   empty[s]  both CTAs; 1 arrival from the leader's commit (multicast)
//   accf[b]   both CTAs; 1 arrival from the leader's commit (multicast)
//   acce[b]   leader only; 8 arrivals (4 epilogue warps of each CTA)
// Every wait is bounded as in the single-CTA kernel.
#pragma once

#include "gemm_kernel.cuh"

// Accumulator buffers per CTA (1: the epilogue and the next tile's k-loop
// alternate; 2: they overlap).
#ifndef DGT_PAIR_ACC_BUFS
#define DGT_PAIR_ACC_BUFS 2
#endif

namespace dgt {

template <int KIND, bool B_KMAJOR, int BN_>
struct PairCfg {
  using T = typename KindTraits<KIND>::T;
  static constexpr int ES = sizeof(T);
  static constexpr int BM = 128;   // rows per CTA
  static constexpr int BMP = 256;  // rows per pair
  static constexpr int BN = BN_;   // tile width (columns of the pair's tile)
  static constexpr int BNH = BN / 2;
  static constexpr int BK = 128 / ES;
  static constexpr int UK = 32 / ES;
  static constexpr int KSTEPS = BK / UK;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int BOXN = 128 / ES;
  static constexpr int NBOX = BNH / BOXN;
  static constexpr int BOX_BYTES = BK * 128;
  static constexpr int B_BYTES = B_KMAJOR ? BNH * 128 : NBOX * BOX_BYTES;
  static constexpr bool B_ATOM32 = (ES == 4) && !B_KMAJOR;
  static constexpr uint32_t B_SWZ = B_ATOM32 ? SWZ_128B_ATOM32 : SWZ_128B;
  static constexpr uint32_t B_SBO = B_ATOM32 ? DGT_ATOM32_SBO : 1024;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int RESERVED = 1024 + 256;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - RESERVED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_BUFS = DGT_PAIR_ACC_BUFS;
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = (ACC_BUFS * BN <= 256) ? 256 : 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + RESERVED;
  static_assert(B_KMAJOR || NBOX * BOXN == BNH, "MN-major B: each CTA's half must be whole 128-byte slabs");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
  static_assert(ACC_BUFS * BN <= 512, "tensor memory");
  static_assert(NUM_BARS * 8 + 16 <= 256, "barrier area");
  static_assert(STAGES >= 3, "pipeline depth");
  // Instruction descriptor without N (set per work item: BN, or BN / tail_split).
  static constexpr uint32_t IDESC_NO_N = (1u << 4) | (KindTraits<KIND>::fmt << 7) |
                                         (KindTraits<KIND>::fmt << 10) | ((B_KMAJOR ? 0u : 1u) << 16) |
                                         (uint32_t(BMP >> 4) << 24);
};

// Work item w of the pair kernel -> tile rows, first column and width.
struct PairWork {
  int mb, col0, width;
};
__device__ __forceinline__ PairWork pair_work(const GemmParams& p, int w, int bn) {
  int t = w, part = 0, width = bn;
  if (w >= p.tail_start) {
    const int f = (w - p.tail_start) / p.tail_split;
    part = w - p.tail_start - f * p.tail_split;
    t = p.tail_start + f;
    width = bn / p.tail_split;
  }
  int mb, nb;
  tile_coords(p, t, mb, nb);
  return PairWork{mb, nb * bn + part * width, width};
}

template <int KIND, bool B_KMAJOR, int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB_half, const GemmParams p) {
  // tmB_half: K-major B with half-height boxes, for the split work items.
  using Cf = PairCfg<KIND, B_KMAJOR, BN>;
  constexpr int S = Cf::STAGES;
  constexpr int NB = Cf::ACC_BUFS;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + S * Cf::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sptr + S * Cf::STAGE_BYTES);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 8 * NB;
  const uint32_t drain_bar = acce0 + 8 * NB;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + Cf::NUM_BARS);
  volatile int* issued_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 1;
  volatile int* consumed_slot = reinterpret_cast<volatile int*>(bars + Cf::NUM_BARS) + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
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
    if (B_KMAJOR && p.tail_split > 1) tma_prefetch_desc(&tmB_half);
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

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0 && !(p.debug & DEBUG_STALL_PRODUCER)) {
      int it = 0;
      bool ok = true;
      for (int w = pair; ok && w < p.num_work; w += npairs) {
        const PairWork wk = pair_work(p, w, BN);
        const int half = wk.width / 2;  // B columns this CTA loads
        const int row0 = wk.mb * Cf::BMP + int(rank) * Cf::BM;
        const int col0 = wk.col0 + int(rank) * half;
        const uint32_t tx = 2u * (Cf::A_BYTES + half * 128u);
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!wait_phase(p, empty0 + 8 * s, ph ^ 1, ROLE_PRODUCER | (s << 8))) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full0 + 8 * s, tx);
          const uint32_t fb = mapa_shared(full0 + 8 * s, 0);
          tma_load_2d_pair(sA + s * Cf::A_BYTES, &tmA, fb, kb * Cf::BK, row0);
          if constexpr (B_KMAJOR) {
            tma_load_2d_pair(sB + s * Cf::B_BYTES, half == Cf::BNH ? &tmB : &tmB_half, fb, kb * Cf::BK, col0);
          } else {
            const int nbox = half / Cf::BOXN;
#pragma unroll
            for (int j = 0; j < Cf::NBOX; ++j)
              if (j < nbox)
                tma_load_2d_pair(sB + s * Cf::B_BYTES + j * Cf::BOX_BYTES, &tmB, fb, col0 + j * Cf::BOXN,
                                 kb * Cf::BK);
          }
        }
      }
      *issued_slot = it;
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer (leader only)
    if (leader && lane == 0) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int w = pair; ok && w < p.num_work; w += npairs, ++tc) {
        const int b = tc % NB;
        const uint32_t use = (tc / NB) & 1;
        const uint32_t idesc = Cf::IDESC_NO_N | (uint32_t(pair_work(p, w, BN).width >> 3) << 17);
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
#pragma unroll
          for (int kk = 0; kk < Cf::KSTEPS; ++kk) {
            const uint64_t ad = sdesc(a_addr + kk * 32, 16, 1024, SWZ_128B);
            uint64_t bd;
            if constexpr (B_KMAJOR)
              bd = sdesc(b_addr + kk * 32, 16, 1024, SWZ_128B);
            else
              bd = sdesc(b_addr + kk * Cf::UK * 128, Cf::BOX_BYTES, Cf::B_SBO, Cf::B_SWZ);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            if constexpr (KIND == KIND_TF32)
              mma_tf32_pair(d, ad, bd, idesc, acc);
            else
              mma_f16_pair(d, ad, bd, idesc, acc);
          }
          mma_commit_pair(empty0 + 8 * s, 0x3);  // both CTAs may refill stage s
        }
        if (!ok) break;
        mma_commit_pair(accf0 + 8 * b, 0x3);  // both halves of the accumulator ready
      }
      *consumed_slot = it;
      mma_commit_pair(drain_bar, 0x1);
      wait_phase_drain(p, drain_bar, 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    int tc = 0;
    for (int w = pair; w < p.num_work; w += npairs, ++tc) {
      const PairWork wk = pair_work(p, w, BN);
      const int b = tc % NB;
      const uint32_t use = (tc / NB) & 1;
      if (!warp_wait_phase(p, accf0 + 8 * b, use, ROLE_EPILOGUE | (b << 8))) break;
      tc_fence_after();
      const int row = wk.mb * Cf::BMP + int(rank) * Cf::BM + warp * 32 + lane;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + b * Cf::ACC_COLS;
      const int ncols = min(wk.width, p.N - wk.col0);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        if (c * 32 >= ncols) break;  // warp-uniform
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_wait_ld();
        store_row_chunk<KIND>(p, row, wk.col0 + c * 32, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce0 + 8 * b, 0));
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (leader && threadIdx.x == 0 && ld_volatile_u32(p.status + 1) == p.epoch) {
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
