// gemm_pipeline.cuh -- persistent tcgen05 GEMM D[M,N] = A[M,K] B[N,K]^T with
// (128 x CG) x 256 or (128 x CG) x 512 output tiles and an epilogue policy,
// for the two GEMMs of the backward (dh = G W and dW = G^T h).
//
// Operands may be K-major (K contiguous) or MN-major (M or N contiguous):
//   K-major  : one TMA box {64 (K), rows} per stage, 128-byte swizzle rows
//              along K; descriptor sbo = 1024 (8-row groups), K step +32 B.
//   MN-major : boxes {64 (M or N), 64 (K)}: each box is 64 K-rows of 128
//              bytes (64 M/N elements), i.e. swizzle atoms of 8 K-rows x 64
//              elements; descriptor lbo = 8192 (next 64-element M/N block =
//              next box), sbo = 1024 (next 8 K-rows), K step of 16 = +2048 B.
// Roles are those of the vocabulary pipeline: warp 0 TMA producer, warp 1
// TMEM allocation + MMA issue, then the epilogue warps.  With CG = 2 (cluster
// of 2) the pair computes a 256-row tile: each CTA loads its 128 rows of A and
// its half of every 256-column block of B, the leader issues
// tcgen05.mma.cta_group::2, and each CTA's TMEM holds its 128 output rows (the
// same protocol as the vocabulary pipeline).
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

constexpr int kGemmBN = 256;

// Work items: tiles [0, full_tiles) are computed whole and go through the
// epilogue policy; each of the remaining tiles (the last, partial wave of a
// persistent launch) is split into `split` K segments of kb_per_seg k-blocks,
// one item each, whose FP32 partial tiles are stored to `part` (segment s of
// tail tile j at slot j * split + s, (128 CG) x kTileN row-major floats) and
// summed by a separate pass.  Without a split: full_tiles = tiles, split = 1.
struct GemmShape {
  int M, N, K;
  int m_tiles, n_tiles, tiles, k_blocks;
  int items, full_tiles, split, kb_per_seg;
  float *part;
  unsigned long long wait_ns;  // limit of the main loops' barrier waits (0: the default)

  // Item `i` -> output tile, its k-block range [kb0, kb1), and the partial
  // slot (-1: a whole tile).
  __device__ __forceinline__ void item(int i, int &t, int &kb0, int &kb1, int &slot) const {
    if (i < full_tiles) {
      t = i;
      kb0 = 0;
      kb1 = k_blocks;
      slot = -1;
      return;
    }
    const int j = i - full_tiles;
    const int seg = j % split;
    t = full_tiles + j / split;
    kb0 = seg * kb_per_seg;
    kb1 = min(k_blocks, kb0 + kb_per_seg);
    slot = j;
  }
};

// WIDE = false: 256-column output tiles, double-buffered accumulators, 4
// epilogue warps.  WIDE = true: 512-column output tiles made of two N = 256
// MMAs sharing the A operand, one accumulator buffer (512 TMEM columns), 8
// epilogue warps each storing 256 columns.
template <int CG, bool WIDE = false>
struct GemmCfg {
  static constexpr int kStages = WIDE ? 4 : (CG == 2 ? 6 : 4);
  static constexpr int kNops = WIDE ? 2 : 1;
  static constexpr int kNacc = WIDE ? 1 : 2;
  static constexpr int kEpiw = WIDE ? 8 : 4;
  static constexpr int kTileN = kNops * kGemmBN;
  using L = PipeLayout<kGemmBN, kStages, kNops, CG, kNacc, true>;
};

// Epi must provide: struct Params; Epi(const Params&);
//   void tile(uint32_t taddr, int row0, int col0, int ncols)
// where row0 is this thread's output row and [col0, col0 + ncols) the
// output columns this warp stores from taddr on.
template <bool A_MN, bool B_MN, class Epi, int CG = 1, bool WIDE = false>
__global__ void __launch_bounds__(pipe_threads(GemmCfg<CG, WIDE>::kEpiw), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmShape g, const uint32_t idesc, const typename Epi::Params ep,
                uint32_t *status) {
  using C = GemmCfg<CG, WIDE>;
  using L = typename C::L;
  constexpr int STAGES = C::kStages;
  constexpr int BN = kGemmBN;
  constexpr int NOPS = C::kNops;
  constexpr int EPIW = C::kEpiw;
  constexpr bool kPair = CG == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * L::kStageBytes);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // k-block iterations the peer's producer issued (written there at teardown)
  volatile uint32_t *peer_issued = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG;
  const int num_units = gridDim.x / CG;
  const uint64_t lim = wait_limit(g.wait_ns);  // limit of the main loops' waits
  uint32_t issued = 0;  // producer: k-block iterations whose copies were issued

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPIW * CG);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *peer_issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, L::kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if (kPair)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // The producer and the MMA issuer run on one lane each (the other lanes of
  // their warps wait at the end): no warp-wide exchange sits between one
  // k-block's MMAs and the next's.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t full_dst = kPair ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
      for (int it = unit; ok && it < g.items; it += num_units) {
        int t, kb0, kb1, slot;
        g.item(it, t, kb0, kb1, slot);
        const int mt = t / g.n_tiles, nt = t - (t / g.n_tiles) * g.n_tiles;
        const int arow = mt * (kBM * CG) + static_cast<int>(rank) * kBM;   // M offset
        // N offset of this CTA's share of MMA op 0 (op k adds k * BN)
        const int bcol = nt * C::kTileN + static_cast<int>(rank) * L::kBRows;
        for (int kb = kb0; kb < kb1; ++kb) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, lim);
          if (!ok) break;
          uint8_t *sa = smem + stage * L::kStageBytes;
          uint8_t *sb = sa + L::kABytes;
          if (leader) mbar_arrive_expect_tx(&full[stage], CG * L::kStageBytes);
          const uint32_t fb = full_dst + stage * 8;
          auto load = [&](void *dst, const CUtensorMap *m, int c0, int c1) {
            if (kPair)
              tma_load_2d_pair(dst, m, fb, c0, c1);
            else
              tma_load_2d(dst, m, &full[stage], c0, c1);
          };
          if (A_MN) {
            load(sa, &tmA, arow, kb * kBK);
            load(sa + 8192, &tmA, arow + 64, kb * kBK);
          } else {
            load(sa, &tmA, kb * kBK, arow);
          }
#pragma unroll
          for (int op = 0; op < NOPS; ++op) {
            uint8_t *sbo = sb + op * L::kBBytes;
            if (B_MN) {
#pragma unroll
              for (int i = 0; i < L::kBRows / 64; ++i)
                load(sbo + i * 8192, &tmB, bcol + op * BN + i * 64, kb * kBK);
            } else {
              load(sbo, &tmB, kb * kBK, bcol + op * BN);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int it = unit; ok && it < g.items; it += num_units) {
        int t, kb0, kb1, slot;
        g.item(it, t, kb0, kb1, slot);
        ok = mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, lim);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * L::kAccCols);
        for (int kb = kb0; kb < kb1; ++kb) {
          ok = mbar_wait(&full[stage], phase, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t b0 = a0 + L::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a0 + kk * kUmmaK * 2, 16, 1024);
#pragma unroll
            for (int op = 0; op < NOPS; ++op) {
              const uint32_t bo = b0 + op * L::kBBytes;
              const uint64_t bd = B_MN ? sdesc_sw128(bo + kk * 2048, 8192, 1024)
                                       : sdesc_sw128(bo + kk * kUmmaK * 2, 16, 1024);
              if (kPair)
                mma_f16_pair(d_tmem + op * BN, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
              else
                mma_f16(d_tmem + op * BN, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
            }
          }
          if (kPair)
            mma_commit_pair(&empty[stage], 0x3);
          else
            mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (kPair)
          mma_commit_pair(&tfull[acc], 0x3);
        else
          mma_commit(&tfull[acc]);
        if (C::kNacc == 2) acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int lg = warp & 3;
    const int half = (warp - 2) / 4;                    // column half (8 epilogue warps)
    constexpr int kWarpCols = C::kTileN / (EPIW / 4);  // output columns per warp
    const uint32_t lane_off = (static_cast<uint32_t>(lg * 32) << 16) +
                              static_cast<uint32_t>(half * kWarpCols);
    const uint32_t tempty_dst = kPair ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);
    Epi epi(ep);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int it = unit; it < g.items; it += num_units) {
      int t, kb0, kb1, slot;
      g.item(it, t, kb0, kb1, slot);
      const int mt = t / g.n_tiles, nt = t - (t / g.n_tiles) * g.n_tiles;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, lim);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_off + static_cast<uint32_t>(acc * L::kAccCols);
      if (slot < 0) {
        epi.tile(taddr, mt * (kBM * CG) + static_cast<int>(rank) * kBM + lg * 32 + lane,
                 nt * C::kTileN + half * kWarpCols, kWarpCols);
      } else {
        // a K segment of a tail tile: the FP32 partial tile, row-major
        float *prow = g.part + static_cast<size_t>(slot) * (kBM * CG) * C::kTileN +
                      static_cast<size_t>(static_cast<int>(rank) * kBM + lg * 32 + lane) * C::kTileN +
                      half * kWarpCols;
#pragma unroll 1
        for (int c = 0; c < kWarpCols / 32; ++c) {
          float x[32];
          tmem_ld32(taddr + c * 32, x);
          float4 *d = reinterpret_cast<float4 *>(prow + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(tempty_dst + acc * 8);
        else
          mbar_arrive(&tempty[acc]);
      }
      if (C::kNacc == 2) acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) record_timeout<CG>(status, abort_flag);
  }

  // Teardown, as in the vocabulary pipeline: in-flight copies and MMAs are
  // drained after a wait gave up, before TMEM is freed and the CTAs exit.
  if (kPair && warp == 0 && lane == 0 && !leader)
    st_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(peer_issued)), 0), issued);
  pipe_sync<CG>();
  if (*abort_flag) {
    if (leader && lane == 0) {
      if (warp == 0)
        drain_copies<STAGES, CG>(full, issued, kPair ? *peer_issued : issued, L::kStageBytes);
      else if (warp == 1)
        drain_mmas<CG>(drain);
    }
    pipe_sync<CG>();
  }
  if (warp == 1) tmem_dealloc<CG>(tmem_base, L::kTmemCols);
}

}  // namespace flp
