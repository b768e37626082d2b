// gemm_pipeline.cuh -- persistent tcgen05 GEMM D[M,N] = A[M,K] B[N,K]^T with
// 128 x 256 output tiles and an epilogue policy, for the two GEMMs of the
// backward (dh = G W and dW = G^T h).
//
// Operands may be K-major (K contiguous) or MN-major (M or N contiguous):
//   K-major  : one TMA box {64 (K), rows} per stage, 128-byte swizzle rows
//              along K; descriptor sbo = 1024 (8-row groups), K step +32 B.
//   MN-major : boxes {64 (M or N), 64 (K)}: each box is 64 K-rows of 128
//              bytes (64 M/N elements), i.e. swizzle atoms of 8 K-rows x 64
//              elements; descriptor lbo = 8192 (next 64-element M/N block =
//              next box), sbo = 1024 (next 8 K-rows), K step of 16 = +2048 B.
// Roles are those of the vocabulary pipeline: warp 0 TMA producer, warp 1
// TMEM allocation + MMA issue, warps 2-5 epilogue; 4-stage ring of
// A 16 KB + B 32 KB; double-buffered 256-column TMEM accumulators.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

constexpr int kGemmBN = 256;
constexpr int kGemmStages = 4;

struct GemmShape {
  int M, N, K;
  int m_tiles, n_tiles, tiles, k_blocks;
};

using GemmLayout = PipeLayout<kGemmBN, kGemmStages, 1>;

// Epi must provide: struct Params; Epi(const Params&);
//   void tile(uint32_t taddr, int mt, int nt, int lg, int lane)
template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kPipeThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmShape g, const uint32_t idesc, const typename Epi::Params ep,
                uint32_t *status) {
  using L = GemmLayout;
  constexpr int STAGES = kGemmStages;
  constexpr int BN = kGemmBN;
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, L::kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < g.tiles; t += gridDim.x) {
      const int mt = t / g.n_tiles, nt = t - (t / g.n_tiles) * g.n_tiles;
      for (int kb = 0; kb < g.k_blocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t *sa = smem + stage * L::kStageBytes;
          uint8_t *sb = sa + L::kABytes;
          mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          if (A_MN) {
            tma_load_2d(sa, &tmA, &full[stage], mt * kBM, kb * kBK);
            tma_load_2d(sa + 8192, &tmA, &full[stage], mt * kBM + 64, kb * kBK);
          } else {
            tma_load_2d(sa, &tmA, &full[stage], kb * kBK, mt * kBM);
          }
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + i * 8192, &tmB, &full[stage], nt * BN + i * 64, kb * kBK);
          } else {
            tma_load_2d(sb, &tmB, &full[stage], kb * kBK, nt * BN);
          }
        }
        armed |= 1u << stage;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      record_timeout(status, abort_flag);
      for (int s = 0; s < STAGES; ++s) {
        if (!(armed & (1u << s))) continue;
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        int never = 0;
        mbar_wait(&full[s], par, &never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < g.tiles; t += gridDim.x) {
      if (lane == 0) ok = mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < g.k_blocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&full[stage], phase, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t b0 = a0 + L::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a0 + kk * kUmmaK * 2, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b0 + kk * kUmmaK * 2, 16, 1024);
            mma_f16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      record_timeout(status, abort_flag);
      mma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lg = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
    Epi epi(ep);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < g.tiles; t += gridDim.x) {
      const int mt = t / g.n_tiles, nt = t - (t / g.n_tiles) * g.n_tiles;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      epi.tile(tmem_base + lane_off + static_cast<uint32_t>(acc * BN), mt, nt, lg, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) record_timeout(status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem_base, L::kTmemCols);
}

}  // namespace flp
