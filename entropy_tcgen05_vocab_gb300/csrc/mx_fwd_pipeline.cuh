// mx_fwd_pipeline.cuh -- log-prob and entropy with the logits formed on the
// block-scaled tensor-core path (tcgen05.mma kind::mxf8f6f4).
//
// DeepSeek-V4 book ch. 19, "1. FP4 in OPD": every forward that needs no
// backward -- rollout, the teachers, and the reference model whose
// log-probs give the KL baseline -- runs in native 4-bit precision.  Here
// the head is MXFP4 (E2M1 codes, one E8M0 scale per 32, in the layout of
// flp_mx_head_quantize) and the scored hidden rows are quantised to MXFP8
// (E4M3 codes, one E8M0 scale per 32) once per call; the logits come out of
// the block-scaled MMA, with the scales applied inside it, at twice the
// bf16 rate, and the epilogue is the forward's online log-sum-exp/entropy
// fold (lse_epilogue.cuh).
//
// CTA pairs (cluster of 2), persistent, one item = (256-row tile,
// vocabulary split) as in vocab_pipeline.cuh, on 256-row x 448-column tiles:
// two N = 224 MMAs, one per 224-row tile of the head, share the A operand
// (as the bf16 forward's 512-column tiles do) and fill 448 TMEM columns, one
// accumulator buffer.  Per CTA, an operand ring of kMxFStages stages of one
// 128-wide k-chunk each:
//   A     128 rows x 128 E4M3, 128B-swizzled
//   B0/1  112 rows x 128 E2M1 of head tiles 2 vt and 2 vt + 1, in the padded
//         layout the MMA reads (each 16 elements as 8 bytes of codes and an
//         8-byte gap, written so by the tensor-map copy of type
//         16U4_ALIGN16B), 128B-swizzled
// and a scale ring of kMxFSfStages entries, one per k-chunk: the scale atoms
// of A's 128 rows (512 B) and of both whole 224-row head tiles (1 KB each:
// every CTA of the pair needs the scales of all N columns).  The scale ring
// has its own producer lane, so a chunk's atoms are in shared memory well
// before its operands.
// TMEM: the accumulator at [0, 448) (MMA 0 at columns [0, 224), MMA 1 at
// [224, 448), so tile column c is vocabulary column 448 vt + c), then
// kMxFSlots slots of 20 scale columns (4 for A, 8 per head tile).  Per
// k-chunk a scale-copier warp copies the chunk's five atoms into the chunk's
// slot with tcgen05.cp (the layout the block-scaled MMA reads; see
// mx_pipeline.cuh), commits that to the slot's "ready" barrier and frees the
// ring entry; the MMA issuer waits for "ready" and the operand stage, issues
// the four K = 32 steps of both MMAs with scale id = step, and commits once
// to release the stage.  The slots are fewer than the stages, so before it
// rewrites slot g % kMxFSlots for k-chunk g the copier waits for the release
// of k-chunk g - kMxFSlots, whose MMAs were that slot's last readers.  The
// tensor pipe runs a copy after the MMAs issued before it, so the earlier
// the copier issues a chunk's copies -- with the atoms already in shared
// memory, right after that release -- the less the chunk's MMAs wait.
// (With the copies and that wait on the issuer's own thread, the issuer
// spent about 12 % of its time in that wait and a call took a quarter
// longer.)  Eight epilogue warps (two per TMEM lane quarter, 224 columns
// each) fold the accumulator 32 columns at a time.
#pragma once

#include "launch.h"
#include "mx_pipeline.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

constexpr int kMxFStages = 4;
constexpr int kMxFSlots = 3;
constexpr int kMxFSfStages = 8;
// warps: 0 operand producer, 1 TMEM allocation + MMA issuer, 2..9 epilogue,
// 10 scale copier (leader CTA), 11 scale producer
constexpr int kMxFScaleWarp = 2 + kMxFEpiWarps;
constexpr int kMxFSfProdWarp = kMxFScaleWarp + 1;
constexpr int kMxFThreads = 32 * (kMxFSfProdWarp + 1);
// The copier's parity wait for the release of chunk g - kMxFSlots is
// unambiguous: that stage's next release (chunk g - kMxFSlots + kMxFStages)
// comes after chunk g's MMAs, which wait for this copier.
static_assert(kMxFStages > kMxFSlots, "the release waited for is its stage's latest");

struct MxFwdLayout {
  static constexpr int kA = kBM * kMxChunk;             // 16384: 128 rows x 128 E4M3
  static constexpr int kB = kMxBRows * kMxChunk;        // 14336: padded E2M1 of one head tile
  static constexpr int kBTx = kMxBRows * kMxChunk / 2;  // 7168: code bytes the copy counts
  static constexpr int kSfa = 512;
  static constexpr int kSfb = 1024;                     // per head tile
  static constexpr int kOffB0 = kA;
  static constexpr int kOffB1 = kA + kB;
  static constexpr int kStage = kA + 2 * kB;            // 45056
  static constexpr int kTx = kA + 2 * kBTx;             // operand bytes one CTA's copies count
  static constexpr int kOffSfb0 = kSfa;                 // within a scale-ring entry
  static constexpr int kOffSfb1 = kOffSfb0 + kSfb;
  static constexpr int kSfStage = kSfa + 2 * kSfb;      // 2560
  static constexpr int kRingBytes = kMxFStages * kStage;
  static constexpr int kSfRingBytes = kMxFSfStages * kSfStage;
  static constexpr int kBarrierBytes =
      8 * (2 * kMxFStages + kMxFSlots + 4 + 2 * kMxFSfStages) + 32;
  static constexpr int kSmemBytes = kRingBytes + kSfRingBytes + kBarrierBytes + 1024;
  static constexpr int kTmemCols = 512;
  static constexpr int kAccCols = kMxFwdTileCols;        // 448
  static constexpr int kSfCols = 20;
};
static_assert(MxFwdLayout::kAccCols == 2 * kMxBN, "two head tiles per tile");
static_assert(MxFwdLayout::kStage % 1024 == 0 && MxFwdLayout::kOffB1 % 1024 == 0,
              "swizzled operands stay aligned to swizzle atoms");
static_assert(MxFwdLayout::kRingBytes % 128 == 0 && MxFwdLayout::kSfStage % 128 == 0 &&
                  MxFwdLayout::kOffSfb0 % 128 == 0 && MxFwdLayout::kOffSfb1 % 128 == 0,
              "tensor-copy destinations are 128-byte aligned");
static_assert(MxFwdLayout::kAccCols + kMxFSlots * MxFwdLayout::kSfCols <= MxFwdLayout::kTmemCols,
              "scale columns fit beside the accumulator");
static_assert(MxFwdLayout::kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Epi as in vocab_pipeline.cuh (tile() gets nchunks of 32 columns).  Maps:
// tmA the MXFP8 codes of the scored rows (uint8, box 128 x 128), tmB the
// head's codes (16U4_ALIGN16B, box 128 x 112), tmSfa / tmSfb the scale atoms
// (uint8 rows of 16 bytes, boxes 16 x 32 and 16 x 64).  sch.k_blocks counts
// 128-wide k-chunks and sch.vocab_tiles 448-column tiles.  Launched with a
// cluster dimension of 2 and kMxFThreads threads.
template <class Epi>
__global__ void __launch_bounds__(kMxFThreads, 1)
    mx_fwd_pipeline_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmSfa,
                           const __grid_constant__ CUtensorMap tmSfb, const Schedule sch,
                           const uint32_t idesc, const typename Epi::Params ep, uint32_t *status) {
  using L = MxFwdLayout;
  constexpr int CG = 2;
  constexpr int kHalves = kMxFEpiWarps / 4;
  constexpr int kWarpCols = L::kAccCols / kHalves;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sring = smem + L::kRingBytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(sring + L::kSfRingBytes);
  uint64_t *empty = full + kMxFStages;
  uint64_t *afull = empty + kMxFStages;  // accumulator ready for the epilogue
  uint64_t *aempty = afull + 1;          // accumulator drained
  uint64_t *drain = aempty + 1;          // MMA issuer's teardown
  uint64_t *sready = drain + 1;          // [kMxFSlots] a k-chunk's scales are in TMEM
  uint64_t *sdrain = sready + kMxFSlots;  // scale copier's teardown
  uint64_t *sfull = sdrain + 1;           // [kMxFSfStages] a k-chunk's atoms landed (leader)
  uint64_t *sempty = sfull + kMxFSfStages;  // [kMxFSfStages] the copier's copies read them
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sempty + kMxFSfStages);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // k-chunks the peer's operand [0] and scale [1] producers issued (written
  // at teardown)
  volatile uint32_t *peer_issued = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG;
  const int num_units = gridDim.x / CG;
  const int kc_n = sch.k_blocks;  // 128-wide k-chunks
  const uint64_t lim = wait_limit(sch.wait_ns);
  uint32_t issued = 0;     // operand producer: k-chunks issued
  uint32_t sf_issued = 0;  // scale producer: k-chunks issued

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxFStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(afull, 1);
    mbar_init(aempty, kMxFEpiWarps * CG);
    mbar_init(drain, 1);
    for (int s = 0; s < kMxFSlots; ++s) mbar_init(&sready[s], 1);
    mbar_init(sdrain, 1);
    for (int s = 0; s < kMxFSfStages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1);
    }
    *abort_flag = 0;
    peer_issued[0] = 0;
    peer_issued[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSfa);
    prefetch_tmap(&tmSfb);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, L::kTmemCols);
    tmem_relinquish<CG>();
  }
  pipe_sync<CG>();
  const uint32_t tmem_base = *tmem_slot;

  // The producer, the MMA issuer and the scale copier run on one lane each
  // (the other lanes of their warps wait at the end): no warp-wide exchange
  // sits between one k-chunk's MMAs and the next's.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      const uint32_t full_dst = mapa_shared(smem_u32(full), 0);
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        const int arow = mt * (kBM * CG) + static_cast<int>(rank) * kBM;
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int t0 = 2 * vt, t1 = 2 * vt + 1;  // the tile's two 224-row head tiles
          const int brow0 = t0 * kMxBN + static_cast<int>(rank) * kMxBRows;
          const int brow1 = t1 * kMxBN + static_cast<int>(rank) * kMxBRows;
          for (int c = 0; c < kc_n; ++c) {
            ok = mbar_wait(&empty[st], ph ^ 1u, abort_flag, lim);
            if (!ok) break;
            uint8_t *base = smem + st * L::kStage;
            if (leader) mbar_arrive_expect_tx(&full[st], CG * L::kTx);
            const uint32_t fb = full_dst + st * 8;
            tma_load_2d_pair(base, &tmA, fb, c * kMxChunk, arow);
            tma_load_2d_pair(base + L::kOffB0, &tmB, fb, c * kMxChunk, brow0);
            tma_load_2d_pair(base + L::kOffB1, &tmB, fb, c * kMxChunk, brow1);
            ++issued;
            if (++st == kMxFStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (warp == kMxFSfProdWarp) {
    // ------------------------------------------------------ scale producer
    // Both CTAs' atoms counted on the leader's barrier, as the operands are.
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      const uint32_t sfull_dst = mapa_shared(smem_u32(sfull), 0);
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        const int ablk = mt * CG + static_cast<int>(rank);  // 128-row block of the A atoms
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int t0 = 2 * vt, t1 = 2 * vt + 1;
          for (int c = 0; c < kc_n; ++c) {
            ok = mbar_wait(&sempty[st], ph ^ 1u, abort_flag, lim);
            if (!ok) break;
            uint8_t *base = sring + st * L::kSfStage;
            if (leader) mbar_arrive_expect_tx(&sfull[st], CG * L::kSfStage);
            const uint32_t fb = sfull_dst + st * 8;
            tma_load_2d_pair(base, &tmSfa, fb, 0, (ablk * kc_n + c) * 32);
            tma_load_2d_pair(base + L::kOffSfb0, &tmSfb, fb, 0, (t0 * kc_n + c) * 64);
            tma_load_2d_pair(base + L::kOffSfb1, &tmSfb, fb, 0, (t1 * kc_n + c) * 64);
            ++sf_issued;
            if (++st == kMxFSfStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int st = 0;
      uint32_t ph = 0, aph = 0, g = 0;  // g: k-chunks consumed
      bool ok = true;
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          ok = mbar_wait(aempty, aph ^ 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          for (int c = 0; c < kc_n; ++c) {
            // the scale copier put this k-chunk's scales into its slot, then
            // the operand stage landed
            ok = mbar_wait(&sready[g % kMxFSlots], (g / kMxFSlots) & 1u, abort_flag, lim) &&
                 mbar_wait(&full[st], ph, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = smem_u32(smem + st * L::kStage);
            const uint32_t sf =
                tmem_base + static_cast<uint32_t>(L::kAccCols + (g % kMxFSlots) * L::kSfCols);
#pragma unroll
            for (int j = 0; j < kMxChunk / kMxUmmaK; ++j) {
              const uint64_t ad = sdesc_sw128(tb + j * kMxUmmaK, 16, 1024);
              const uint64_t bd0 = sdesc_sw128(tb + L::kOffB0 + j * kMxUmmaK, 16, 1024);
              const uint64_t bd1 = sdesc_sw128(tb + L::kOffB1 + j * kMxUmmaK, 16, 1024);
              const uint32_t id = idesc_mx_sf(idesc, static_cast<uint32_t>(j));
              const uint32_t acc = (c | j) != 0 ? 1u : 0u;
              mma_mx_pair(tmem_base, ad, bd0, id, sf, sf + 4, acc);
              mma_mx_pair(tmem_base + kMxBN, ad, bd1, id, sf, sf + 12, acc);
            }
            mma_commit_pair(&empty[st], 0x3);
            ++g;
            if (++st == kMxFStages) {
              st = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(afull, 0x3);  // the accumulator is ready
          aph ^= 1u;
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (warp == kMxFScaleWarp) {
    // ------------------------------------------------------- scale copier
    // Copies each k-chunk's five scale atoms from its ring entry into the
    // chunk's TMEM slot, commits that to the slot's "ready" barrier and, once
    // the copies have read the entry, frees it in both CTAs.  A slot is
    // rewritten only after the MMAs of the chunk kMxFSlots earlier, its last
    // readers, were released; waiting for that here, off the MMA issuer,
    // keeps the issuer's thread on MMAs.  The release also paces this warp:
    // it never runs more than kMxFSlots chunks ahead, so each "ready" phase
    // is consumed before the slot's next one.
    if (leader && lane == 0) {
      int st = 0;
      uint32_t ph = 0, g = 0;
      bool ok = true;
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          for (int c = 0; c < kc_n; ++c) {
            ok = mbar_wait(&sfull[st], ph, abort_flag, lim);
            if (ok && g >= static_cast<uint32_t>(kMxFSlots)) {
              const uint32_t gp = g - kMxFSlots;
              ok = mbar_wait(&empty[gp % kMxFStages], (gp / kMxFStages) & 1u, abort_flag, lim);
            }
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = smem_u32(sring + st * L::kSfStage);
            const uint32_t sf =
                tmem_base + static_cast<uint32_t>(L::kAccCols + (g % kMxFSlots) * L::kSfCols);
            tmem_cp_32x128b_x4_pair(sf, sdesc_rows16(tb));
            tmem_cp_32x128b_x4_pair(sf + 4, sdesc_rows16(tb + L::kOffSfb0));
            tmem_cp_32x128b_x4_pair(sf + 8, sdesc_rows16(tb + L::kOffSfb0 + 512));
            tmem_cp_32x128b_x4_pair(sf + 12, sdesc_rows16(tb + L::kOffSfb1));
            tmem_cp_32x128b_x4_pair(sf + 16, sdesc_rows16(tb + L::kOffSfb1 + 512));
            mma_commit_pair_local(&sready[g % kMxFSlots]);
            mma_commit_pair(&sempty[st], 0x3);
            ++g;
            if (++st == kMxFSfStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int lg = warp & 3;
    const int half = (warp - 2) / 4;
    const uint32_t lane_off = (static_cast<uint32_t>(lg * 32) << 16) +
                              static_cast<uint32_t>(half * kWarpCols);
    const uint32_t aempty_dst = mapa_shared(smem_u32(aempty), 0);
    Epi epi(ep);
    uint32_t aph = 0;
    bool ok = true;
    for (int it = unit; ok && it < sch.items; it += num_units) {
      int mt, sp, vt0, vt1;
      sch.item(it, mt, sp, vt0, vt1);
      const int row = mt * (kBM * CG) + static_cast<int>(rank) * kBM + lg * 32 + lane;
      epi.begin(mt, row);
      for (int vt = vt0; vt < vt1; ++vt) {
        if (lane == 0) ok = mbar_wait(afull, aph, abort_flag, lim);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        epi.tile(tmem_base + lane_off, vt * L::kAccCols + half * kWarpCols, kWarpCols / 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(aempty_dst);
        aph ^= 1u;
      }
      if (!ok) break;
      epi.end(sp * kHalves + half, row);
    }
    if (!ok && lane == 0) record_timeout<CG>(status, abort_flag);
  }

  // Teardown (as in vocab_pipeline_kernel, for both rings).
  if ((warp == 0 || warp == kMxFSfProdWarp) && lane == 0 && !leader) {
    const int k = warp == 0 ? 0 : 1;
    const uint32_t pi = mapa_shared(smem_u32(const_cast<uint32_t *>(peer_issued + k)), 0);
    st_cluster_u32(pi, warp == 0 ? issued : sf_issued);
  }
  pipe_sync<CG>();
  if (*abort_flag) {
    if (leader && lane == 0) {
      if (warp == 0)
        drain_copies<kMxFStages, CG>(full, issued, peer_issued[0], L::kTx);
      else if (warp == kMxFSfProdWarp)
        drain_copies<kMxFSfStages, CG>(sfull, sf_issued, peer_issued[1], L::kSfStage);
      else if (warp == 1)
        drain_mmas<CG>(drain);
      else if (warp == kMxFScaleWarp)
        drain_mmas<CG>(sdrain);  // the scale copies
    }
    pipe_sync<CG>();
  }
  if (warp == 1) tmem_dealloc<CG>(tmem_base, L::kTmemCols);
}

}  // namespace flp
