// mx_pipeline.cuh -- the KL pipeline with the teacher GEMM on the
// block-scaled tensor-core path (tcgen05.mma kind::mxf8f6f4).
//
// DeepSeek-V4 book ch. 19, "1. FP4 in OPD": the inference-only teacher
// forward runs in native 4-bit precision.  Here the teacher head is MXFP4
// (E2M1 codes, one E8M0 scale per 32) and the teacher's hidden rows are
// quantised to MXFP8 (E4M3 codes, one E8M0 scale per 32) per call, so the
// teacher logits come out of the tensor cores' block-scaled MMA at twice the
// bf16 rate, with the scales applied inside the MMA.  The student stays on
// the bf16/fp16 path, and the epilogue is the KL fold of the bf16 pipeline.
//
// CTA pairs (cluster of 2) on 256-row x 224-column tiles, persistent, one
// item = (256-row tile, vocabulary split) as in vocab_pipeline.cuh.  Two
// operand rings per CTA, each with its own producer warp and (in the leader
// CTA) its own MMA-issuing thread:
//   student ring  kMxSStages stages of kMxSKb 64-wide k-blocks: A_s (128
//                 rows) and B_s (112 rows) bf16, 128B-swizzled, two
//                 tensor-map copies per k-block;
//   teacher ring  kMxTStages stages of one 128-wide k-chunk: A_t (128 x 128
//                 E4M3), B_t (112 x 128 E2M1 in the padded layout the MMA
//                 reads: each 16 elements as 8 bytes of codes and an 8-byte
//                 gap, written so by the tensor-map copy of type
//                 16U4_ALIGN16B), 128B-swizzled, and the scale atoms of A_t's
//                 128 rows (512 B) and of the whole 224-row B_t tile (1 KB:
//                 every CTA of the pair needs the scales of all N columns).
// A scale atom holds the scales of 128 rows for the four 32-element steps
// of a k-chunk: byte (r % 32) * 16 + (r / 32) * 4 + j for row r, step j.
// One tcgen05.cp (32 rows x 16 bytes, to every lane quarter) moves an atom
// into four TMEM columns, which is the layout the block-scaled MMA reads
// (row m's scale at lane m, column m / 32; column n's at lane n % 32 of the
// row's lane quarter, column n / 32; step j in byte j).
// TMEM (512 columns): student accumulator [0, 224), teacher accumulator
// [224, 448), and 12 scale columns per teacher stage from 448 (4 for A, 8 for
// B).  Per 128-wide k-chunk the teacher's issuer copies the chunk's scales
// into its stage's columns, issues four block-scaled MMAs (K = 32, scale
// id = step) into the teacher accumulator and commits once to release the
// stage; the student's issuer issues four bf16 MMAs (K = 16) per k-block
// stage into the student accumulator and commits each stage.  Issuing an
// MMA blocks the thread for about the MMA's own execution time (the tensor
// pipe's queue is shallow), so every other operation an issuing thread adds
// between MMAs -- a commit, a wait -- would stretch the pipe's critical path
// if one thread issued both heads; with two issuers one keeps the pipe fed
// while the other waits or commits.  Small student stages keep more of that
// ring's bytes in flight: with two 128-wide stages the student issuer
// waited for data 44 % of its time.  The copies and MMAs of one thread
// execute in issue order, and a stage's scale columns are rewritten only
// after the MMAs that read them released that stage.  Each issuer
// commits to the accumulators' "full" barrier once per tile (two arrivals)
// and both wait for the epilogue to hand the accumulators back.
// Eight epilogue warps (two per TMEM lane quarter, 112 columns each) fold
// the two accumulators 16 columns at a time with the KL epilogue.
#pragma once

#include "launch.h"
#include "vocab_pipeline.cuh"

namespace flp {

constexpr int kMxBRows = kMxBN / 2;   // B rows per CTA
constexpr int kMxSKb = 1;      // 64-wide k-blocks per student stage
constexpr int kMxSStages = 4;
constexpr int kMxTStages = 3;
// warps: 0 student producer, 1 TMEM allocation + student MMA issuer, 2..9
// epilogue, 10 teacher producer, 11 teacher MMA issuer
constexpr int kMxTProdWarp = 2 + kMxEpiWarps;
constexpr int kMxTMmaWarp = kMxTProdWarp + 1;
constexpr int kMxThreads = 32 * (kMxTMmaWarp + 1);
constexpr int kMxUmmaK = 32;          // K per block-scaled MMA

struct MxPipeLayout {
  static constexpr int kSA = kBM * kBK * 2;             // 16384: one 64-wide k-block of A_s
  static constexpr int kSB = kMxBRows * kBK * 2;        // 14336: one k-block of B_s
  static constexpr int kSStage = kMxSKb * (kSA + kSB);  // A_s k-blocks, then B_s k-blocks
  static constexpr int kTA = kBM * kMxChunk;            // 16384: 128 rows x 128 E4M3
  static constexpr int kTB = kMxBRows * kMxChunk;       // 14336: padded E2M1 in shared memory
  static constexpr int kTBTx = kMxBRows * kMxChunk / 2; // 7168: code bytes the copy counts
  static constexpr int kSfa = 512;
  static constexpr int kSfb = 1024;
  static constexpr int kTStage = 32768;
  static constexpr int kTTx = kTA + kTBTx + kSfa + kSfb;  // bytes one CTA's teacher copies count
  static constexpr int kTRing = kMxSStages * kSStage;
  static constexpr int kRingBytes = kTRing + kMxTStages * kTStage;
  static constexpr int kBarrierBytes = 8 * (2 * kMxSStages + 2 * kMxTStages + 4) + 32;
  static constexpr int kSmemBytes = kRingBytes + kBarrierBytes + 1024;
  static constexpr int kTmemCols = 512;
  static constexpr int kSfCol0 = 2 * kMxBN;
  static constexpr int kSfCols = 12;
};
static_assert(MxPipeLayout::kSStage % 1024 == 0 && MxPipeLayout::kTStage % 1024 == 0,
              "stages stay aligned to swizzle atoms");
static_assert(MxPipeLayout::kTA + MxPipeLayout::kTB + MxPipeLayout::kSfa + MxPipeLayout::kSfb <=
                  MxPipeLayout::kTStage,
              "teacher stage fits");
static_assert(MxPipeLayout::kSfCol0 + kMxTStages * MxPipeLayout::kSfCols <= MxPipeLayout::kTmemCols,
              "scale columns fit beside the accumulators");
static_assert(MxPipeLayout::kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Epi as in vocab_pipeline.cuh (tile() gets nchunks in units of Epi::kChunk).
// Maps: tmAs / tmBs the student rows and head (bf16/fp16, boxes 64 x 128 and
// 64 x 112), tmAt the teacher's MXFP8 codes (uint8, box 128 x 128), tmBt the
// teacher head's codes (16U4_ALIGN16B, box 128 x 112), tmSfa / tmSfb the
// scale atoms (uint8 rows of 16 bytes, boxes 16 x 32 and 16 x 64).
// sch.k_blocks counts 128-wide k-chunks.  Launched with a cluster dimension
// of 2 and kMxThreads threads.
template <class Epi>
__global__ void __launch_bounds__(kMxThreads, 1)
    mx_kl_pipeline_kernel(const __grid_constant__ CUtensorMap tmAs,
                          const __grid_constant__ CUtensorMap tmBs,
                          const __grid_constant__ CUtensorMap tmAt,
                          const __grid_constant__ CUtensorMap tmBt,
                          const __grid_constant__ CUtensorMap tmSfa,
                          const __grid_constant__ CUtensorMap tmSfb, const Schedule sch,
                          const uint32_t idesc_s, const uint32_t idesc_t,
                          const typename Epi::Params ep, uint32_t *status) {
  using L = MxPipeLayout;
  constexpr int CG = 2;
  constexpr int kHalves = kMxEpiWarps / 4;
  constexpr int kWarpCols = kMxBN / kHalves;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *sfull = reinterpret_cast<uint64_t *>(smem + L::kRingBytes);
  uint64_t *sempty = sfull + kMxSStages;
  uint64_t *tfull = sempty + kMxSStages;
  uint64_t *tempty = tfull + kMxTStages;
  uint64_t *afull = tempty + kMxTStages;  // accumulators ready for the epilogue
  uint64_t *aempty = afull + 1;           // accumulators drained
  uint64_t *drain = aempty + 1;           // student issuer's teardown
  uint64_t *tdrain = drain + 1;           // teacher issuer's teardown
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tdrain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // iterations of the two rings the peer's producer issued (written at teardown)
  volatile uint32_t *peer_issued = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG;
  const int num_units = gridDim.x / CG;
  const int kc_n = sch.k_blocks;  // 128-wide k-chunks
  const uint64_t lim = wait_limit(sch.wait_ns);
  uint32_t s_issued = 0, t_issued = 0;  // producer: iterations issued per ring

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxSStages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1);
    }
    for (int s = 0; s < kMxTStages; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 1);
    }
    mbar_init(afull, 2);  // one commit per issuer
    mbar_init(aempty, kMxEpiWarps * CG);
    mbar_init(drain, 1);
    mbar_init(tdrain, 1);
    *abort_flag = 0;
    peer_issued[0] = 0;
    peer_issued[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmAs);
    prefetch_tmap(&tmBs);
    prefetch_tmap(&tmAt);
    prefetch_tmap(&tmBt);
    prefetch_tmap(&tmSfa);
    prefetch_tmap(&tmSfb);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, L::kTmemCols);
    tmem_relinquish<CG>();
  }
  pipe_sync<CG>();
  const uint32_t tmem_base = *tmem_slot;

  // Producers and MMA issuers run on one lane each (the other lanes of their
  // warps wait at the end): no warp-wide exchange sits between one k-chunk's
  // MMAs and the next's.
  if (warp == 0 || warp == kMxTProdWarp) {
    // ----------------------------------------------------------- producers
    // Warp 0 fills the student ring, warp kMxTProdWarp the teacher ring.
    const bool teacher = warp == kMxTProdWarp;
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, issued = 0;
      bool ok = true;
      const uint32_t full_dst = mapa_shared(smem_u32(teacher ? tfull : sfull), 0);
      uint64_t *empty = teacher ? tempty : sempty;
      const int stages = teacher ? kMxTStages : kMxSStages;
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        const int arow = mt * (kBM * CG) + static_cast<int>(rank) * kBM;
        const int ablk = mt * CG + static_cast<int>(rank);  // 128-row block of the scale atoms
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int brow = vt * kMxBN + static_cast<int>(rank) * kMxBRows;
          for (int c = 0; c < kc_n; ++c) {
            ok = mbar_wait(&empty[st], ph ^ 1u, abort_flag, lim);
            if (!ok) break;
            const uint32_t fb = full_dst + st * 8;
            if (teacher) {
              // teacher k-chunk c: codes of A_t and B_t, then the scale atoms
              uint8_t *base = smem + L::kTRing + st * L::kTStage;
              if (leader) mbar_arrive_expect_tx(&tfull[st], CG * L::kTTx);
              tma_load_2d_pair(base, &tmAt, fb, c * kMxChunk, arow);
              tma_load_2d_pair(base + L::kTA, &tmBt, fb, c * kMxChunk, brow);
              tma_load_2d_pair(base + L::kTA + L::kTB, &tmSfa, fb, 0, (ablk * kc_n + c) * 32);
              tma_load_2d_pair(base + L::kTA + L::kTB + L::kSfa, &tmSfb, fb, 0,
                               (vt * kc_n + c) * 64);
              ++issued;
              if (++st == stages) {
                st = 0;
                ph ^= 1u;
              }
            } else {
              // student k-blocks 2c and 2c + 1, kMxSKb per stage
              for (int hb = 0; hb < 2; hb += kMxSKb) {
                if (hb > 0) {
                  ok = mbar_wait(&empty[st], ph ^ 1u, abort_flag, lim);
                  if (!ok) break;
                }
                uint8_t *sa = smem + st * L::kSStage;
                if (leader) mbar_arrive_expect_tx(&sfull[st], CG * L::kSStage);
                const uint32_t fbs = full_dst + st * 8;
                for (int h = 0; h < kMxSKb; ++h) {
                  const int kb = 2 * c + hb + h;
                  tma_load_2d_pair(sa + h * L::kSA, &tmAs, fbs, kb * kBK, arow);
                  tma_load_2d_pair(sa + kMxSKb * L::kSA + h * L::kSB, &tmBs, fbs, kb * kBK, brow);
                }
                ++issued;
                if (++st == stages) {
                  st = 0;
                  ph ^= 1u;
                }
              }
              if (!ok) break;
            }
          }
        }
      }
      if (teacher)
        t_issued = issued;
      else
        s_issued = issued;
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMxTMmaWarp) {
    // --------------------------------------------------------- MMA issuers
    // Warp 1 issues the student's bf16 MMAs, warp kMxTMmaWarp the teacher's
    // scale copies and block-scaled MMAs.  Each thread's commits track only
    // its own tcgen05 operations, so while one issuer waits for a stage or
    // commits, the other keeps the tensor pipe fed.  Both commit to "afull"
    // (two arrivals per tile) and both wait for the epilogue's "aempty".
    if (leader && lane == 0) {
      const bool teacher = warp == kMxTMmaWarp;
      int st = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      uint64_t *full = teacher ? tfull : sfull;
      uint64_t *empty = teacher ? tempty : sempty;
      const int stages = teacher ? kMxTStages : kMxSStages;
      const uint32_t d_student = tmem_base;
      const uint32_t d_teacher = tmem_base + kMxBN;
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          ok = mbar_wait(aempty, aph ^ 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          for (int c = 0; c < kc_n; ++c) {
            ok = mbar_wait(&full[st], ph, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            if (teacher) {
              const uint32_t tb = smem_u32(smem + L::kTRing + st * L::kTStage);
              const uint32_t sf = tmem_base + static_cast<uint32_t>(L::kSfCol0 + st * L::kSfCols);
              tmem_cp_32x128b_x4_pair(sf, sdesc_rows16(tb + L::kTA + L::kTB));
              tmem_cp_32x128b_x4_pair(sf + 4, sdesc_rows16(tb + L::kTA + L::kTB + L::kSfa));
              tmem_cp_32x128b_x4_pair(sf + 8, sdesc_rows16(tb + L::kTA + L::kTB + L::kSfa + 512));
#pragma unroll
              for (int j = 0; j < kMxChunk / kMxUmmaK; ++j) {
                const uint64_t ad = sdesc_sw128(tb + j * kMxUmmaK, 16, 1024);
                const uint64_t bd = sdesc_sw128(tb + L::kTA + j * kMxUmmaK, 16, 1024);
                mma_mx_pair(d_teacher, ad, bd, idesc_mx_sf(idesc_t, static_cast<uint32_t>(j)), sf,
                            sf + 4, (c | j) != 0 ? 1u : 0u);
              }
              mma_commit_pair(&empty[st], 0x3);
              if (++st == stages) {
                st = 0;
                ph ^= 1u;
              }
            } else {
              // student k-blocks 2c and 2c + 1, kMxSKb per stage
              for (int hb = 0; hb < 2; hb += kMxSKb) {
                if (hb > 0) {
                  ok = mbar_wait(&full[st], ph, abort_flag, lim);
                  if (!ok) break;
                  tc_fence_after();
                }
                const uint32_t sa = smem_u32(smem + st * L::kSStage);
#pragma unroll
                for (int h = 0; h < kMxSKb; ++h)
#pragma unroll
                  for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                    const uint64_t ad = sdesc_sw128(sa + h * L::kSA + kk * kUmmaK * 2, 16, 1024);
                    const uint64_t bd = sdesc_sw128(
                        sa + kMxSKb * L::kSA + h * L::kSB + kk * kUmmaK * 2, 16, 1024);
                    mma_f16_pair(d_student, ad, bd, idesc_s, (c | hb | h | kk) != 0 ? 1u : 0u);
                  }
                mma_commit_pair(&empty[st], 0x3);
                if (++st == stages) {
                  st = 0;
                  ph ^= 1u;
                }
              }
              if (!ok) break;
            }
          }
          if (!ok) break;
          mma_commit_pair(afull, 0x3);  // this issuer's accumulator is ready
          aph ^= 1u;
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
        epi.tile(tmem_base + lane_off, vt * kMxBN + half * kWarpCols, kWarpCols / Epi::kChunk);
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

  // Teardown (as in vocab_pipeline_kernel, for both rings and both issuers).
  if (lane == 0 && !leader && (warp == 0 || warp == kMxTProdWarp)) {
    const uint32_t pi = mapa_shared(smem_u32(const_cast<uint32_t *>(peer_issued)), 0);
    if (warp == 0)
      st_cluster_u32(pi, s_issued);
    else
      st_cluster_u32(pi + 4, t_issued);
  }
  pipe_sync<CG>();
  if (*abort_flag) {
    if (leader && lane == 0) {
      if (warp == 0)
        drain_copies<kMxSStages, CG>(sfull, s_issued, peer_issued[0], L::kSStage);
      else if (warp == kMxTProdWarp)
        drain_copies<kMxTStages, CG>(tfull, t_issued, peer_issued[1], L::kTTx);
      else if (warp == 1)
        drain_mmas<CG>(drain);
      else if (warp == kMxTMmaWarp)
        drain_mmas<CG>(tdrain);
    }
    pipe_sync<CG>();
  }
  if (warp == 1) tmem_dealloc<CG>(tmem_base, L::kTmemCols);
}

}  // namespace flp
