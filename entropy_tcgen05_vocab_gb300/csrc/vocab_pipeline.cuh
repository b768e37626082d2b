// vocab_pipeline.cuh -- the persistent tensor-core pipeline that streams the
// LM-head weight W past tiles of hidden-state rows and hands each FP32 logit
// tile, straight out of tensor memory, to an epilogue.
//
// This is the "output layer on the rows it scores, a tile at a time" loop of
// miles PR #4645 ("How it works": Op) with the tile living in TMEM instead
// of a [tile, vocab] buffer: no logit ever reaches global memory.
//
// Work decomposition.  Rows are cut into row tiles of 128 x CG rows, the
// vocabulary into tiles of BN columns (NOPS x BN with SHARED_A).  A work
// item is (row tile, vocabulary split): one CTA (CG = 1) or one CTA pair
// (CG = 2) sweeps the split's vocabulary tiles for its row tile, keeping
// per-row running state in registers, and emits one partial state per row
// and item.  Items are ordered band by band (a band = `band` consecutive row
// tiles, all splits of the band, row tiles fastest) so the CTAs resident at
// one time share the same weight tiles and each W tile is read from HBM
// about once per band while the band's hidden rows stay in L2.  Persistent
// CTAs (pairs) take items round robin.
//
// Roles (64 + 32 x EPIW threads per CTA, plus 320 with MX):
//   warp 0     TMA producer: A (hidden rows, K-major) and B (W rows, K-major)
//              per 64-wide K block into a STAGES-deep ring of 128B-swizzled
//              shared-memory stages.
//   warp 1     TMEM allocation + tcgen05.mma issue (one elected lane),
//              M = 128 x CG, N = BN, K = 16 per instruction, FP32 accumulators
//              in NACC TMEM buffers (2: the epilogue of one tile overlaps the
//              MMAs of the next; 1: the producer keeps filling stages while
//              the epilogue drains the single buffer).
//   warps 2..  EPIW epilogue warps: tcgen05.ld of their 32 TMEM lanes (= 32
//              rows), 32 columns at a time, folded by the Epi policy; with
//              EPIW = 8 two warps share each lane quarter and split its
//              columns.
//   MX only    eight converter warps and two relay warps (below).
//
// MX: the second GEMM's B operand (a teacher head) is stored in MXFP4 (E2M1
// elements with an E8M0 scale per 32, in the blocked layout of MxOperand).
// Eight converter warps per CTA own it, in two groups of four that take
// alternate k-blocks, and a ring of kDSlots decoded slots, one deeper than
// the stage ring.  Each warp keeps a ring of kQStages small staging buffers
// filled with bulk copies of its 32 rows' codes and scales, ahead of the
// MMAs.  For each of its k-blocks a warp waits until the MMAs have released
// the decoded slot ("released"), decodes the codes exactly into bf16 in the
// 128B-swizzled layout a TMA copy would have written, fences them into the
// async proxy and arrives on a CTA-local barrier.  A relay warp per group
// turns the four local arrivals into one arrival on the leader's "converted"
// barrier, which the MMA issuer waits on with the "full" one (the
// cluster-scope release that arrival needs costs about a microsecond).
// Every E2M1 value times a power of two is a bf16 value, so the bf16 MMA
// computes exactly the product with the decoded weights.
//
// CTA pairs (CG = 2, cluster of 2): each CTA loads its own 128 rows of A and
// its half (BN/2 rows) of B; the leader (rank 0) issues tcgen05.mma.cta_group::2
// for the 256 x BN tile, which reads both CTAs' shared memory and writes
// each CTA's 128 rows of the accumulator into that CTA's TMEM.  Both halves'
// TMA bytes complete on the leader's "full" barrier; the leader's commits
// multicast to both CTAs' "empty" and "accumulator full" barriers; both
// CTAs' epilogues arrive on the leader's "accumulator empty" barrier.  This
// halves the B traffic each SM pulls from L2 per flop.
#pragma once

#include <cfloat>
#include <cstdint>

#include "ptx.cuh"
#include "schedule.h"

namespace flp {

constexpr int kBM = 128;         // rows per CTA tile (TMEM lanes)
constexpr int kBK = 64;          // K elements per stage = one 128-byte swizzle row
constexpr int kUmmaK = 16;       // K per tcgen05.mma kind::f16
constexpr int kEpiWarps = 4;                        // epilogue warps of the GEMM kernels
constexpr int kPipeThreads = 64 + 32 * kEpiWarps;

// Threads of a vocabulary-pipeline CTA with EPIW epilogue warps (4 or 8).
// With 8, two warps share each 32-lane TMEM quarter and split its columns.
__host__ __device__ constexpr int pipe_threads(int epiw) { return 64 + 32 * epiw; }
// Eight more warps decode an MX operand and two relay their completion.
__host__ __device__ constexpr int pipe_threads(int epiw, bool mx) {
  return pipe_threads(epiw) + (mx ? 320 : 0);
}

// NOPS independent GEMMs share one tile (the KL pipeline runs the student and
// the teacher head side by side, NOPS = 2).  Per-CTA stage layout:
// [A_0 .. A_{NOPS-1} | B_0 .. B_{NOPS-1}] with B_i holding BN / CG rows; TMEM:
// NACC accumulator buffers (2: the epilogue of one tile overlaps the MMAs of
// the next) of NOPS x BN columns (GEMM op at column offset op * BN).
// SHARED_A: the NOPS GEMMs share one A operand and take their B operands from
// consecutive BN-row blocks of the same matrix, so the vocabulary tile is
// NOPS x BN columns wide (one A load feeds NOPS MMAs of N = BN).
// MXFP4 -> bf16.  A code (sign, e, m) with block scale code s is
// (-1)^sign (e ? 1 + m/2 : m/2) 2^(e - 1 + s - 127), so for s in [2, 252] the
// seven non-zero magnitudes have bf16 exponent fields s-1, s, s, s+1, s+1,
// s+2, s+2 and mantissa 0x40 for the odd magnitude codes from 3.  Per block
// the high and low bytes of the eight bf16 patterns form two 8-entry byte
// tables, and one byte permute looks four elements up at once.  Other scale
// codes (never produced from bf16 weights) take the field-by-field path.
struct MxTable {
  uint32_t hlo, hhi, llo, lhi;
};

__device__ __forceinline__ MxTable mx_table(uint32_t s) {
  const uint32_t f1 = s - 1, f2 = s, f4 = s + 1, f6 = s + 2;  // exponent fields
  MxTable t;
  t.hlo = ((f1 >> 1) << 8) | ((f2 >> 1) << 16) | ((f2 >> 1) << 24);
  t.hhi = (f4 >> 1) | ((f4 >> 1) << 8) | ((f6 >> 1) << 16) | ((f6 >> 1) << 24);
  const uint32_t l1 = (f1 & 1u) << 7, l2 = (f2 & 1u) << 7, l4 = (f4 & 1u) << 7,
                 l6 = (f6 & 1u) << 7;
  t.llo = (l1 << 8) | (l2 << 16) | ((l2 | 0x40u) << 24);
  t.lhi = l4 | ((l4 | 0x40u) << 8) | (l6 << 16) | ((l6 | 0x40u) << 24);
  return t;
}

// Field-by-field decode of one code (any scale code; exponent fields below 1
// flush to zero).
__device__ __forceinline__ uint32_t mx_bf16_slow(uint32_t code, uint32_t s) {
  const uint32_t mag = code & 7u, e = mag >> 1;
  const int32_t ex = static_cast<int32_t>(s + e) - 1;
  const uint32_t mant = (e != 0u) ? (mag & 1u) : 0u;
  const uint32_t bits = ((code & 8u) << 12) | (static_cast<uint32_t>(ex) << 7) | (mant << 6);
  return (mag != 0u && ex > 0 && ex < 255) ? bits : ((code & 8u) << 12);
}

// PTX prmt in its default mode: selector nibble i picks byte (nibble & 7) of
// {a, b} for result byte i, replicated from that byte's top bit when the
// nibble's top bit is set.
__device__ __forceinline__ uint32_t prmt_sign(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Eight codes (one word, element i in nibble i) -> four bf16 pairs.
__device__ __forceinline__ void mx_word(uint32_t w, const MxTable &t, uint32_t s, bool fast,
                                        uint32_t (&o)[4]) {
  if (fast) {
    const uint32_t sel0 = w & 0x7777u, sel1 = (w >> 16) & 0x7777u;
    const uint32_t h0 = __byte_perm(t.hlo, t.hhi, sel0), l0 = __byte_perm(t.llo, t.lhi, sel0);
    const uint32_t h1 = __byte_perm(t.hlo, t.hhi, sel1), l1 = __byte_perm(t.llo, t.lhi, sel1);
    // Signs: the top bit of byte k of w is the sign of element 2k+1, of w << 4
    // the sign of element 2k; a permute in sign-replicating mode spreads them
    // to the top bytes of each bf16 pair.
    const uint32_t w4 = w << 4;
    o[0] = __byte_perm(l0, h0, 0x5140) | (prmt_sign(w4, w, 0xC080u) & 0x80008000u);
    o[1] = __byte_perm(l0, h0, 0x7362) | (prmt_sign(w4, w, 0xD090u) & 0x80008000u);
    o[2] = __byte_perm(l1, h1, 0x5140) | (prmt_sign(w4, w, 0xE0A0u) & 0x80008000u);
    o[3] = __byte_perm(l1, h1, 0x7362) | (prmt_sign(w4, w, 0xF0B0u) & 0x80008000u);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = mx_bf16_slow((w >> (8 * i)) & 15u, s) | (mx_bf16_slow((w >> (8 * i + 4)) & 15u, s) << 16);
  }
}

// One row of 64 MXFP4 elements -> 64 bf16 written as the row of a
// 128B-swizzled K-major tile: 16-byte chunk c (elements 8c .. 8c+7) goes to
// chunk position c ^ (row % 8) of the row's 128 bytes.
__device__ __forceinline__ void mx_decode_row(const uint8_t *codes, const uint8_t *sc,
                                              uint8_t *row_base, int row) {
  const uint4 q0 = *reinterpret_cast<const uint4 *>(codes);
  const uint4 q1 = *reinterpret_cast<const uint4 *>(codes + 16);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const uint32_t s0 = sc[0], s1 = sc[1];
  const MxTable t0 = mx_table(s0), t1 = mx_table(s1);
  const bool f0 = s0 >= 2u && s0 <= 252u, f1 = s1 >= 2u && s1 <= 252u;
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // chunk c: elements 8c .. 8c+7 = code word c
    uint32_t o[4];
    if (c < 4)
      mx_word(w[c], t0, s0, f0, o);
    else
      mx_word(w[c], t1, s1, f1, o);
    *reinterpret_cast<uint4 *>(row_base + ((c ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The (vocabulary tile, k-block) sequence a CTA (pair) works through, in the
// order of its items; used to run ahead of the MMAs.
struct KSeq {
  int it, vt, vt1, kb;
  bool valid;
  __device__ __forceinline__ void load(const Schedule &s) {
    valid = it < s.items;
    if (valid) {
      int mt, sp, vt0;
      s.item(it, mt, sp, vt0, vt1);
      vt = vt0;
    }
  }
  __device__ __forceinline__ void first(const Schedule &s, int unit) {
    it = unit;
    kb = 0;
    load(s);
  }
  __device__ __forceinline__ void next(const Schedule &s, int num_units) {
    if (++kb < s.k_blocks) return;
    kb = 0;
    if (++vt < vt1) return;
    it += num_units;
    load(s);
  }
};

template <int BN, int STAGES, int NOPS = 1, int CG = 1, int NACC = 2, bool SHARED_A = false,
          bool MX = false>
struct PipeLayout {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kAOps = SHARED_A ? 1 : NOPS;
  static constexpr int kBRows = BN / CG;
  static constexpr int kBBytes = kBRows * kBK * 2;
  // MX: the second GEMM's B lives in a ring of kDSlots decoded slots of its
  // own, one deeper than the stage ring (the decode handshake needs the slack).
  static constexpr int kDSlots = MX ? STAGES + 1 : 0;
  static constexpr int kDMod = MX ? kDSlots : 1;  // index arithmetic MX = false never uses
  static constexpr int kStageBytes = kAOps * kABytes + (MX ? NOPS - 1 : NOPS) * kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes + kDSlots * kBBytes;
  static constexpr int kTileCols = SHARED_A ? NOPS * BN : BN;  // vocabulary columns per tile
  static constexpr int kAccCols = NOPS * BN;
  static constexpr int kTmemCols = NACC * kAccCols;
  static_assert(NACC == 1 || NACC == 2, "one or two accumulator buffers");
  static constexpr int kBarrierBytes = 8 * (2 * STAGES + 5) + 16;
  // MX: a "converted" barrier per stage, then for each of the eight
  // converter warps (two groups of four, taking alternate k-blocks) a ring of
  // kQStages staging buffers (a "staged" barrier each) holding its 32 B rows'
  // codes (32 bytes each) and scale codes (2 bytes each) of one k-block.
  static constexpr int kCvtWarps = 8;
  static constexpr int kQStages = 2;
  static constexpr int kMxBarrierBytes = MX ? 8 * (3 * kDSlots + kCvtWarps * kQStages) : 0;
  static constexpr int kQCodeBytes = 32 * 32;
  static constexpr int kQBytes = MX ? 32 * 34 : 0;  // one warp's slot
  static constexpr int kQOffset =
      (kRingBytes + kBarrierBytes + kMxBarrierBytes + 127) / 128 * 128;
  // + 1024 so the stage ring can be aligned to a swizzle atom.
  static constexpr int kSmemBytes = kQOffset + kCvtWarps * kQStages * kQBytes + 1024;
  static_assert(!MX || (NOPS == 2 && !SHARED_A && kBRows == 128),
                "the MX operand is the second GEMM's B, 128 rows per CTA");
  static_assert(kQBytes % 16 == 0, "staging buffers stay 16-byte aligned");
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM columns must be a power of two");
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
};

// Sets this CTA's abort flag (and, for a pair, the peer's) and counts the
// timeout in the device status word.
template <int CG>
__device__ __forceinline__ void record_timeout(uint32_t *status, volatile int *abort_flag) {
  *abort_flag = 1;
  if (CG == 2) {
    const uint32_t peer = cluster_ctarank() ^ 1u;
    st_cluster_u32(mapa_shared(smem_u32(const_cast<int *>(abort_flag)), peer), 1u);
  }
  atomicAdd(status + kStatTimeout, 1u);
}

__device__ __forceinline__ void record_timeout(uint32_t *status, volatile int *abort_flag) {
  record_timeout<1>(status, abort_flag);
}

// Teardown after a wait gave up (the abort flag is set once every role has
// left its loop).  The producers may have left operand copies in flight and
// the MMA issuer MMAs that still read shared memory and write TMEM; both are
// waited for before TMEM is freed and before a CTA exits.
//
// drain_copies runs in the thread that arms the "full" barriers (the
// leader's producer lane).  `own` and `peer` are the k-block iterations the
// leader's and (pair) the peer's producer issued.  Every iteration that may
// still be in flight lies in the last STAGES of max(own, peer): a producer
// issues iteration i only after the MMAs released iteration i - STAGES, so
// neither runs more than STAGES ahead of the MMAs, and each of those stages
// holds one of them.  In a pair the two producers may have stopped at
// different iterations.  An iteration the leader never armed but the peer
// issued is armed now for the peer's bytes alone; one the leader armed but
// the peer never issued has the peer's missing bytes counted as arrived.
// Then each phase completes once the copies really issued have landed.
template <int STAGES, int CG>
__device__ __forceinline__ void drain_copies(uint64_t *full, uint32_t own, uint32_t peer,
                                             uint32_t cta_stage_bytes) {
  const uint32_t hi = own > peer ? own : peer;
  const uint32_t lo = hi > static_cast<uint32_t>(STAGES) ? hi - STAGES : 0u;
  for (uint32_t i = lo; i < hi; ++i) {
    uint64_t *bar = &full[i % STAGES];
    if (CG == 2) {
      if (i >= own)
        mbar_arrive_expect_tx(bar, cta_stage_bytes);
      else if (i >= peer)
        mbar_complete_tx(bar, cta_stage_bytes);
    }
    int never = 0;
    mbar_wait(bar, (i / STAGES) & 1u, &never);
  }
}

// Run by the MMA-issuing thread: waits until every MMA it issued has
// completed (a commit tracks all of the thread's earlier tcgen05 operations).
template <int CG>
__device__ __forceinline__ void drain_mmas(uint64_t *drain) {
  if (CG == 2)
    mma_commit_pair_local(drain);
  else
    mma_commit(drain);
  int never = 0;
  mbar_wait(drain, 0, &never);
}

template <int CG>
__device__ __forceinline__ void pipe_sync() {
  tc_fence_before();
  if (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
}

// Epi must provide:
//   struct Params;
//   __device__ Epi(const Params&);
//   __device__ void begin(int mt, int row);               row = global scored row of this thread
//   __device__ void tile(uint32_t taddr, int col0, int nchunks);
//                       taddr = TMEM address of this warp's lanes at its first column (the
//                       same columns of GEMM op at + op * BN); col0 = first vocabulary column;
//                       nchunks = 32-column chunks this warp folds
//   __device__ void end(int slot, int row);               slot = split * (EPIW / 4) + column half
// CG = 2 kernels must be launched with a cluster dimension of 2.

// Called by all 32 lanes of a warp after they stored their rows' partial
// states for one item: returns (to the whole warp) true if this warp is the
// last of `expected` arrivals for its 32-row group, so every split's partial
// of these rows is complete and visible to it (fence, count, fence: the last
// arriver merges).  Warp-local on purpose: no barrier across warps that a
// timed-out warp could leave waiting.
__device__ __forceinline__ bool last_arrival(uint32_t *counter, uint32_t expected) {
  __threadfence();
  __syncwarp();
  uint32_t last = 0;
  if ((threadIdx.x & 31) == 0) last = atomicAdd(counter, 1u) == expected - 1u;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

template <int BN, int STAGES, int NOPS, class Epi, int CG = 1, int NACC = 2, int EPIW = 4,
          bool SHARED_A = false, bool MX = false>
__global__ void __launch_bounds__(pipe_threads(EPIW, MX), 1)
    vocab_pipeline_kernel(const __grid_constant__ CUtensorMap tmA0,
                          const __grid_constant__ CUtensorMap tmB0,
                          const __grid_constant__ CUtensorMap tmA1,
                          const __grid_constant__ CUtensorMap tmB1, const Schedule sch,
                          const uint32_t idesc, const typename Epi::Params ep,
                          uint32_t *status) {
  using L = PipeLayout<BN, STAGES, NOPS, CG, NACC, SHARED_A, MX>;
  static_assert(NOPS == 1 || NOPS == 2, "one or two GEMMs per tile");
  static_assert(EPIW == 4 || EPIW == 8, "four or eight epilogue warps");
  constexpr int kHalves = EPIW / 4;          // warps sharing one TMEM lane quarter
  constexpr int kWarpCols = L::kTileCols / kHalves;  // vocabulary columns one epilogue warp folds
  constexpr bool kPair = CG == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kRingBytes);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // k-block iterations the peer's producer issued (written there at teardown)
  volatile uint32_t *peer_issued = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);
  // MX barriers per decoded slot: "converted" (leader; one relay arrival per
  // CTA), "released" (the MMAs' commit), and this CTA's four decode warps done
  uint64_t *dfull = reinterpret_cast<uint64_t *>(smem + L::kRingBytes + L::kBarrierBytes);
  uint64_t *dempty = dfull + L::kDSlots;
  uint64_t *ldec = dempty + L::kDSlots;
  uint64_t *qfull = ldec + L::kDSlots;  // [8 warps][kQStages]
  uint8_t *dring = smem + STAGES * L::kStageBytes;  // decoded B slots
  uint8_t *qbuf = smem + L::kQOffset;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG;          // CTA (pair) index
  const int num_units = gridDim.x / CG;
  const uint64_t lim = wait_limit(sch.wait_ns);  // limit of the main loops' waits
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
    if (MX) {
      for (int d = 0; d < L::kDSlots; ++d) {
        mbar_init(&dfull[d], CG);   // one relay arrival per CTA
        mbar_init(&dempty[d], 1);   // the MMAs' commit
        mbar_init(&ldec[d], 4);     // the four decode warps of the k-block's group
      }
      for (int q = 0; q < L::kCvtWarps * L::kQStages; ++q) mbar_init(&qfull[q], 1);
    }
    *abort_flag = 0;
    *peer_issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmB0);
    if (NOPS == 2) {
      prefetch_tmap(&tmA1);
      prefetch_tmap(&tmB1);
    }
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
      // the pair's bytes all complete on the leader's "full" barriers
      const uint32_t full_dst = kPair ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        const int arow = mt * (kBM * CG) + static_cast<int>(rank) * kBM;
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          const int brow = vt * L::kTileCols + static_cast<int>(rank) * L::kBRows;
          for (int kb = 0; kb < sch.k_blocks; ++kb) {
            ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, lim);
            if (!ok) break;
            uint8_t *sa = smem + stage * L::kStageBytes;
            uint8_t *sb = sa + L::kAOps * L::kABytes;
            if (leader) mbar_arrive_expect_tx(&full[stage], CG * L::kStageBytes);

            // second GEMM: its own A and B maps, or (SHARED_A) the next BN rows of B
            const CUtensorMap *tb1 = SHARED_A ? &tmB0 : &tmB1;
            const int brow1 = SHARED_A ? brow + BN : brow;
            if (kPair) {
              const uint32_t fb = full_dst + stage * 8;
              tma_load_2d_pair(sa, &tmA0, fb, kb * kBK, arow);
              tma_load_2d_pair(sb, &tmB0, fb, kb * kBK, brow);
              if (NOPS == 2) {
                if (!SHARED_A) tma_load_2d_pair(sa + L::kABytes, &tmA1, fb, kb * kBK, arow);
                if (!MX) tma_load_2d_pair(sb + L::kBBytes, tb1, fb, kb * kBK, brow1);
              }
            } else {
              tma_load_2d(sa, &tmA0, &full[stage], kb * kBK, arow);
              tma_load_2d(sb, &tmB0, &full[stage], kb * kBK, brow);
              if (NOPS == 2) {
                if (!SHARED_A) tma_load_2d(sa + L::kABytes, &tmA1, &full[stage], kb * kBK, arow);
                if (!MX) tma_load_2d(sb + L::kBBytes, tb1, &full[stage], kb * kBK, brow1);
              }
            }
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
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
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t g = 0;  // k-blocks issued (MX: decoded slot g % kDSlots)
      bool ok = true;
      for (int it = unit; ok && it < sch.items; it += num_units) {
        int mt, sp, vt0, vt1;
        sch.item(it, mt, sp, vt0, vt1);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          ok = mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * L::kAccCols);
          for (int kb = 0; kb < sch.k_blocks; ++kb) {
            const int dslot = static_cast<int>(g % L::kDMod);
            ok = mbar_wait(&full[stage], phase, abort_flag, lim);
            if (MX && ok)
              ok = mbar_wait_cluster(&dfull[dslot], (g / L::kDMod) & 1u, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t b0 = a0 + L::kAOps * L::kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
#pragma unroll
              for (int op = 0; op < NOPS; ++op) {
                const uint64_t ad = sdesc_sw128(
                    a0 + (SHARED_A ? 0 : op) * L::kABytes + kk * kUmmaK * 2, 16, 1024);
                const uint32_t bop = (MX && op == 1)
                                         ? smem_u32(dring + dslot * L::kBBytes)
                                         : b0 + op * L::kBBytes;
                const uint64_t bd = sdesc_sw128(bop + kk * kUmmaK * 2, 16, 1024);
                if (kPair)
                  mma_f16_pair(d_tmem + op * BN, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                else
                  mma_f16(d_tmem + op * BN, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
              }
            }
            // frees the stage (in both CTAs of a pair) when these MMAs finish
            if (kPair)
              mma_commit_pair(&empty[stage], 0x3);
            else
              mma_commit(&empty[stage]);
            if (MX) {  // and the decoded slot
              if (kPair)
                mma_commit_pair(&dempty[dslot], 0x3);
              else
                mma_commit(&dempty[dslot]);
            }
            ++g;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          // accumulator ready for the epilogue(s)
          if (kPair)
            mma_commit_pair(&tfull[acc], 0x3);
          else
            mma_commit(&tfull[acc]);
          if (NACC == 2) acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      if (!ok) record_timeout<CG>(status, abort_flag);
    }
    __syncwarp();
  } else if (MX && warp >= 2 + EPIW + L::kCvtWarps) {
    // ------------------------------------------------------------ MX relays
    // Relay warp r forwards group r's "this CTA decoded the stage" (a local
    // barrier the group's four warps arrive on) to the leader's "converted"
    // barrier.  That remote arrive needs a cluster-scope release, which costs
    // about a microsecond; doing it here keeps it off the decode warps.
    if constexpr (MX) {
      const int group = warp - 2 - EPIW - L::kCvtWarps;
      const uint32_t dfull_dst = kPair ? mapa_shared(smem_u32(dfull), 0) : smem_u32(dfull);
      KSeq cur;
      cur.first(sch, unit);
      if (group == 1) cur.next(sch, num_units);
      bool ok = true;
      uint32_t g = static_cast<uint32_t>(group);
      while (cur.valid) {
        const int d = static_cast<int>(g % L::kDMod);
        if (lane == 0) {
          ok = mbar_wait(&ldec[d], (g / L::kDMod) & 1u, abort_flag, lim);
          if (ok) {
            if (kPair)
              mbar_arrive_cluster(dfull_dst + d * 8);
            else
              mbar_arrive(&dfull[d]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        g += 2;
        cur.next(sch, num_units);
        cur.next(sch, num_units);
      }
      if (!ok && lane == 0) record_timeout<CG>(status, abort_flag);
    }
  } else if (MX && warp >= 2 + EPIW) {
    // ------------------------------------------------------------ MX converters
    // Two groups of four warps take alternate k-blocks (group 0 the even
    // ones of this CTA's sequence), so each has two k-blocks of MMA time per
    // decode.  Thread t of warp cw decodes B row 32 (cw % 4) + t of this CTA's
    // half.  Lane 0 keeps the warp's own staging ring kQStages of its
    // k-blocks ahead; a slot is refilled right after the warp decoded it.
    if constexpr (MX) {
      constexpr int QS = L::kQStages;
      const int cw = warp - 2 - EPIW;
      const int group = cw >> 2;
      const int crow = (cw & 3) * 32 + lane;
      const MxOperand &mx = ep.mx;
      uint64_t *wfull = qfull + cw * QS;
      uint8_t *wbuf = qbuf + cw * QS * L::kQBytes;
      KSeq ahead, cur;
      ahead.first(sch, unit);
      cur.first(sch, unit);
      if (group == 1) {
        ahead.next(sch, num_units);
        cur.next(sch, num_units);
      }
      uint32_t issued = 0, consumed = 0;
      // lane 0: stage the k-block `ahead` points at into slot issued % QS
      auto stage_next = [&]() {
        const int q = static_cast<int>(issued % QS);
        const int64_t brow = static_cast<int64_t>(ahead.vt) * L::kTileCols +
                             static_cast<int64_t>(rank) * L::kBRows + (cw & 3) * 32;
        const int64_t blk = static_cast<int64_t>(ahead.kb) * mx.v_pad + brow;
        uint8_t *dst = wbuf + q * L::kQBytes;
        mbar_arrive_expect_tx(&wfull[q], L::kQBytes);
        bulk_load(dst, mx.packed + blk * 32, L::kQCodeBytes, &wfull[q]);
        bulk_load(dst + L::kQCodeBytes, mx.scales + blk * 2, 64, &wfull[q]);
        ++issued;
        ahead.next(sch, num_units);
        ahead.next(sch, num_units);
      };
      if (lane == 0)
        for (int i = 0; i < QS && ahead.valid; ++i) stage_next();
      bool ok = true;
      uint32_t g = static_cast<uint32_t>(group);  // index of `cur` in the CTA's k-block sequence
      while (ok && cur.valid) {
        const int d = static_cast<int>(g % L::kDMod);
        const int q = static_cast<int>(consumed % QS);
        // the MMAs are done with the decoded slot, and the codes have landed
        if (lane == 0) ok = mbar_wait(&dempty[d], ((g / L::kDMod) & 1u) ^ 1u, abort_flag, lim);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) ok = mbar_wait(&wfull[q], (consumed / QS) & 1u, abort_flag, lim);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const uint8_t *src = wbuf + q * L::kQBytes;
        uint8_t *b1 = dring + d * L::kBBytes;
        mx_decode_row(src + lane * 32, src + L::kQCodeBytes + lane * 2, b1 + crow * 128, crow);
        // the MMAs read the rows, and the next bulk copy rewrites the slot,
        // through the async proxy
        fence_async_smem();
        __syncwarp();
        ++consumed;
        if (lane == 0) {
          mbar_arrive(&ldec[d]);  // CTA-scope release; the relay warp forwards it
          if (ahead.valid) stage_next();
        }
        g += 2;
        cur.next(sch, num_units);
        cur.next(sch, num_units);
      }
      if (lane == 0) {
        if (!ok) record_timeout<CG>(status, abort_flag);
        for (uint32_t c = consumed; c < issued; ++c) {  // let the copies in flight land
          int never = 0;
          mbar_wait(&wfull[c % QS], (c / QS) & 1u, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lg = warp & 3;  // the TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;  // which columns of the quarter it folds
    const uint32_t lane_off = (static_cast<uint32_t>(lg * 32) << 16) +
                              static_cast<uint32_t>(half * kWarpCols);
    // the pair's "accumulator empty" barriers live in the leader
    const uint32_t tempty_dst = kPair ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);
    Epi epi(ep);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int it = unit; ok && it < sch.items; it += num_units) {
      int mt, sp, vt0, vt1;
      sch.item(it, mt, sp, vt0, vt1);
      const int row = mt * (kBM * CG) + static_cast<int>(rank) * kBM + lg * 32 + lane;
      epi.begin(mt, row);
      for (int vt = vt0; vt < vt1; ++vt) {
        if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, lim);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        epi.tile(tmem_base + lane_off + static_cast<uint32_t>(acc * L::kAccCols),
                 vt * L::kTileCols + half * kWarpCols, kWarpCols / 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair)
            mbar_arrive_cluster(tempty_dst + acc * 8);
          else
            mbar_arrive(&tempty[acc]);
        }
        if (NACC == 2) acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) break;
      epi.end(sp * kHalves + half, row);
    }
    if (!ok && lane == 0) record_timeout<CG>(status, abort_flag);
  }

  // Teardown.  The peer's producer tells the leader how far it got; after
  // the sync every role has left its loop and the abort flag (set in both
  // CTAs of a pair by record_timeout) is final, so all threads of the pair
  // take the same branch.
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
