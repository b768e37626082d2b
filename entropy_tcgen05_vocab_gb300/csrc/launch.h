// launch.h -- internal interface between the host API (api.cu) and the
// kernel translation units.  Not installed; the public interface is
// include/fusedlogp.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "schedule.h"

namespace flp {

// Forward scoring (and the backward's statistics pass): CTA pairs
// (cta_group::2) on 256-row x 512-column tiles made of two N = 256 MMAs that
// share the A operand, one accumulator buffer (512 TMEM columns), eight
// epilogue warps, 4 stages of 48 KB per CTA.  Against 256-column tiles with
// double-buffered accumulators this needs a quarter less operand traffic per
// flop (48 vs 64 B/clk/SM at full rate), which pays for the epilogue no
// longer overlapping the MMAs.
// Largest number of target tokens per row of the K-candidate forward
// (FLP_MAX_TARGETS in the public header).
constexpr int kMaxTargets = 8;
constexpr int kFwdBN = 256;        // N of one MMA
constexpr int kFwdTileCols = 512;  // vocabulary columns per tile
constexpr int kFwdCG = 2;
constexpr int kFwdStages = 4;
constexpr int kFwdEpiWarps = 8;
// Few scored rows (n <= kSmallRows): single CTAs on
// 128-row x 256-column tiles with double-buffered accumulators.  A pair tile
// would be at least half padding there, and the call is bound by the
// weight stream, not by the tensor cores.
constexpr int kSmallRows = 128;
constexpr int kFwd1Stages = 4;
constexpr int kFwd1EpiWarps = 4;
// Gradient pass of the backward: the same 256 x 512 shared-A tiles, one
// accumulator buffer, eight epilogue warps, 4 stages of 48 KB.
constexpr int kGradBN = 256;
constexpr int kGradTileCols = 512;
constexpr int kGradCG = 2;
constexpr int kGradStages = 4;
constexpr int kGradEpiWarps = 8;
// Tile shape of the KL pipeline (student and teacher accumulators per tile):
// CTA pairs on 256-row x 256-column tiles, 3 stages of 64 KB per CTA, one
// accumulator buffer (2 x 256 TMEM columns).  Against 128-column tiles with
// double-buffered accumulators this needs a third less operand traffic per
// flop, which pays for the epilogue no longer overlapping the MMAs.
constexpr int kKlBN = 256;
constexpr int kKlCG = 2;
constexpr int kKlStages = 3;
constexpr int kKlAcc = 1;
// Eight epilogue warps (two per TMEM lane quarter, each folding half the
// columns) halve the epilogue that the single accumulator buffer exposes.
constexpr int kKlEpiWarps = 8;


// Block-scaled KL (the teacher GEMM on tcgen05.mma kind::mxf8f6f4, E4M3
// hidden rows x E2M1 head, one E8M0 scale per 32): CTA pairs on 256-row x
// 224-column tiles (224 = 512 TMEM columns minus room for the scale factors
// beside the student and teacher accumulators), 128-wide teacher k-chunks,
// eight epilogue warps.  The head's scale atoms are laid out per 224-row
// vocabulary tile (see flp_mx_head_quantize).
constexpr int kMxBN = 224;
constexpr int kMxChunk = 128;
constexpr int kMxEpiWarps = 8;
// Block-scaled forward (E4M3 scored rows x the same E2M1 head): CTA pairs on
// 256-row x 448-column tiles, two N = 224 MMAs (two head tiles) sharing A,
// one accumulator buffer, eight epilogue warps.
constexpr int kMxFwdTileCols = 2 * kMxBN;
constexpr int kMxFEpiWarps = 8;

struct FwdArgs {
  CUtensorMap tmA;  // scored hidden rows [n, H], box 64 x 128
  CUtensorMap tmB;  // W [V, H], box 64 x kFwdBN
  Schedule sch;
  int grid;
  bool bf16;
  const int64_t *targets;  // [T, K]
  int K;                   // targets per row (1 .. kMaxTargets)
  const int64_t *row_idx;
  int64_t T;
  float inv_tau;
  float scale_log2;
  float *pm, *ps, *pb, *zt;  // zt: [n, K]
  uint32_t *counters;  // [ceil(n / 32)] zeroed before the launch
  float *out_logp, *out_ent, *out_lse, *out_ez;
  uint32_t *status;
  const uint32_t *support;  // [T, ld_support] sampling-support words, or null
  int64_t ld_support;
};

struct KlArgs {
  CUtensorMap tmAs, tmAt;  // student / teacher hidden rows, box 64 x 128
  CUtensorMap tmBs, tmBt;  // student / teacher W, box 64 x kKlBN
  Schedule sch;
  int grid;
  bool bf16;
  const int64_t *row_idx;
  int64_t T;
  float *pmt, *pst, *pct, *pms, *pss;  // [splits][n] partial states
  uint32_t *counters;                   // [ceil(n / 32)] zeroed before the launch
  float *out_kl;
  uint32_t *status;
  MxOperand mx;  // teacher head in MXFP4 (packed == null: W_t through tmBt)
};

struct KlBsArgs {
  CUtensorMap tmAs, tmBs;    // student rows [n, H] (box 64 x 128) and head [V, H] (box 64 x 112)
  CUtensorMap tmAt, tmBt;    // teacher MXFP8 codes [n, H] uint8 (box 128 x 128), head codes
                             // [V, H] 16U4_ALIGN16B (box 128 x 112)
  CUtensorMap tmSfa, tmSfb;  // scale atoms as rows of 16 bytes (boxes 16 x 32, 16 x 64)
  Schedule sch;              // k_blocks = H / 128
  int grid;
  bool bf16;
  const int64_t *row_idx;
  int64_t T;
  float *pmt, *pst, *pct, *pms, *pss;
  uint32_t *counters;
  float *out_kl;
  uint32_t *status;
};

struct FwdBsArgs {
  CUtensorMap tmA;           // MXFP8 codes of the scored rows [n, H] uint8, box 128 x 128
  CUtensorMap tmB;           // head codes [V, H] 16U4_ALIGN16B, box 128 x 112
  CUtensorMap tmSfa, tmSfb;  // scale atoms as rows of 16 bytes (boxes 16 x 32, 16 x 64)
  Schedule sch;              // k_blocks = H / 128, vocabulary tiles of kMxFwdTileCols
  int grid;
  const int64_t *targets;    // [T]
  const int64_t *row_idx;
  int64_t T;
  float inv_tau;
  float scale_log2;
  float *pm, *ps, *pb, *zt;
  uint32_t *counters;        // [ceil(n / 32)] zeroed before the launch
  float *out_logp, *out_ent, *out_lse, *out_ez;
  uint32_t *status;
};

struct GradArgs {
  CUtensorMap tmA;  // the chunk's scored hidden rows [R, H], box 64 x 128
  CUtensorMap tmB;  // W [V, H], box 64 x kFwdBN
  Schedule sch;     // over the chunk's R rows
  int grid;
  bool bf16;
  int r0;           // first scored position of the chunk
  int64_t T;
  const int64_t *targets;
  const int64_t *row_idx;
  const float *lse, *ez, *g1, *g2;  // indexed by scored position
  float scale_log2, inv_tau;
  void *G;          // [R, ldg] model dtype
  int64_t ldg;
  uint32_t *status;
  const uint32_t *support;  // [T, ld_support] sampling-support words, or null
  int64_t ld_support;
};

// The dh GEMM's split of its last, partial wave (see dh_split_plan).
struct DhSplit {
  int tiles;       // output tiles of the product
  int full_tiles;  // tiles computed whole
  int tail;        // tiles split along K (tiles - full_tiles)
  int split;       // K segments per tail tile (1: no split)
  int kb_per_seg;  // 64-wide k-blocks per segment
  int items;       // work items of the persistent launch
};
// Minimum k-blocks per K segment, and the 512 KB partial-tile slots the
// backward's workspace holds at most.
constexpr int kDhSplitMinKb = 16;
constexpr int kDhSplitSlots = 80;
constexpr size_t kDhSlotBytes = static_cast<size_t>(256) * 512 * 4;

// Plan of the dh GEMM (M x N output, K contraction) on `units` CTA pairs: if
// its last wave would leave at least half of the pairs idle, its tiles are
// each split into up to units / tail K segments of >= kDhSplitMinKb
// k-blocks, using at most max_slots partial tiles.
DhSplit dh_split_plan(int M, int N, int K, int units, int max_slots);

struct GemmArgs {
  CUtensorMap tmA, tmB;
  int M, N, K;
  int grid;
  DhSplit dh_split;  // dh GEMM only; split 1 (or zero-initialised) = no split
  float *part;       // dh GEMM with a split: dh_split.tail * split slots of kDhSlotBytes
  bool bf16;
  uint32_t *status;
  // dh epilogue: row i of the product goes to dh[row_idx[r0 + i]]
  int r0;
  int64_t T;
  const int64_t *row_idx;
  const uint32_t *rowcnt;  // scored rows per h row (null when row_idx is null)
  void *dh;
  int64_t ld_dh;
  // dW epilogue
  float *dW;
  int64_t ld_dw;
  int accumulate;
  unsigned long long wait_ns;  // limit of the kernel's barrier waits (0: the default)
};

cudaError_t launch_gather(const void *h, int64_t ld_h, const int64_t *row_idx, int64_t n,
                          int64_t T, int64_t H, void *hs, int num_sms, cudaStream_t stream);
cudaError_t launch_fwd_scoring(const FwdArgs &a, cudaStream_t stream);
// The single-CTA variant (tmB box 64 x kFwdBN rows; plan with 128-row tiles
// of kFwdBN columns, in CTAs).
cudaError_t launch_fwd_scoring_1cta(const FwdArgs &a, cudaStream_t stream);
int fwd1_units(int num_sms);
cudaError_t launch_kl(const KlArgs &a, cudaStream_t stream);
cudaError_t launch_grad(const GradArgs &a, cudaStream_t stream);
cudaError_t launch_dh_gemm(const GemmArgs &a, cudaStream_t stream);
cudaError_t launch_dw_gemm(const GemmArgs &a, cudaStream_t stream);
// cnt[r] += 1 for every row_idx entry r in [0, T) (cnt zeroed by the caller).
cudaError_t launch_count_rows(const int64_t *row_idx, int64_t n, int64_t T, uint32_t *cnt,
                              int num_sms, cudaStream_t stream);
int dh_gemm_tiles(int M, int N);
int dw_gemm_tiles(int M, int N);
int gemm_cta_group();
int gemm_units(int num_sms);
int fwd_smem_bytes();
// support[r, w] (w < ld_support) = bits 32w .. 32w+31 of mask row r (a byte
// per token, non-zero = in the support); bits past V and words past
// ceil(V/32) are 0.
cudaError_t launch_pack_support(const uint8_t *mask, int64_t T, int64_t V, int64_t ld_mask,
                                uint32_t *support, int64_t ld_support, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t *status, cudaStream_t stream);
cudaError_t launch_kl_blockscaled(const KlBsArgs &a, cudaStream_t stream);
int kl_bs_units(int num_sms);
cudaError_t launch_fwd_blockscaled(const FwdBsArgs &a, cudaStream_t stream);
int fwd_bs_units(int num_sms);
// MXFP8 quantisation of R rows (row_idx[i], or i, of X [*, ld] bf16/fp16;
// rows outside [0, T) read as zeros) into codes [R, H] and scales: the
// pipeline's 512-byte atoms (atoms = true, rows up to the next multiple of
// 128 get scale 0) or a plain [R, H / 32] array.  H a multiple of 128
// (atoms) or 32.
cudaError_t launch_mxfp8_quantize(const void *X, bool bf16, int64_t R, int64_t H, int64_t ld,
                                  const int64_t *row_idx, int64_t T, uint8_t *codes,
                                  uint8_t *scales, bool atoms, int num_sms, cudaStream_t stream);
// MXFP4 quantisation of W [V, ld_w] into the block-scaled head: codes [V, H/2]
// row-major, scale atoms per 224-row vocabulary tile.
cudaError_t launch_mx_head_quantize(const void *W, bool bf16, int64_t V, int64_t H, int64_t ld_w,
                                    uint8_t *codes, uint8_t *atoms, int num_sms,
                                    cudaStream_t stream);
// CTAs or CTA pairs of each pipeline that can be resident at once.
int fwd_units(int num_sms);
int grad_units(int num_sms);
int kl_units(int num_sms);
int kl_mx_units(int num_sms);
// MXFP4 quantisation of W [V, ld_w] (bf16/fp16) into the blocked layout of
// MxOperand with v_pad rows (rows past V zero); H a multiple of 64.
cudaError_t launch_mxfp4_quantize(const void *W, bool bf16, int64_t V, int64_t H, int64_t ld_w,
                                  int64_t v_pad, uint8_t *packed, uint8_t *scales, int num_sms,
                                  cudaStream_t stream);

}  // namespace flp
