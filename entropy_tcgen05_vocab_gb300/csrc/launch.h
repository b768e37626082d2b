// launch.h -- internal interface between the host API (api.cpp) and the
// kernel translation units.  Not installed; the public interface is
// include/fusedlogp.h.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "schedule.h"

namespace flp {

// Tile shape of the forward scoring pipeline.
constexpr int kFwdBN = 256;
constexpr int kFwdStages = 4;
// Tile shape of the KL pipeline (two accumulators per tile).
constexpr int kKlBN = 128;
constexpr int kKlStages = 3;


struct FwdArgs {
  CUtensorMap tmA;  // scored hidden rows [n, H], box 64 x 128
  CUtensorMap tmB;  // W [V, H], box 64 x kFwdBN
  Schedule sch;
  int grid;
  bool bf16;
  const int64_t *targets;
  const int64_t *row_idx;
  int64_t T;
  float inv_tau;
  float scale_log2;
  float *pm, *ps, *pb, *zt;
  float *out_logp, *out_ent, *out_lse, *out_ez;
  uint32_t *status;
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
  float *out_kl;
  uint32_t *status;
};

cudaError_t launch_gather(const void *h, int64_t ld_h, const int64_t *row_idx, int64_t n,
                          int64_t T, int64_t H, void *hs, int num_sms, cudaStream_t stream);
cudaError_t launch_fwd_scoring(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_merge(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_kl(const KlArgs &a, cudaStream_t stream);
cudaError_t launch_kl_merge(const KlArgs &a, cudaStream_t stream);
int fwd_smem_bytes();

}  // namespace flp
