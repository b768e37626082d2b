// kernels_fwdmx.cu -- log-prob and entropy with the logits on the
// block-scaled tensor cores (DeepSeek-V4 book ch. 19, "1. FP4 in OPD": the
// forwards that need no backward, the reference model's scoring among them,
// run in native low precision).
//
// A call quantises the scored hidden rows to MXFP8 (mxfp8_quantize_kernel in
// kernels_klmx.cu, gathering the rows on the way), then runs
// mx_fwd_pipeline_kernel: the logits of E4M3 rows x the E2M1 head from
// block-scaled MMAs, folded by the forward's log-sum-exp/entropy epilogue.
#include <cuda_runtime.h>

#include "launch.h"
#include "launch_util.cuh"
#include "lse_epilogue.cuh"
#include "mx_fwd_pipeline.cuh"

namespace flp {

using FwdBsEpi = LseEpi<1, false>;
#define FWD_BS_KERNEL mx_fwd_pipeline_kernel<FwdBsEpi>

cudaError_t launch_fwd_blockscaled(const FwdBsArgs &a, cudaStream_t stream) {
  FwdBsEpi::Params p{};
  p.targets = a.targets;
  p.K = 1;
  p.row_idx = a.row_idx;
  p.T = a.T;
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.sl = a.scale_log2;
  p.zsent = 0.f;  // no sampling support
  p.pm = a.pm;
  p.ps = a.ps;
  p.pb = a.pb;
  p.zt = a.zt;
  p.counters = a.counters;
  p.splits = a.sch.splits * (kMxFEpiWarps / 4);  // partial slots per row
  p.inv_tau = a.inv_tau;
  p.out_logp = a.out_logp;
  p.out_ent = a.out_ent;
  p.out_lse = a.out_lse;
  p.out_ez = a.out_ez;
  p.status = a.status;
  p.support = nullptr;
  p.ld_support = 0;
  p.tile_cols = kMxFwdTileCols;
  const uint32_t idesc = idesc_mx_e4m3_e2m1(kBM * 2, kMxBN);
  return launch_persistent(FWD_BS_KERNEL, a.grid, kMxFThreads, MxFwdLayout::kSmemBytes, 2, stream,
                           a.tmA, a.tmB, a.tmSfa, a.tmSfb, a.sch, idesc, p, a.status);
}

int fwd_bs_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64)
    return resident_units(FWD_BS_KERNEL, kMxFThreads, MxFwdLayout::kSmemBytes, 2, num_sms);
  if (!cached[dev])
    cached[dev] = resident_units(FWD_BS_KERNEL, kMxFThreads, MxFwdLayout::kSmemBytes, 2, num_sms);
  return cached[dev];
}

}  // namespace flp
