// kernels_kl.cu -- full-vocabulary KL(teacher || student) without either
// logit tensor in memory (DeepSeek-V4 book ch. 19, "Never materialize
// logits" and "TileLang KL kernel": the teacher's logits are rebuilt from its
// cached hidden states through its prediction head and the exact KL is taken
// directly).
//
// Both heads run on the same (row tile, vocabulary tile): the pipeline issues
// two tcgen05 GEMMs per K step into two TMEM accumulators, z_s = h_s W_s^T and
// z_t = h_t W_t^T.  The epilogue keeps, per row, in base 2 (y = z log2 e):
//   teacher  m_t = max y_t,  S_t = sum 2^(y_t - m_t),
//            C_t = sum 2^(y_t - m_t) (z_t - z_s)      (natural units)
//   student  m_s = max y_s,  S_s = sum 2^(y_s - m_s)
// rescaling S and C by 2^(m - m') when a running max grows.  The last warp
// to finish a 32-row group merges the group's split partials and finishes
//   KL = sum_v p_t (log p_t - log p_s) = C_t / S_t - LSE_t + LSE_s,
//   LSE = ln 2 (m + log2 S).
#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "launch_util.cuh"
#include "kl_epilogue.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

using KlEpi = KlEpiT<kKlBN, 32>;

using KlLayout = PipeLayout<kKlBN, kKlStages, 2, kKlCG, kKlAcc>;
using KlMxLayout = PipeLayout<kKlBN, kKlStages, 2, kKlCG, kKlAcc, false, true>;
// With the MX teacher head, four epilogue warps (the eight converter warps
// take the place of the other four).
constexpr int kKlMxEpiWarps = 4;
#define KL_KERNEL vocab_pipeline_kernel<kKlBN, kKlStages, 2, KlEpi, kKlCG, kKlAcc, kKlEpiWarps>
// the teacher head's B operand decoded from MXFP4 in shared memory
#define KL_MX_KERNEL \
  vocab_pipeline_kernel<kKlBN, kKlStages, 2, KlEpi, kKlCG, kKlAcc, kKlMxEpiWarps, false, true>
constexpr int kKlThreads = pipe_threads(kKlEpiWarps);
constexpr int kKlMxThreads = pipe_threads(kKlMxEpiWarps, true);

cudaError_t launch_kl(const KlArgs &a, cudaStream_t stream) {
  KlEpi::Params p;
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.pmt = a.pmt;
  p.pst = a.pst;
  p.pct = a.pct;
  p.pms = a.pms;
  p.pss = a.pss;
  p.counters = a.counters;
  // partial slots per row
  p.splits = a.sch.splits * ((a.mx.packed ? kKlMxEpiWarps : kKlEpiWarps) / 4);
  p.row_idx = a.row_idx;
  p.T = a.T;
  p.out_kl = a.out_kl;
  p.status = a.status;
  p.mx = a.mx;
  const uint32_t idesc = idesc_f16(a.bf16, kBM * kKlCG, kKlBN, false, false);
  if (a.mx.packed)  // tmBt is unused: the teacher's B comes from the MXFP4 operand
    return launch_persistent(KL_MX_KERNEL, a.grid, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG,
                             stream, a.tmAs, a.tmBs, a.tmAt, a.tmBs, a.sch, idesc, p, a.status);
  return launch_persistent(KL_KERNEL, a.grid, kKlThreads, KlLayout::kSmemBytes, kKlCG, stream, a.tmAs, a.tmBs,
                           a.tmAt, a.tmBt, a.sch, idesc, p, a.status);
}

int kl_mx_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64)
    return resident_units(KL_MX_KERNEL, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG, num_sms);
  if (!cached[dev])
    cached[dev] = resident_units(KL_MX_KERNEL, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG, num_sms);
  return cached[dev];
}

int kl_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return resident_units(KL_KERNEL, kKlThreads, KlLayout::kSmemBytes, kKlCG, num_sms);
  if (!cached[dev]) cached[dev] = resident_units(KL_KERNEL, kKlThreads, KlLayout::kSmemBytes, kKlCG, num_sms);
  return cached[dev];
}

}  // namespace flp
